// api.cu -- the C ABI of libmoe: argument validation, workspace layout and
// the launch sequence of each entry point.  Nothing here allocates device
// memory; every buffer is the caller's.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

using moe::GemmProblem;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// physical expert slots of the replicated dispatch at most
constexpr int32_t kMaxPhysical = 65536;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace regions, in this order (each 256-byte aligned):
//   status word | split flags [kPairSplitFlagWords] | mtile_base [E+1] | dispatch chunk counts [chunks*E] |
//   logits [T*E] f32 | padded router weight | h [h_rows*inter] bf16 |
//   (layer only) ids [T*k] | w [T*k] | counts [E] | offsets [E+1] |
//   dest [T*k] | src [T*k] | x_perm [T*k*d] bf16 | y_perm [T*k*d] f32
struct Layout {
  size_t status, flags, mtile, doff, kept, ovf, chunk, logits, wr32, h, ids, w, counts, offsets, dest,
      src, x_perm, y_perm;
  size_t end_route, end_dispatch, end_ffn, end_layer;
};

// h_rows: rows of h; perm_rows: rows of x_perm / y_perm / src (T*k, or
// E*C + T*k for the capacity layer)
Layout make_layout(const moe_shape_t &s, int64_t h_rows, int64_t perm_rows = -1) {
  Layout L;
  const int64_t n = static_cast<int64_t>(s.T) * s.k;
  if (perm_rows < 0) perm_rows = n;
  size_t off = 0;
  L.status = off;
  off = align_up(off + 4);
  L.flags = off;
  off = align_up(off + 4 * static_cast<size_t>(moe::kPairSplitFlagWords));
  L.mtile = off;
  off = align_up(off + 4 * static_cast<size_t>(s.E + 1));
  L.doff = off;  // expert offsets of the capacity dispatch
  off = align_up(off + 4 * static_cast<size_t>(s.E + 1));
  L.kept = off;
  off = align_up(off + 4 * static_cast<size_t>(s.E));
  L.ovf = off;
  off = align_up(off + 4 * static_cast<size_t>(s.E + 1));
  L.chunk = off;
  off = align_up(off + 4 * static_cast<size_t>(moe::dispatch_num_chunks(n)) * s.E);
  L.end_dispatch = off;
  L.logits = off;
  off = align_up(off + 4 * static_cast<size_t>(s.T) * s.E);
  L.wr32 = off;
  off = align_up(off + moe::router_scratch_bytes(s.T, s.d, s.E));
  L.end_route = off;
  L.h = off;
  off = align_up(off + 2 * static_cast<size_t>(h_rows) * s.inter);
  L.end_ffn = off;
  L.ids = off;
  off = align_up(off + 4 * static_cast<size_t>(n));
  L.w = off;
  off = align_up(off + 4 * static_cast<size_t>(n));
  L.counts = off;
  off = align_up(off + 4 * static_cast<size_t>(s.E));
  L.offsets = off;
  off = align_up(off + 4 * static_cast<size_t>(s.E + 1));
  L.dest = off;
  off = align_up(off + 4 * static_cast<size_t>(n));
  L.src = off;
  off = align_up(off + 4 * static_cast<size_t>(perm_rows));
  L.x_perm = off;
  off = align_up(off + 2 * static_cast<size_t>(perm_rows) * s.d);
  L.y_perm = off;
  off = align_up(off + 4 * static_cast<size_t>(perm_rows) * s.d);
  L.end_layer = off;
  return L;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

moe_status_t check_shape(const moe_shape_t *s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->d <= 0 || s->E <= 0 || s->G <= 0 || s->k <= 0 || s->inter <= 0)
    return MOE_ERR_INVALID_ARG;
  if (s->E > 1024 || s->G > 32) return MOE_ERR_INVALID_ARG;
  if (s->E % s->G != 0) return MOE_ERR_INVALID_ARG;
  if (s->topk_group < 1 || s->topk_group > s->G) return MOE_ERR_INVALID_ARG;
  if (s->k > 32 || s->k > s->topk_group * (s->E / s->G)) return MOE_ERR_INVALID_ARG;
  if (s->d % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (s->score != MOE_SCORE_SIGMOID_BIAS && s->score != MOE_SCORE_SOFTMAX)
    return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s->T) * s->k >= (int64_t{1} << 31)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t check_ffn_shape(const moe_shape_t *s) {
  if (s->d % 64 != 0 || s->inter % 64 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t check_ws(void *ws, size_t ws_bytes, size_t need) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                    \
  do {                                   \
    moe_status_t _st = (expr);           \
    if (_st != MOE_OK) return _st;       \
  } while (0)

moe_status_t ffn_rows(const moe_shape_t *s, int32_t layout, int32_t M_max, int64_t *rows) {
  if (layout == MOE_LAYOUT_CONTIGUOUS) {
    *rows = static_cast<int64_t>(s->T) * s->k;
    return MOE_OK;
  }
  if (layout == MOE_LAYOUT_MASKED) {
    if (M_max < 0) return MOE_ERR_INVALID_ARG;
    const int64_t r = static_cast<int64_t>(s->E) * M_max;
    if (r >= (int64_t{1} << 31)) return MOE_ERR_INVALID_ARG;
    *rows = r;
    return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

// gate_up + SwiGLU (and optionally down) over `rows` rows with mtile_base
// already computed in the workspace.
// Pair (2-CTA, 256-row) tiles when the T*k routed rows average at least
// kPairRowsPerExpert per expert; for the masked layout the slabs must also
// hold that many rows (M_max >= kPairRowsPerExpert).
bool use_pair(const moe_shape_t *s, int32_t layout, int32_t M_max) {
  if (s->inter % 128 != 0 || s->d % 256 != 0) return false;
  if (static_cast<int64_t>(s->T) * s->k < static_cast<int64_t>(moe::kPairRowsPerExpert) * s->E)
    return false;
  if (layout == MOE_LAYOUT_CONTIGUOUS || layout == moe::kLayoutTwoSeg) return true;
  return layout == MOE_LAYOUT_MASKED && M_max >= moe::kPairRowsPerExpert;
}
int tile_rows_for(const moe_shape_t *s, int32_t layout, int32_t M_max) {
  return use_pair(s, layout, M_max) ? 256 : 128;
}

// The layers keep the down GEMM's rows compact (fp16 values and a code byte
// per 32 columns, common.cuh) when d is a multiple of 256 (whole 256-column
// down tiles in both GEMM forms).  The fp32 region of `rows` rows holds the
// values, then the codes, then the split tiles' partial sums.
bool compact_rows(const moe_shape_t &s) { return s.d % 256 == 0; }
struct CompactRows {
  void *vals;
  uint8_t *codes;
  float *part;
  int slots;
};
CompactRows compact_layout(void *region, int64_t rows, int d) {
  CompactRows c;
  const size_t vals = align_up(2 * static_cast<size_t>(rows) * d);
  const size_t cods = align_up(static_cast<size_t>(rows) * (d / 32));
  const size_t bytes = 4 * static_cast<size_t>(rows) * d;
  const size_t slot_bytes = 256 * 256 * 4;
  c.slots = bytes > vals + cods
                ? static_cast<int>(std::min<size_t>((bytes - vals - cods) / slot_bytes,
                                                    moe::kPairSplitSlots))
                : 0;
  uint8_t *base = static_cast<uint8_t *>(region);
  c.vals = base;
  c.codes = base + vals;
  c.part = c.slots > 0 ? reinterpret_cast<float *>(base + vals + cods) : nullptr;
  return c;
}

// seg2: the overflow offsets of the two-segment layout (moe::kLayoutTwoSeg)
moe_status_t run_gate_up(const moe_shape_t *s, int32_t layout, const void *x_in,
                         const int32_t *seg, int32_t M_max, int64_t rows, const int32_t *mtile,
                         const void *w_gate_up, void *h, uint32_t *status, cudaStream_t st,
                         const int32_t *seg2 = nullptr) {
  GemmProblem p;
  std::memset(&p, 0, sizeof p);
  p.seg2 = seg2;
  p.E = s->E;
  p.K = s->d;
  p.n_out = s->inter;
  p.layout = layout;
  p.seg = seg;
  p.M_max = M_max;
  p.rows_total = rows;
  p.mtile_base = mtile;
  p.a = x_in;
  p.b = w_gate_up;
  p.b_rows = 2 * s->inter;
  p.out = h;
  p.status = status;
  p.pair = use_pair(s, layout, M_max);
  return cuda_status(moe::launch_gemm_gate_up_swiglu(p, st));
}

// y16_codes: compact output (pair form only): y receives the fp16 values and
// y16_codes the code bytes; split_part / split_slots the split-tile scratch
moe_status_t run_down(const moe_shape_t *s, int32_t layout, const void *h, const int32_t *seg,
                      int32_t M_max, int64_t rows, const int32_t *mtile, const void *w_down,
                      void *y, uint32_t *status, uint32_t *split_flags, cudaStream_t st,
                      uint8_t *y16_codes = nullptr, float *split_part = nullptr,
                      int split_slots = 0, const int32_t *seg2 = nullptr) {
  GemmProblem p;
  std::memset(&p, 0, sizeof p);
  p.seg2 = seg2;
  p.out_codes = y16_codes;
  p.split_part = split_part;
  p.split_part_slots = split_slots;
  p.E = s->E;
  p.K = s->inter;
  p.n_out = s->d;
  p.layout = layout;
  p.seg = seg;
  p.M_max = M_max;
  p.rows_total = rows;
  p.mtile_base = mtile;
  p.a = h;
  p.b = w_down;
  p.b_rows = s->d;
  p.out = y;
  p.status = status;
  p.split_flags = split_flags;
  p.pair = use_pair(s, layout, M_max);
  return cuda_status(moe::launch_gemm_down(p, st));
}

}  // namespace

moe_status_t moe::check_shape_for_abi(const moe_shape_t *shape) { return check_shape(shape); }

extern "C" {

const char *moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_OVERFLOW: return "MOE_ERR_OVERFLOW";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_workspace_size(const moe_shape_t *shape, size_t *bytes) {
  MOE_TRY(check_shape(shape));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*shape, static_cast<int64_t>(shape->T) * shape->k).end_layer;
  return MOE_OK;
}

moe_status_t moe_expert_ffn_workspace_size(const moe_shape_t *shape, int32_t layout,
                                           int32_t M_max, size_t *bytes) {
  MOE_TRY(check_shape(shape));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  int64_t rows = 0;
  MOE_TRY(ffn_rows(shape, layout, M_max, &rows));
  *bytes = make_layout(*shape, rows).end_ffn;
  return MOE_OK;
}

moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_ws(ws, ws_bytes, 4));
  // the status word and the split flags of the down GEMM (all zero at rest)
  const size_t n = std::min(ws_bytes, kAlign + 4 * static_cast<size_t>(moe::kPairSplitFlagWords));
  return cuda_status(cudaMemsetAsync(ws, 0, n, stream));
}

moe_status_t moe_get_device_status(void *ws, size_t ws_bytes, moe_stream_t stream,
                                   moe_status_t *status) {
  MOE_TRY(check_ws(ws, ws_bytes, 4));
  if (!status) return MOE_ERR_INVALID_ARG;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, ws, 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, 4, stream) != cudaSuccess) return MOE_ERR_CUDA;
  // A launch that stopped early (a wait ran out) may have left split flags
  // of the down GEMM raised, and a replay of a captured graph raises the
  // same value again: clear them with the error, so that the next launch
  // cannot take a stale flag for its own.
  const size_t flags_off = align_up(4);
  const size_t flags_bytes = 4 * static_cast<size_t>(moe::kPairSplitFlagWords);
  if (word != 0 && ws_bytes >= flags_off + flags_bytes &&
      cudaMemsetAsync(static_cast<char *>(ws) + flags_off, 0, flags_bytes, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  moe_status_t out = MOE_OK;
  for (int b = 31; b >= 1; --b)
    if (word & (1u << b)) {
      out = static_cast<moe_status_t>(b);
      break;
    }
  *status = out;
  return MOE_OK;
}

moe_status_t moe_route(const moe_shape_t *shape, const void *x, const void *w_r,
                       const float *bias, int32_t *topk_ids, float *topk_w, float *logits,
                       void *ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (shape->T == 0) return MOE_OK;
  const moe_shape_t &s = *shape;
  if (!x || !w_r || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (s.score == MOE_SCORE_SIGMOID_BIAS && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(s, 0);
  MOE_TRY(check_ws(ws, ws_bytes, L.end_route));
  if (!logits)
    return cuda_status(moe::launch_router(x, w_r, bias, s.T, s.d, s.E, s.G, s.topk_group, s.k,
                                          s.score, s.bias_scale, at<float>(ws, L.logits),
                                          topk_ids, topk_w, at<void>(ws, L.wr32),
                                          at<uint32_t>(ws, L.status), stream));
  MOE_TRY(cuda_status(
      moe::launch_router_logits(x, w_r, s.T, s.d, s.E, logits, at<void>(ws, L.wr32), stream)));
  return cuda_status(moe::launch_router_select(logits, bias, s.T, s.E, s.G, s.topk_group, s.k,
                                               s.score, s.bias_scale, 0, topk_ids, topk_w,
                                               stream));
}

moe_status_t moe_route_from_logits(const moe_shape_t *shape, const float *logits,
                                   const float *bias, int32_t *topk_ids, float *topk_w,
                                   moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (shape->T == 0) return MOE_OK;
  const moe_shape_t &s = *shape;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (s.score == MOE_SCORE_SIGMOID_BIAS && !bias) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_router_select(logits, bias, s.T, s.E, s.G, s.topk_group, s.k,
                                               s.score, s.bias_scale, 0, topk_ids, topk_w,
                                               stream));
}

moe_status_t moe_group_topk(const moe_shape_t *shape, const float *scores, int32_t *topk_ids,
                            moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (shape->T == 0) return MOE_OK;
  const moe_shape_t &s = *shape;
  if (!scores || !topk_ids) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_router_select(scores, nullptr, s.T, s.E, s.G, s.topk_group,
                                               s.k, s.score, s.bias_scale, 1, topk_ids,
                                               nullptr, stream));
}

moe_status_t moe_dispatch(const moe_shape_t *shape, const int32_t *topk_ids, const void *x,
                          int32_t *counts, int32_t *offsets, int32_t *src_token, int32_t *dest,
                          void *x_perm, void *ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (shape->T == 0) return MOE_OK;
  const moe_shape_t &s = *shape;
  if (!topk_ids || !counts || !offsets || !src_token || !dest) return MOE_ERR_INVALID_ARG;
  if (x && !x_perm) return MOE_ERR_INVALID_ARG;
  if (x && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(s, 0);
  MOE_TRY(check_ws(ws, ws_bytes, L.end_dispatch));
  return cuda_status(moe::launch_dispatch(topk_ids, s.T, s.k, s.E, x, s.d, counts, offsets,
                                          src_token, dest, x_perm, at<int32_t>(ws, L.chunk),
                                          nullptr, 128, at<uint32_t>(ws, L.status), stream));
}

// scratch of moe_dispatch_replicated, in this order (each 256-byte aligned):
// status word | chunk histograms | counts_log [E] | offsets_log [E+1] |
// mtile [E+1] | dest_log [T*k] | src_log [T*k] | n_rep [E] | rep_first [E+1] |
// rep_slots [P] | slot_rank [P]
struct ReplicaLayout {
  size_t chunk, counts, offsets, mtile, dest, src, n_rep, rep_first, rep_slots, slot_rank, end;
};
ReplicaLayout make_replica_layout(const moe_shape_t &s, int32_t P) {
  ReplicaLayout L;
  const int64_t n = static_cast<int64_t>(s.T) * s.k;
  size_t off = align_up(4);
  auto take = [&](size_t bytes) {
    const size_t at_ = off;
    off = align_up(off + bytes);
    return at_;
  };
  L.chunk = take(4 * static_cast<size_t>(moe::dispatch_num_chunks(n)) * s.E);
  L.counts = take(4 * static_cast<size_t>(s.E));
  L.offsets = take(4 * static_cast<size_t>(s.E + 1));
  L.mtile = take(4 * static_cast<size_t>(s.E + 1));
  L.dest = take(4 * static_cast<size_t>(n));
  L.src = take(4 * static_cast<size_t>(n));
  L.n_rep = take(4 * static_cast<size_t>(s.E));
  L.rep_first = take(4 * static_cast<size_t>(s.E + 1));
  L.rep_slots = take(4 * static_cast<size_t>(P));
  L.slot_rank = take(4 * static_cast<size_t>(P));
  L.end = off;
  return L;
}

moe_status_t moe_dispatch_replicated_workspace_size(const moe_shape_t *shape,
                                                    int32_t num_physical, size_t *bytes) {
  MOE_TRY(check_shape(shape));
  if (!bytes || num_physical < 1 || num_physical > kMaxPhysical) return MOE_ERR_INVALID_ARG;
  *bytes = make_replica_layout(*shape, num_physical).end;
  return MOE_OK;
}

moe_status_t moe_dispatch_replicated(const moe_shape_t *shape, int32_t num_physical,
                                     const int32_t *phys_expert, const int32_t *topk_ids,
                                     const void *x, int32_t *counts_phys, int32_t *offsets_phys,
                                     int32_t *src_token, int32_t *dest, void *x_perm, void *ws,
                                     size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (num_physical < 1 || num_physical > kMaxPhysical) return MOE_ERR_INVALID_ARG;
  if (shape->T == 0) return MOE_OK;
  const moe_shape_t &s = *shape;
  if (!phys_expert || !topk_ids || !counts_phys || !offsets_phys || !src_token || !dest)
    return MOE_ERR_INVALID_ARG;
  if (x && !x_perm) return MOE_ERR_INVALID_ARG;
  if (x && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  const ReplicaLayout L = make_replica_layout(s, num_physical);
  MOE_TRY(check_ws(ws, ws_bytes, L.end));
  moe::ReplicaScratch w;
  w.chunk = at<int32_t>(ws, L.chunk);
  w.counts_log = at<int32_t>(ws, L.counts);
  w.offsets_log = at<int32_t>(ws, L.offsets);
  w.mtile = at<int32_t>(ws, L.mtile);
  w.dest_log = at<int32_t>(ws, L.dest);
  w.src_log = at<int32_t>(ws, L.src);
  w.n_rep = at<int32_t>(ws, L.n_rep);
  w.rep_first = at<int32_t>(ws, L.rep_first);
  w.rep_slots = at<int32_t>(ws, L.rep_slots);
  w.slot_rank = at<int32_t>(ws, L.slot_rank);
  return cuda_status(moe::launch_dispatch_replicated(
      topk_ids, s.T, s.k, s.E, x, s.d, num_physical, phys_expert, counts_phys, offsets_phys,
      src_token, dest, x_perm, w, at<uint32_t>(ws, 0), stream));
}

static moe_status_t ffn_common(const moe_shape_t *shape, int32_t layout, const void *x_in,
                               const int32_t *seg, int32_t M_max, void *ws, size_t ws_bytes,
                               int64_t *rows, Layout *L) {
  MOE_TRY(check_shape(shape));
  MOE_TRY(check_ffn_shape(shape));
  MOE_TRY(ffn_rows(shape, layout, M_max, rows));
  if (!x_in || !seg) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_in)) return MOE_ERR_INVALID_ARG;
  *L = make_layout(*shape, *rows);
  return check_ws(ws, ws_bytes, L->end_ffn);
}

moe_status_t moe_expert_ffn(const moe_shape_t *shape, int32_t layout, const void *x_in,
                            const int32_t *seg, int32_t M_max, const void *w_gate_up,
                            const void *w_down, float *y_out, void *ws, size_t ws_bytes,
                            moe_stream_t stream) {
  if (shape && shape->T == 0 && layout == MOE_LAYOUT_CONTIGUOUS) return check_shape(shape);
  int64_t rows = 0;
  Layout L;
  MOE_TRY(ffn_common(shape, layout, x_in, seg, M_max, ws, ws_bytes, &rows, &L));
  if (!w_gate_up || !w_down || !y_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(y_out))
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  uint32_t *status = at<uint32_t>(ws, L.status);
  int32_t *mtile = at<int32_t>(ws, L.mtile);
  void *h = at<void>(ws, L.h);
  MOE_TRY(cuda_status(moe::launch_ffn_tiles(seg, layout, shape->E, M_max,
                                            tile_rows_for(shape, layout, M_max), mtile, status,
                                            stream, nullptr, at<uint32_t>(ws, L.flags))));
  MOE_TRY(run_gate_up(shape, layout, x_in, seg, M_max, rows, mtile, w_gate_up, h, status,
                      stream));
  return run_down(shape, layout, h, seg, M_max, rows, mtile, w_down, y_out, status,
                  at<uint32_t>(ws, L.flags), stream);
}

moe_status_t moe_expert_gate_up(const moe_shape_t *shape, int32_t layout, const void *x_in,
                                const int32_t *seg, int32_t M_max, const void *w_gate_up,
                                void *h_out, void *ws, size_t ws_bytes, moe_stream_t stream) {
  if (shape && shape->T == 0 && layout == MOE_LAYOUT_CONTIGUOUS) return check_shape(shape);
  int64_t rows = 0;
  Layout L;
  MOE_TRY(ffn_common(shape, layout, x_in, seg, M_max, ws, ws_bytes, &rows, &L));
  if (!w_gate_up || !h_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate_up) || !aligned16(h_out)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  uint32_t *status = at<uint32_t>(ws, L.status);
  int32_t *mtile = at<int32_t>(ws, L.mtile);
  MOE_TRY(cuda_status(moe::launch_ffn_tiles(seg, layout, shape->E, M_max,
                                            tile_rows_for(shape, layout, M_max), mtile, status,
                                            stream)));
  return run_gate_up(shape, layout, x_in, seg, M_max, rows, mtile, w_gate_up, h_out, status,
                     stream);
}

moe_status_t moe_expert_down(const moe_shape_t *shape, int32_t layout, const void *h_in,
                             const int32_t *seg, int32_t M_max, const void *w_down,
                             float *y_out, void *ws, size_t ws_bytes, moe_stream_t stream) {
  if (shape && shape->T == 0 && layout == MOE_LAYOUT_CONTIGUOUS) return check_shape(shape);
  int64_t rows = 0;
  Layout L;
  MOE_TRY(ffn_common(shape, layout, h_in, seg, M_max, ws, ws_bytes, &rows, &L));
  if (!w_down || !y_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_down) || !aligned16(y_out)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  uint32_t *status = at<uint32_t>(ws, L.status);
  int32_t *mtile = at<int32_t>(ws, L.mtile);
  MOE_TRY(cuda_status(moe::launch_ffn_tiles(seg, layout, shape->E, M_max,
                                            tile_rows_for(shape, layout, M_max), mtile, status,
                                            stream, nullptr, at<uint32_t>(ws, L.flags))));
  return run_down(shape, layout, h_in, seg, M_max, rows, mtile, w_down, y_out, status,
                  at<uint32_t>(ws, L.flags), stream);
}

moe_status_t moe_combine(const moe_shape_t *shape, const float *y_perm, const int32_t *dest,
                         const float *topk_w, void *y, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (shape->T == 0) return MOE_OK;
  if (!y_perm || !dest || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      moe::launch_combine(y_perm, static_cast<int64_t>(shape->T) * shape->k, dest, topk_w,
                          shape->T, shape->k, shape->d, y, stream));
}

moe_status_t moe_layer(const moe_shape_t *shape, const void *x, const void *w_r,
                       const float *bias, const void *w_gate_up, const void *w_down, void *y,
                       int32_t *topk_ids, float *topk_w, int32_t *counts, void *ws,
                       size_t ws_bytes, void *const *stage_events, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (shape->T == 0) return MOE_OK;
  MOE_TRY(check_ffn_shape(shape));
  const moe_shape_t &s = *shape;
  if (!x || !w_r || !w_gate_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (s.score == MOE_SCORE_SIGMOID_BIAS && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_r) || !aligned16(w_gate_up) || !aligned16(w_down) ||
      !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(s.T) * s.k;
  const Layout L = make_layout(s, n);
  MOE_TRY(check_ws(ws, ws_bytes, L.end_layer));
  uint32_t *status = at<uint32_t>(ws, L.status);
  int32_t *ids = topk_ids ? topk_ids : at<int32_t>(ws, L.ids);
  float *w = topk_w ? topk_w : at<float>(ws, L.w);
  int32_t *cnt = counts ? counts : at<int32_t>(ws, L.counts);
  int32_t *offsets = at<int32_t>(ws, L.offsets);
  int32_t *mtile = at<int32_t>(ws, L.mtile);
  int32_t *dest = at<int32_t>(ws, L.dest);
  int32_t *src = at<int32_t>(ws, L.src);
  void *x_perm = at<void>(ws, L.x_perm);
  float *y_perm = at<float>(ws, L.y_perm);
  void *h = at<void>(ws, L.h);
  float *logits = at<float>(ws, L.logits);

  auto mark = [&](int i) -> moe_status_t {
    if (!stage_events) return MOE_OK;
    return cuda_status(cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), stream));
  };
  MOE_TRY(mark(0));
  MOE_TRY(cuda_status(moe::launch_router(x, w_r, bias, s.T, s.d, s.E, s.G, s.topk_group, s.k,
                                         s.score, s.bias_scale, logits, ids, w,
                                         at<void>(ws, L.wr32), status, stream)));
  MOE_TRY(mark(1));
  MOE_TRY(cuda_status(moe::launch_dispatch(ids, s.T, s.k, s.E, x, s.d, cnt, offsets, src, dest,
                                           x_perm, at<int32_t>(ws, L.chunk), mtile,
                                           tile_rows_for(shape, MOE_LAYOUT_CONTIGUOUS, 0),
                                           status, stream,
                                           moe::CapacityArgs{0, 0, 0, nullptr, nullptr},
                                           at<uint32_t>(ws, L.flags))));
  MOE_TRY(mark(2));
  MOE_TRY(run_gate_up(shape, MOE_LAYOUT_CONTIGUOUS, x_perm, offsets, 0, n, mtile, w_gate_up, h,
                      status, stream));
  MOE_TRY(mark(3));
  if (compact_rows(s)) {
    // the down GEMM writes the compact rows (2 + 1/32 bytes per value instead
    // of 4) into the y_perm region; the combine reads them
    const CompactRows c = compact_layout(y_perm, n, s.d);
    MOE_TRY(run_down(shape, MOE_LAYOUT_CONTIGUOUS, h, offsets, 0, n, mtile, w_down, c.vals,
                     status, at<uint32_t>(ws, L.flags), stream, c.codes, c.part, c.slots));
    MOE_TRY(mark(4));
    MOE_TRY(cuda_status(
        moe::launch_combine16(c.vals, c.codes, n, dest, w, s.T, s.k, s.d, y, stream)));
    return mark(5);
  }
  MOE_TRY(run_down(shape, MOE_LAYOUT_CONTIGUOUS, h, offsets, 0, n, mtile, w_down, y_perm, status,
                   at<uint32_t>(ws, L.flags), stream));
  MOE_TRY(mark(4));
  MOE_TRY(cuda_status(moe::launch_combine(y_perm, n, dest, w, s.T, s.k, s.d, y, stream)));
  return mark(5);
}

// ---------------------------------------------------------------------------
// FP8 quantization
// ---------------------------------------------------------------------------

moe_status_t moe_quantize_fp8_rows(const void *x, int64_t rows, int32_t cols, void *q,
                                   float *scales, moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !scales || !aligned16(x) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_quantize_rows_fp8(x, rows, cols, q, scales, stream));
}

moe_status_t moe_quantize_fp8_blocks(const void *w, int32_t mats, int32_t rows, int32_t cols,
                                     void *q, float *scales, moe_stream_t stream) {
  if (mats < 0 || rows < 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (mats == 0 || rows == 0) return MOE_OK;
  if (!w || !q || !scales || !aligned16(w) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_quantize_blocks_fp8(w, mats, rows, cols, q, scales, stream));
}

// ---------------------------------------------------------------------------
// FP8 expert FFN and layer
// ---------------------------------------------------------------------------

struct LayoutF8 {
  size_t status, mtile, chunk, logits, wr32, hq, hs, ids, w, counts, offsets, dest, src, xq,
      xs, xq_perm, xs_perm, y_perm;
  size_t end_ffn, end_layer;
};

// FFN part (the FP8 codes and scales of h) for `rows` rows; the
// layer part adds routing, dispatch and the FP8 activations
LayoutF8 make_fp8_layout(const moe_shape_t &s, int64_t rows) {
  LayoutF8 L;
  const int64_t n = static_cast<int64_t>(s.T) * s.k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at_ = off;
    off = align_up(off + bytes);
    return at_;
  };
  L.status = take(4);
  L.mtile = take(4 * static_cast<size_t>(s.E + 1));
  L.hq = take(static_cast<size_t>(rows) * s.inter);
  L.hs = take(4 * static_cast<size_t>(rows) * (s.inter / 128));
  L.end_ffn = off;
  L.chunk = take(4 * static_cast<size_t>(moe::dispatch_num_chunks(n)) * s.E);
  L.logits = take(4 * static_cast<size_t>(s.T) * s.E);
  L.wr32 = take(moe::router_scratch_bytes(s.T, s.d, s.E));
  L.ids = take(4 * static_cast<size_t>(n));
  L.w = take(4 * static_cast<size_t>(n));
  L.counts = take(4 * static_cast<size_t>(s.E));
  L.offsets = take(4 * static_cast<size_t>(s.E + 1));
  L.dest = take(4 * static_cast<size_t>(n));
  L.src = take(4 * static_cast<size_t>(n));
  L.xq = take(static_cast<size_t>(s.T) * s.d);
  L.xs = take(4 * static_cast<size_t>(s.T) * (s.d / 128));
  L.xq_perm = take(static_cast<size_t>(n) * s.d);
  L.xs_perm = take(4 * static_cast<size_t>(n) * (s.d / 128));
  L.y_perm = take(4 * static_cast<size_t>(n) * s.d);
  L.end_layer = off;
  return L;
}

moe_status_t check_fp8_shape(const moe_shape_t *s) {
  if (s->d % 128 != 0 || s->inter % 128 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// FP8 GEMMs on CTA pairs (256 x 256 tiles: d a multiple of 256) under the
// bf16 GEMMs' row criterion
bool use_pair_fp8(const moe_shape_t *s, int32_t layout, int32_t M_max) {
  if (s->d % 256 != 0) return false;
  if (static_cast<int64_t>(s->T) * s->k < static_cast<int64_t>(moe::kPairRowsPerExpert) * s->E)
    return false;
  if (layout == MOE_LAYOUT_CONTIGUOUS) return true;
  return layout == MOE_LAYOUT_MASKED && M_max >= moe::kPairRowsPerExpert;
}

// FP8 gate_up + SwiGLU -> h (bf16) -> FP8 codes of h -> FP8 down, over rows
// whose m-tile prefix (128-row tiles) is in the workspace
moe_status_t run_ffn_fp8(const moe_shape_t *s, int32_t layout, const void *xq, const float *xs,
                         const int32_t *seg, int32_t M_max, int64_t rows, int32_t *mtile,
                         const void *wgu_q, const float *wgu_s, const void *wd_q,
                         const float *wd_s, void *y, void *ws, const LayoutF8 &L,
                         cudaStream_t st, uint8_t *y16_codes = nullptr) {
  uint32_t *status = at<uint32_t>(ws, L.status);
  GemmProblem p;
  std::memset(&p, 0, sizeof p);
  p.E = s->E;
  p.layout = layout;
  p.seg = seg;
  p.M_max = M_max;
  p.rows_total = rows;
  p.mtile_base = mtile;
  p.status = status;
  p.pair = use_pair_fp8(s, layout, M_max);
  p.K = s->d;
  p.n_out = s->inter;
  p.a = xq;
  p.b = wgu_q;
  p.b_rows = 2 * s->inter;
  // gate_up quantizes h (its bf16 values, per row and 128 columns) in its
  // epilogue: h leaves as e4m3 codes and scales
  p.out = at<void>(ws, L.hq);
  p.out_h_scales = at<float>(ws, L.hs);
  MOE_TRY(cuda_status(moe::launch_gemm_fp8_gate_up_swiglu(p, xs, wgu_s, st)));
  p.out_h_scales = nullptr;
  p.K = s->inter;
  p.n_out = s->d;
  p.a = at<void>(ws, L.hq);
  p.b = wd_q;
  p.b_rows = s->d;
  p.out = y;
  p.out_codes = y16_codes;  // compact rows (nullptr: fp32)
  return cuda_status(moe::launch_gemm_fp8_down(p, at<float>(ws, L.hs), wd_s, st));
}

moe_status_t moe_expert_ffn_fp8_workspace_size(const moe_shape_t *shape, int32_t layout,
                                               int32_t M_max, size_t *bytes) {
  MOE_TRY(check_shape(shape));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  int64_t rows = 0;
  MOE_TRY(ffn_rows(shape, layout, M_max, &rows));
  *bytes = make_fp8_layout(*shape, rows).end_ffn;
  return MOE_OK;
}

moe_status_t moe_expert_ffn_fp8(const moe_shape_t *shape, int32_t layout, const void *x_q,
                                const float *x_scale, const int32_t *seg, int32_t M_max,
                                const void *w_gate_up_q, const float *w_gate_up_scale,
                                const void *w_down_q, const float *w_down_scale, float *y_out,
                                void *ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  MOE_TRY(check_fp8_shape(shape));
  int64_t rows = 0;
  MOE_TRY(ffn_rows(shape, layout, M_max, &rows));
  if (rows == 0) return MOE_OK;
  if (!x_q || !x_scale || !seg || !w_gate_up_q || !w_gate_up_scale || !w_down_q ||
      !w_down_scale || !y_out)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_q) || !aligned16(w_gate_up_q) || !aligned16(w_down_q) || !aligned16(y_out))
    return MOE_ERR_INVALID_ARG;
  const LayoutF8 L = make_fp8_layout(*shape, rows);
  MOE_TRY(check_ws(ws, ws_bytes, L.end_ffn));
  int32_t *mtile = at<int32_t>(ws, L.mtile);
  MOE_TRY(cuda_status(moe::launch_ffn_tiles(seg, layout, shape->E, M_max,
                                            use_pair_fp8(shape, layout, M_max) ? 256 : 128, mtile,
                                            at<uint32_t>(ws, L.status), stream)));
  return run_ffn_fp8(shape, layout, x_q, x_scale, seg, M_max, rows, mtile, w_gate_up_q,
                     w_gate_up_scale, w_down_q, w_down_scale, y_out, ws, L, stream);
}

moe_status_t moe_layer_fp8_workspace_size(const moe_shape_t *shape, size_t *bytes) {
  MOE_TRY(check_shape(shape));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_fp8_layout(*shape, static_cast<int64_t>(shape->T) * shape->k).end_layer;
  return MOE_OK;
}

moe_status_t moe_layer_fp8(const moe_shape_t *shape, const void *x, const void *w_r,
                           const float *bias, const void *w_gate_up_q,
                           const float *w_gate_up_scale, const void *w_down_q,
                           const float *w_down_scale, void *y, int32_t *counts, void *ws,
                           size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (shape->T == 0) return MOE_OK;
  MOE_TRY(check_fp8_shape(shape));
  const moe_shape_t &s = *shape;
  if (!x || !w_r || !w_gate_up_q || !w_gate_up_scale || !w_down_q || !w_down_scale || !y)
    return MOE_ERR_INVALID_ARG;
  if (s.score == MOE_SCORE_SIGMOID_BIAS && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_r) || !aligned16(w_gate_up_q) || !aligned16(w_down_q) ||
      !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(s.T) * s.k;
  const LayoutF8 L = make_fp8_layout(s, n);
  MOE_TRY(check_ws(ws, ws_bytes, L.end_layer));
  uint32_t *status = at<uint32_t>(ws, L.status);
  int32_t *ids = at<int32_t>(ws, L.ids);
  float *w = at<float>(ws, L.w);
  int32_t *cnt = counts ? counts : at<int32_t>(ws, L.counts);
  int32_t *offsets = at<int32_t>(ws, L.offsets);
  int32_t *mtile = at<int32_t>(ws, L.mtile);
  int32_t *dest = at<int32_t>(ws, L.dest);
  int32_t *src = at<int32_t>(ws, L.src);
  float *y_perm = at<float>(ws, L.y_perm);
  MOE_TRY(cuda_status(moe::launch_router(x, w_r, bias, s.T, s.d, s.E, s.G, s.topk_group, s.k,
                                         s.score, s.bias_scale, at<float>(ws, L.logits), ids, w,
                                         at<void>(ws, L.wr32), status, stream)));
  // the dispatch moves FP8 rows and their scales
  MOE_TRY(cuda_status(moe::launch_quantize_rows_fp8(x, s.T, s.d, at<void>(ws, L.xq),
                                                    at<float>(ws, L.xs), stream)));
  MOE_TRY(cuda_status(moe::launch_dispatch(
      ids, s.T, s.k, s.E, nullptr, s.d, cnt, offsets, src, dest, nullptr,
      at<int32_t>(ws, L.chunk), mtile, use_pair_fp8(shape, MOE_LAYOUT_CONTIGUOUS, 0) ? 256 : 128,
      status, stream)));
  MOE_TRY(cuda_status(moe::launch_gather_rows(at<void>(ws, L.xq), s.d, at<float>(ws, L.xs),
                                              s.d / 128, ids, dest, s.k, s.E, src,
                                              offsets + s.E, n, s.T,
                                              at<void>(ws, L.xq_perm), at<float>(ws, L.xs_perm),
                                              stream)));
  if (compact_rows(s)) {
    // the down GEMM writes the compact rows, as in moe_layer
    const CompactRows c = compact_layout(y_perm, n, s.d);
    MOE_TRY(run_ffn_fp8(shape, MOE_LAYOUT_CONTIGUOUS, at<void>(ws, L.xq_perm),
                        at<float>(ws, L.xs_perm), offsets, 0, n, mtile, w_gate_up_q,
                        w_gate_up_scale, w_down_q, w_down_scale, c.vals, ws, L, stream,
                        c.codes));
    return cuda_status(
        moe::launch_combine16(c.vals, c.codes, n, dest, w, s.T, s.k, s.d, y, stream));
  }
  MOE_TRY(run_ffn_fp8(shape, MOE_LAYOUT_CONTIGUOUS, at<void>(ws, L.xq_perm),
                      at<float>(ws, L.xs_perm), offsets, 0, n, mtile, w_gate_up_q,
                      w_gate_up_scale, w_down_q, w_down_scale, y_perm, ws, L, stream));
  return cuda_status(moe::launch_combine(y_perm, n, dest, w, s.T, s.k, s.d, y, stream));
}

// ---------------------------------------------------------------------------
// capacity variant
// ---------------------------------------------------------------------------

int32_t moe_expert_capacity(int32_t T, int32_t k, int32_t E, double c) {
  if (T < 0 || k < 1 || E < 1 || !(c >= 0.0) || !std::isfinite(c)) return -1;
  const double v = std::ceil(c * (static_cast<double>(T) * k / E));
  if (v >= 2147483647.0) return -1;
  return static_cast<int32_t>(v);
}

static moe_status_t check_capacity(const moe_shape_t *s, int32_t capacity, int32_t overflow) {
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  if (overflow != MOE_OVERFLOW_DROP && overflow != MOE_OVERFLOW_SECOND_ROUND)
    return MOE_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(s->E) * capacity + static_cast<int64_t>(s->T) * s->k;
  if (rows >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t moe_dispatch_capacity(const moe_shape_t *shape, int32_t capacity,
                                   int32_t overflow, const int32_t *topk_ids, const void *x,
                                   int32_t *counts, int32_t *kept, int32_t *ovf_offsets,
                                   int32_t *dest, int32_t *src_row, void *x_rows, void *ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  MOE_TRY(check_capacity(shape, capacity, overflow));
  const moe_shape_t &s = *shape;
  if (!topk_ids || !counts || !kept || !ovf_offsets || !dest || !src_row)
    return MOE_ERR_INVALID_ARG;
  if (x && !x_rows) return MOE_ERR_INVALID_ARG;
  if (x && (!aligned16(x) || !aligned16(x_rows))) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(s, 0);
  MOE_TRY(check_ws(ws, ws_bytes, L.end_dispatch));
  if (s.T == 0) {
    // no assignments: every count is zero
    MOE_TRY(cuda_status(cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.E, stream)));
    MOE_TRY(cuda_status(cudaMemsetAsync(kept, 0, sizeof(int32_t) * s.E, stream)));
    return cuda_status(cudaMemsetAsync(ovf_offsets, 0, sizeof(int32_t) * (s.E + 1), stream));
  }
  moe::CapacityArgs cap{capacity, overflow, s.E, kept, ovf_offsets};
  return cuda_status(moe::launch_dispatch(topk_ids, s.T, s.k, s.E, x, s.d, counts,
                                          at<int32_t>(ws, L.doff), src_row, dest, x_rows,
                                          at<int32_t>(ws, L.chunk), nullptr, 128,
                                          at<uint32_t>(ws, L.status), stream, cap));
}

static Layout capacity_layout(const moe_shape_t &s, int32_t capacity) {
  const int64_t rows = static_cast<int64_t>(s.E) * capacity + static_cast<int64_t>(s.T) * s.k;
  return make_layout(s, rows, rows);
}

moe_status_t moe_layer_capacity_workspace_size(const moe_shape_t *shape, int32_t capacity,
                                               size_t *bytes) {
  MOE_TRY(check_shape(shape));
  MOE_TRY(check_capacity(shape, capacity, MOE_OVERFLOW_DROP));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = capacity_layout(*shape, capacity).end_layer;
  return MOE_OK;
}

moe_status_t moe_layer_capacity(const moe_shape_t *shape, int32_t capacity, int32_t overflow,
                                const void *x, const void *w_r, const float *bias,
                                const void *w_gate_up, const void *w_down, void *y,
                                int32_t *counts, int32_t *kept, void *ws, size_t ws_bytes,
                                moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  MOE_TRY(check_capacity(shape, capacity, overflow));
  if (shape->T == 0) return MOE_OK;
  MOE_TRY(check_ffn_shape(shape));
  const moe_shape_t &s = *shape;
  if (!x || !w_r || !w_gate_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (s.score == MOE_SCORE_SIGMOID_BIAS && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_r) || !aligned16(w_gate_up) || !aligned16(w_down) ||
      !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(s.T) * s.k;
  const int64_t pad = static_cast<int64_t>(s.E) * capacity;
  const Layout L = capacity_layout(s, capacity);
  MOE_TRY(check_ws(ws, ws_bytes, L.end_layer));
  uint32_t *status = at<uint32_t>(ws, L.status);
  int32_t *ids = at<int32_t>(ws, L.ids);
  float *w = at<float>(ws, L.w);
  int32_t *cnt = counts ? counts : at<int32_t>(ws, L.counts);
  int32_t *kp = kept ? kept : at<int32_t>(ws, L.kept);
  int32_t *ovf = at<int32_t>(ws, L.ovf);
  int32_t *mtile = at<int32_t>(ws, L.mtile);
  int32_t *dest = at<int32_t>(ws, L.dest);
  uint8_t *x_rows = at<uint8_t>(ws, L.x_perm);
  float *y_rows = at<float>(ws, L.y_perm);
  // compact rows (when d allows): the padded rows, then the overflow rows
  const CompactRows cr = compact_rows(s) ? compact_layout(y_rows, pad + n, s.d)
                                         : CompactRows{nullptr, nullptr, nullptr, 0};
  uint8_t *h = at<uint8_t>(ws, L.h);
  float *logits = at<float>(ws, L.logits);

  MOE_TRY(cuda_status(moe::launch_router(x, w_r, bias, s.T, s.d, s.E, s.G, s.topk_group, s.k,
                                         s.score, s.bias_scale, logits, ids, w,
                                         at<void>(ws, L.wr32), status, stream)));
  moe::CapacityArgs cap{capacity, overflow, s.E, kp, ovf};
  MOE_TRY(cuda_status(moe::launch_dispatch(ids, s.T, s.k, s.E, x, s.d, cnt,
                                           at<int32_t>(ws, L.doff), at<int32_t>(ws, L.src),
                                           dest, x_rows, at<int32_t>(ws, L.chunk), nullptr,
                                           128, status, stream, cap)));
  // Second round: where the expert GEMMs stream weights (the 1-CTA form, few
  // rows per expert), both rounds run as one launch per GEMM -- each
  // expert's padded rows, then its overflow rows (the two-segment layout) --
  // so its weights stream once; where they are compute-bound (CTA pairs) the
  // overflow rows run after the padded ones, which measured faster there.
  const bool one_launch = overflow == MOE_OVERFLOW_SECOND_ROUND &&
                          !use_pair(shape, MOE_LAYOUT_CONTIGUOUS, 0);
  if (one_launch) {
    MOE_TRY(cuda_status(moe::launch_ffn_tiles(
        kp, moe::kLayoutTwoSeg, s.E, capacity,
        tile_rows_for(shape, moe::kLayoutTwoSeg, capacity), mtile, status, stream, ovf,
        at<uint32_t>(ws, L.flags))));
    MOE_TRY(run_gate_up(shape, moe::kLayoutTwoSeg, x_rows, kp, capacity, pad + n, mtile,
                        w_gate_up, h, status, stream, ovf));
    if (cr.vals)
      MOE_TRY(run_down(shape, moe::kLayoutTwoSeg, h, kp, capacity, pad + n, mtile, w_down,
                       cr.vals, status, at<uint32_t>(ws, L.flags), stream, cr.codes, cr.part,
                       cr.slots, ovf));
    else
      MOE_TRY(run_down(shape, moe::kLayoutTwoSeg, h, kp, capacity, pad + n, mtile, w_down,
                       y_rows, status, at<uint32_t>(ws, L.flags), stream, nullptr, nullptr, 0,
                       ovf));
  } else {
    // first round: the padded rows, masked layout with M_max = C
    if (capacity > 0) {
      MOE_TRY(cuda_status(moe::launch_ffn_tiles(kp, MOE_LAYOUT_MASKED, s.E, capacity,
                                                tile_rows_for(shape, MOE_LAYOUT_MASKED, capacity),
                                                mtile, status, stream, nullptr,
                                                at<uint32_t>(ws, L.flags))));
      MOE_TRY(run_gate_up(shape, MOE_LAYOUT_MASKED, x_rows, kp, capacity, pad, mtile, w_gate_up,
                          h, status, stream));
      if (cr.vals)
        MOE_TRY(run_down(shape, MOE_LAYOUT_MASKED, h, kp, capacity, pad, mtile, w_down, cr.vals,
                         status, at<uint32_t>(ws, L.flags), stream, cr.codes, cr.part, cr.slots));
      else
        MOE_TRY(run_down(shape, MOE_LAYOUT_MASKED, h, kp, capacity, pad, mtile, w_down, y_rows,
                         status, at<uint32_t>(ws, L.flags), stream));
    }
    // second round: the overflow rows, contiguous with offsets ovf_offsets
    if (overflow == MOE_OVERFLOW_SECOND_ROUND) {
      MOE_TRY(cuda_status(moe::launch_ffn_tiles(ovf, MOE_LAYOUT_CONTIGUOUS, s.E, 0,
                                                tile_rows_for(shape, MOE_LAYOUT_CONTIGUOUS, 0),
                                                mtile, status, stream, nullptr,
                                                at<uint32_t>(ws, L.flags))));
      MOE_TRY(run_gate_up(shape, MOE_LAYOUT_CONTIGUOUS, x_rows + pad * s.d * 2, ovf, 0, n, mtile,
                          w_gate_up, h, status, stream));
      if (cr.vals)
        MOE_TRY(run_down(shape, MOE_LAYOUT_CONTIGUOUS, h, ovf, 0, n, mtile, w_down,
                         static_cast<uint8_t *>(cr.vals) + pad * s.d * 2, status,
                         at<uint32_t>(ws, L.flags), stream, cr.codes + pad * (s.d / 32),
                         cr.part, cr.slots));
      else
        MOE_TRY(run_down(shape, MOE_LAYOUT_CONTIGUOUS, h, ovf, 0, n, mtile, w_down,
                         y_rows + pad * s.d, status, at<uint32_t>(ws, L.flags), stream));
    }
  }
  if (cr.vals)
    return cuda_status(moe::launch_combine16(cr.vals, cr.codes, pad + n, dest, w, s.T, s.k, s.d,
                                             y, stream));
  return cuda_status(moe::launch_combine(y_rows, pad + n, dest, w, s.T, s.k, s.d, y, stream));
}

int64_t moe_layer_yperm_row_bytes(const moe_shape_t *shape) {
  if (check_shape(shape) != MOE_OK) return 0;
  if (compact_rows(*shape)) return 2 * int64_t{shape->d} + shape->d / 32;
  return 4 * int64_t{shape->d};
}

int32_t moe_layer_launch_count(const moe_shape_t *shape) {
  if (check_shape(shape) != MOE_OK || shape->T == 0) return 0;
  // router (screened: 5; else logits 1 or 2 + select), count, scan,
  // scatter, gather, gate_up, down, combine
  return moe::router_launches(shape->T, shape->d, shape->E, shape->G, shape->k) + 7;
}

moe_status_t moe_route_refined_count(const moe_shape_t *shape, const void *ws, size_t ws_bytes,
                                     int32_t *count, moe_stream_t stream) {
  MOE_TRY(check_shape(shape));
  if (!count) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*shape, 0);
  MOE_TRY(check_ws(const_cast<void *>(ws), ws_bytes, L.end_route));
  const int32_t *src = moe::router_refined_count(at<void>(const_cast<void *>(ws), L.wr32),
                                                 shape->T, shape->d, shape->E, shape->G,
                                                 shape->k);
  if (!src) return cuda_status(cudaMemsetAsync(count, 0xff, sizeof(int32_t), stream));
  return cuda_status(cudaMemcpyAsync(count, src, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                     stream));
}

moe_status_t moe_router_prep_size(const moe_shape_t *shape, size_t *bytes) {
  MOE_TRY(check_shape(shape));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const moe_shape_t &s = *shape;
  if (!moe::router_screened(s.T > 0 ? s.T : 1, s.d, s.E, s.G, s.k)) return MOE_ERR_UNSUPPORTED;
  *bytes = moe::router_prep_bytes(s.d, s.E);
  return MOE_OK;
}

moe_status_t moe_router_prepare(const moe_shape_t *shape, const void *w_r, void *prep,
                                size_t prep_bytes, moe_stream_t stream) {
  size_t need = 0;
  MOE_TRY(moe_router_prep_size(shape, &need));
  if (!w_r || !aligned16(w_r) || !prep || (reinterpret_cast<uintptr_t>(prep) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  if (prep_bytes < need) return MOE_ERR_WORKSPACE;
  // drop the old record first: until the new one is in, calls make their own copy
  moe::router_release_prepared(w_r);
  MOE_TRY(cuda_status(moe::launch_router_prepare(w_r, shape->d, shape->E, prep, stream)));
  if (!moe::router_register_prepared(w_r, shape->d, shape->E, prep)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t moe_router_release(const void *w_r) {
  if (!w_r) return MOE_ERR_INVALID_ARG;
  moe::router_release_prepared(w_r);
  return MOE_OK;
}

moe_status_t moe_selftest_wait_timeout(void *ws, size_t ws_bytes, uint64_t limit_ns,
                                       moe_stream_t stream) {
  MOE_TRY(check_ws(ws, ws_bytes, 4));
  return cuda_status(moe::launch_wait_selftest(at<uint32_t>(ws, 0), limit_ns, stream));
}

}  // extern "C"

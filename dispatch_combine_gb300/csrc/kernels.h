// kernels.h -- host-side launchers of the MoE kernels (internal to libmoe).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// router.cu
// w_scratch: router_scratch_bytes(T, d, E) bytes of workspace (a zero-padded
// copy of w_r for launch_router_logits; the transposed copy, the token list
// and the GEMM tile table for launch_router)
size_t router_scratch_bytes(int T, int d, int E);
// kernels launch_router_logits launches (1: weights resident; 2: padded copy + tiled)
int router_logits_launches(int d, int E);
cudaError_t launch_router_logits(const void *x, const void *w_r, int T, int d, int E,
                                 float *logits, void *w_scratch, cudaStream_t s);
// mode 0: scores from logits (score kind); mode 1: the input already holds
// selection scores (group top-k only; weights not written).
cudaError_t launch_router_select(const float *logits, const float *bias, int T, int E, int G,
                                 int topk_group, int k, int score, float bias_scale, int mode,
                                 int32_t *ids, float *weights, cudaStream_t s);
// experts per lane of the warp-per-token selection (0: the general kernel)
int router_select_per(int E, int G);

// route_screen.cu
// Routing without a logits output: ids [T,k] and weights [T,k], the same
// values as launch_router_logits + launch_router_select.  Where the shape
// allows (router_screened) the logits come from the tensor cores, every
// score gets an interval that provably holds its fixed-order value, and only
// the experts those intervals leave undecided get their fixed-order logit;
// logits [T,E] is then unused.  status receives the GEMM's wait errors.
bool router_screened(int T, int d, int E, int G, int k);
int router_launches(int T, int d, int E, int G, int k);
size_t screened_scratch_bytes(int T, int d, int E);
cudaError_t launch_router(const void *x, const void *w_r, const float *bias, int T, int d, int E,
                          int G, int topk_group, int k, int score, float bias_scale,
                          float *logits, int32_t *ids, float *weights, void *w_scratch,
                          uint32_t *status, cudaStream_t s);
// The screened path's copy of the router weight: transposed to [E, d], then
// the norms of the columns, router_prep_bytes(d, E) bytes.  A copy made by
// launch_router_prepare into a caller buffer and registered for w_r is used
// by every launch_router call with that w_r (and d, E) instead of one made
// in the scratch on each call.
size_t router_prep_bytes(int d, int E);
cudaError_t launch_router_prepare(const void *w_r, int d, int E, void *prep, cudaStream_t s);
bool router_register_prepared(const void *w_r, int d, int E, void *prep);
bool router_release_prepared(const void *w_r);
// (token, expert) pairs the last screened launch_router call on this scratch
// refined (device int; nullptr when the shape is not screened)
const int32_t *router_refined_count(const void *w_scratch, int T, int d, int E, int G, int k);

// dispatch.cu
// Assignments per dispatch chunk: 128 up to 32768 assignments (enough chunks
// to spread the ordered scatter over many warps), 512 above.
inline int dispatch_chunk(int64_t n) { return n <= 32768 ? 128 : 512; }
inline int64_t dispatch_num_chunks(int64_t n) {
  const int c = dispatch_chunk(n);
  return (n + c - 1) / c;
}
// Capacity variant of the dispatch: kept == nullptr turns it off.  With it,
// expert e keeps its first `capacity` assignments (in increasing t*k+j) in
// padded rows e*capacity + r; later ones go to overflow rows
// E*capacity + ovf_offsets[e] + (r - capacity) (second round) or nowhere,
// dest = -1 (drop).  kept[e] = min(n_e, capacity), ovf_offsets [E+1].
struct CapacityArgs {
  int capacity;
  int policy;  // moe_overflow_t
  int E;       // set by launch_dispatch
  int32_t *kept;
  int32_t *ovf_offsets;
};
// x_perm-style gather of byte rows (row_bytes a multiple of 16) and,
// optionally, of per-row fp32 scales: row t of src goes to the rows
// dest[t*k + j] < min(n, *offsets_end) of its valid assignments (ids in
// [0, E)); scales by src_token: dst_scale[p] = src_scale[src_token[p]]
cudaError_t launch_gather_rows(const void *src, int row_bytes, const float *src_scale,
                               int scales_per_row, const int32_t *ids, const int32_t *dest,
                               int k, int E, const int32_t *src_token,
                               const int32_t *offsets_end, int64_t n, int T, void *dst,
                               float *dst_scale, cudaStream_t s);
cudaError_t launch_dispatch(const int32_t *ids, int T, int k, int E, const void *x, int d,
                            int32_t *counts, int32_t *offsets, int32_t *src_token,
                            int32_t *dest, void *x_perm, int32_t *chunk_scratch,
                            int32_t *mtile_base, int tile_rows, uint32_t *status,
                            cudaStream_t s, CapacityArgs cap = CapacityArgs{0, 0, 0, nullptr, nullptr},
                            uint32_t *zero_flags = nullptr);
// Dispatch onto physical expert copies: phys_expert [P] is the logical
// expert of each physical slot; the r-th assignment (increasing a) of expert
// e goes to its copy r mod n_rep(e), copies in slot order.  Outputs
// counts_phys [P], offsets_phys [P+1], dest [T*k], src_token [T*k] and the
// gathered rows.  Scratch (device, caller-owned) as listed.
struct ReplicaScratch {
  int32_t *chunk;        // dispatch chunk histograms [chunks * E]
  int32_t *counts_log;   // [E]
  int32_t *offsets_log;  // [E+1]
  int32_t *mtile;        // [E+1]
  int32_t *dest_log;     // [T*k]
  int32_t *src_log;      // [T*k]
  int32_t *n_rep;        // [E]
  int32_t *rep_first;    // [E+1]
  int32_t *rep_slots;    // [P]
  int32_t *slot_rank;    // [P]
};
cudaError_t launch_dispatch_replicated(const int32_t *ids, int T, int k, int E, const void *x,
                                       int d, int P, const int32_t *phys_expert,
                                       int32_t *counts_phys, int32_t *offsets_phys,
                                       int32_t *src_token, int32_t *dest, void *x_perm,
                                       const ReplicaScratch &w, uint32_t *status,
                                       cudaStream_t s);
// Internal layout of the capacity layer's two rounds in one launch: expert e
// has the rows of its padded slab, [e * M_max, e * M_max + seg[e]) (seg =
// kept counts, clamped to M_max), then its overflow rows, [pad + seg2[e],
// pad + seg2[e + 1]) (seg2 = overflow offsets [E+1], pad = E * M_max); its
// m-tiles cover the slab's rows first, then the overflow rows.
constexpr int kLayoutTwoSeg = 2;
// mtile_base[e] = sum_{e'<e} ceil(M_e'/tile_rows) for the contiguous (seg =
// offsets) or masked (seg = masked_m, clamped to M_max) layout; for
// kLayoutTwoSeg the tiles of both of an expert's segments (seg2 as above).
// zero_flags (launch_ffn_tiles and launch_dispatch): kPairSplitFlagWords
// words set to zero (the down GEMM's split flags, so that every launch
// sequence, a replayed graph's too, starts with them clear); nullptr: none.
cudaError_t launch_ffn_tiles(const int32_t *seg, int layout, int E, int M_max, int tile_rows,
                             int32_t *mtile_base, uint32_t *status, cudaStream_t s,
                             const int32_t *seg2 = nullptr, uint32_t *zero_flags = nullptr);
// Expert GEMMs run on CTA pairs with 256-row tiles when the average number
// of rows per expert reaches this.  A full pair tile moves half the B bytes
// per FLOP through each SM's shared memory, which bounds the single-CTA
// 128x256 tile (about 1.2x faster on full tiles), and an expert's last tile
// of at most 128 rows runs swapped, costing about its weight bytes.  Below
// this most tiles are such tails, and the single-CTA kernel already streams
// the weights at HBM speed.
constexpr int64_t kPairRowsPerExpert = 256;
// rows of a 1-CTA GEMM tile (the unit mtile_base counts when pair is false)
constexpr int kGemmTileRows = 128;
// The CTA-pair down GEMM splits the tiles of its last, partial wave into two
// K halves on two pairs when the whole launch is at most kPairSplitMaxWaves
// waves and the halves fit in one wave.  Per 32-row slab the two halves
// share a ticket word and a ready word: the half that takes the ticket first
// (an exchange with a value that differs from launch to launch) stores its
// partial sums and raises ready; the other waits for ready (bounded, on a
// warp that is already storing) and adds its sums with fp32 reductions (one
// add per element, so the result does not depend on which came first), then
// clears both words.  Flags: kPairSplitSlots tiles x 8 slabs x 2 words.
constexpr int kPairSplitMaxWaves = 16;
constexpr int kPairSplitSlots = 256;
constexpr int kPairSplitFlagWords = kPairSplitSlots * 16;

// quant.cu: e4m3 codes with fp32 scales, per (row, 128 columns) of [rows,
// cols] bf16, or per 128 x 128 block of [mats, rows, cols] bf16
cudaError_t launch_quantize_rows_fp8(const void *x, int64_t rows, int cols, void *q,
                                     float *scales, cudaStream_t s);
cudaError_t launch_quantize_blocks_fp8(const void *w, int mats, int rows, int cols, void *q,
                                       float *scales, cudaStream_t s);

// combine.cu
// y[t] = sum_j w[t,j] * y_perm[dest[t*k+j]]; rows outside [0, y_rows) add nothing
cudaError_t launch_combine(const float *y_perm, int64_t y_rows, const int32_t *dest,
                           const float *w, int T, int k, int d, void *y, cudaStream_t s);
// the same from the compact rows (fp16 values y16 [y_rows, d], code bytes
// [y_rows, d / 32]; d a multiple of 32)
cudaError_t launch_combine16(const void *y16, const uint8_t *codes, int64_t y_rows,
                             const int32_t *dest, const float *w, int T, int k, int d, void *y,
                             cudaStream_t s);

// gemm.cu
struct GemmProblem {
  int E;
  int K;                     // reduction length (d for gate_up, inter for down)
  int n_out;                 // output columns (inter for gate_up, d for down)
  int layout;                // 0 contiguous, 1 masked, kLayoutTwoSeg
  const int32_t *seg;        // offsets [E+1] or masked_m [E] (kept counts for kLayoutTwoSeg)
  const int32_t *seg2;       // kLayoutTwoSeg: overflow offsets [E+1] (rows after E * M_max)
  int M_max;                 // masked slab rows
  int64_t rows_total;        // rows of A / out (T*k or E*M_max)
  const int32_t *mtile_base; // [E+1]
  const void *a;             // [rows_total, K] bf16
  const void *b;             // [E, b_rows, K] bf16
  int b_rows;                // 2*inter (gate_up) or d (down)
  void *out;                 // bf16 h [rows, inter] or fp32 y [rows, d]
  uint32_t *status;
  uint64_t wait_limit_ns;
  bool pair;  // 256-row tiles on CTA pairs (mtile_base counts 256-row tiles)
  int bn;     // 1-CTA down form: output tile width 64, 128 or 256 (0: widest dividing n_out)
  int ksplit; // 1-CTA down form: K pieces per tile added into out, which must hold zeros (0, 1: none)
  // pair down form: kPairSplitFlagWords zeroed words; with them a short
  // last wave runs its tiles as two K halves (nullptr: never split)
  uint32_t *split_flags;
  // down, compact output (the layer's y16 form, common.cuh): out receives
  // fp16 values [rows_total, n_out], out_codes the code bytes [rows_total,
  // n_out / 32] (n_out a multiple of 256; the 1-CTA form without K pieces);
  // pair form: split_part holds split_part_slots x 256 x 256 floats for the
  // halves of split tiles (fewer slots: fewer tiles split).  nullptr: fp32.
  uint8_t *out_codes;
  float *split_part;
  int split_part_slots;
  // FP8 gate_up with 256-column tiles: out receives h's e4m3 codes [rows,
  // n_out] and out_h_scales its power-of-two scales [rows, n_out / 128], the
  // quantization of the bf16 h done in the epilogue (nullptr: bf16 h)
  float *out_h_scales;
};
cudaError_t launch_gemm_gate_up_swiglu(const GemmProblem &p, cudaStream_t s);
cudaError_t launch_gemm_down(const GemmProblem &p, cudaStream_t s);
// FP8 forms: p.a / p.b hold e4m3 codes; a_scale [rows_total, K/128] and
// b_scale [E, b_rows/128, K/128] fp32 block scales
cudaError_t launch_gemm_fp8_gate_up_swiglu(const GemmProblem &p, const float *a_scale,
                                           const float *b_scale, cudaStream_t s);
cudaError_t launch_gemm_fp8_down(const GemmProblem &p, const float *a_scale,
                                 const float *b_scale, cudaStream_t s);
// one CTA waits on an mbarrier nobody completes, bounded by limit_ns
cudaError_t launch_wait_selftest(uint32_t *status, uint64_t limit_ns, cudaStream_t s);

int num_sms();

// api.cu: the shape validation every entry point applies (MOE_OK or an error)
moe_status_t check_shape_for_abi(const moe_shape_t *shape);

}  // namespace moe

// router.cu -- gating: router logits in a fixed fp32 order, scores, and the
// group-limited top-k selection.
//
// "第十五章：多节点大模型推理" section 4.1: the model's gating picks the top-k
// logical experts from each token's hidden state.  "ep-deploy" handbook page,
// section "EPLB 与路由约束": DeepSeek-V3's 256 experts form 8 groups; a group is
// scored by the sum of its two best expert scores, the 4 best groups are kept
// and the 8 best experts inside them are chosen (score = sigmoid + 0.15-scaled
// per-expert bias in that page's simulation).
//
// Reproducibility: bf16 x bf16 products are exact in fp32, so the logit only
// depends on the summation order.  The order is fixed: "lane" l of 32 owns
// the 8-element chunks c with c mod 32 == l and sums their products in
// increasing index from +0; the 32 lane sums are combined by an xor butterfly
// (offsets 16, 8, 4, 2, 1).  exp is a Cody-Waite reduction plus a degree-7
// Taylor polynomial evaluated with fused multiply-adds, and every operation
// uses an explicit round-to-nearest intrinsic, so the routing decisions are
// reproducible bit for bit by any IEEE implementation of the same steps.
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "route_common.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// logits: a CUDA-core GEMM [T,d] x [d,E] whose K dimension is split in 32
// interleaved slices, each slice summed in order, then combined by a fixed
// pairwise tree.
//
// A "round" covers 256 consecutive inputs i: chunk c of the round (8 inputs
// i = 256r + 8c + j, j = 0..7) belongs to slice c.  The CTA tile is CT tokens
// x CE experts.  Warp w owns slices SW*w .. SW*w+SW-1 (SW = 32 / warps) for
// the whole tile: all lanes of a warp read the same slice's row at the same
// time (shared-memory broadcast), each lane owning LT tokens x LE experts.
// x sits in shared memory as fp32, W_r as bf16 (widened to fp32 pairs in
// registers: exact), so each round brings as few bytes as possible into the
// SM.  W_r tiles come from a zero-padded copy by cp.async, STAGES rounds
// deep; the next round's x tile is loaded into registers while the current
// round is computed; one barrier per round.  The multiply-adds are paired
// over adjacent experts with fma.rn.f32x2 (two IEEE fp32 fused multiply-adds
// per instruction, each rounded exactly as a scalar fma.rn); on this part the
// packed form holds half of the FMA pipe for two cycles, and the kernel runs
// near that ceiling (scalar-FMA layouts measured were issue-bound and not
// faster).  At the end the
// 32 slice sums of every output go through shared memory and are combined as
// s_l <- s_l + s_{l+off}, off = 16, 8, 4, 2, 1 -- the pairs of the xor
// butterfly, so the value equals lane 0's butterfly result.
// ---------------------------------------------------------------------------
constexpr int kRtStages = 3;

template <int LT, int LE, int CE, int NT>
struct RtCfg {
  static constexpr int NW = NT / 32;        // warps
  static constexpr int SW = 32 / NW;        // slices per warp
  static constexpr int EG = CE / LE;        // lane groups along experts
  static constexpr int TG = 32 / EG;        // lane groups along tokens
  static constexpr int CT = TG * LT;        // tokens per CTA
  static constexpr int XS = 8 * CT + 4;     // floats per slice, x tile
  static constexpr int WS = 8 * CE + 8;     // bf16 per slice, w tile
  static constexpr int XBYTES = 32 * XS * 4;
  static constexpr int STAGE = XBYTES + 32 * WS * 2;  // bytes per stage
  static constexpr int RED = 32 * CT * CE * 4;       // bytes of the final exchange
  static constexpr int SMEM = (kRtStages * STAGE > RED ? kRtStages * STAGE : RED);
  static constexpr int XCH = CT * 32 / NT;      // 16-byte x chunks per thread
  static constexpr int WCHUNKS = 256 * CE / 8;  // 16-byte w chunks per round
  static constexpr int WCH = (WCHUNKS + NT - 1) / NT;  // per thread
  static constexpr int OUT = (CT * CE + NT - 1) / NT;  // outputs reduced per thread
  static_assert(EG * TG == 32 && LE == 8 && (LT == 1 || LT == 2 || LT == 4), "lane tile");
  static_assert(NW * SW == 32, "slices");
  static_assert(XCH >= 1 && WCH >= 1 && CT % 8 == 0 && CE % 8 == 0, "tile shape");
  static_assert(STAGE % 16 == 0 && SMEM <= 227 * 1024, "shared memory");
};

// Padded bf16 copy of the router weight: rows rounded up to a whole round,
// columns to 64 experts, zeros outside [d, E).
__host__ __device__ inline int router_e_pad(int E) { return (E + 63) / 64 * 64; }
__host__ __device__ inline int router_d_pad(int d) { return (d + 255) / 256 * 256; }

__global__ void router_pad_kernel(const uint16_t *__restrict__ w_r, int d, int E,
                                  uint16_t *__restrict__ wp) {
  pdl_begin();
  const int ep = router_e_pad(E);
  const int64_t n = static_cast<int64_t>(router_d_pad(d)) * ep;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int i = static_cast<int>(q / ep), e = static_cast<int>(q % ep);
    wp[q] = (i < d && e < E) ? w_r[(size_t)i * E + e] : static_cast<uint16_t>(0);
  }
}

__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// fp32 pair (lo, hi) of a packed bf16 pair
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t v) {
  uint64_t r;
  asm("{\n\t.reg .b32 lo, hi;\n\tshl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xFFFF0000;\n\t"
      "mov.b64 %0, {lo, hi};\n\t}"
      : "=l"(r)
      : "r"(v));
  return r;
}

template <int LT, int LE, int CE, int NT>
__global__ void __launch_bounds__(NT, 1)
    router_logits_kernel(const __nv_bfloat16 *__restrict__ x, const uint16_t *__restrict__ wpad,
                         int T, int d, int E, float *__restrict__ logits) {
  pdl_begin();
  using C = RtCfg<LT, LE, CE, NT>;
  constexpr int SW = C::SW;
  extern __shared__ __align__(16) uint8_t rsm_raw[];
  const int t0 = blockIdx.x * C::CT;
  const int e0 = blockIdx.y * CE;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int tl = (lane / C::EG) * LT;  // first token of this lane
  const int el = (lane % C::EG) * LE;  // first expert of this lane
  const int rounds = (d + 255) / 256;
  const int ep = router_e_pad(E);
  const bool full_tokens = t0 + C::CT <= T;
  auto xbuf = [&](int st) { return reinterpret_cast<float *>(rsm_raw + st * C::STAGE); };
  auto wbuf = [&](int st) {
    return reinterpret_cast<uint16_t *>(rsm_raw + st * C::STAGE + C::XBYTES);
  };

  uint4 xr[C::XCH];

  // x chunk m of this thread: 8 chunks x 4 tokens per warp-sized group, so
  // that the scalar shared stores below hit 32 distinct banks
  auto x_coord = [&](int m, int &t, int &c) {
    const int q = tid + NT * m;
    const int g = q >> 5, l = q & 31;
    c = (g & 3) * 8 + (l & 7);
    t = (g >> 2) * 4 + (l >> 3);
  };
  auto load_x = [&](int r) {
    const bool full = full_tokens && (r + 1) * 256 <= d;
#pragma unroll
    for (int m = 0; m < C::XCH; ++m) {
      int t, c;
      x_coord(m, t, c);
      const int i0 = r * 256 + c * 8;
      if (full || (t0 + t < T && i0 < d))
        xr[m] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + t) * d + i0));
      else
        xr[m] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  auto store_x = [&](float *xs) {
#pragma unroll
    for (int m = 0; m < C::XCH; ++m) {
      int t, c;
      x_coord(m, t, c);
      float *dst = xs + c * C::XS + t;
      const uint4 v = xr[m];
      dst[0 * C::CT] = bf16lo(v.x);
      dst[1 * C::CT] = bf16hi(v.x);
      dst[2 * C::CT] = bf16lo(v.y);
      dst[3 * C::CT] = bf16hi(v.y);
      dst[4 * C::CT] = bf16lo(v.z);
      dst[5 * C::CT] = bf16hi(v.z);
      dst[6 * C::CT] = bf16lo(v.w);
      dst[7 * C::CT] = bf16hi(v.w);
    }
  };
  // w tile of round r: 256 rows x CE experts (bf16) of the padded copy; one
  // commit group per round (empty groups past the last round keep the count)
  auto issue_w = [&](int r) {
    if (r < rounds) {
      uint16_t *ws = wbuf(r % kRtStages);
#pragma unroll
      for (int m = 0; m < C::WCH; ++m) {
        const int q = tid + NT * m;
        if (C::WCHUNKS % NT != 0 && q >= C::WCHUNKS) break;
        const int ii = q / (CE / 8), ec = (q % (CE / 8)) * 8;
        cp_async_16(ws + (ii >> 3) * C::WS + (ii & 7) * CE + ec,
                    wpad + (size_t)(r * 256 + ii) * ep + e0 + ec);
      }
    }
    cp_async_commit();
  };

  // acc2[s][a][b]: slice SW*warp+s, token tl+a, experts el+2b and el+2b+1
  uint64_t acc2[SW][LT][LE / 2];
#pragma unroll
  for (int s4 = 0; s4 < SW; ++s4)
#pragma unroll
    for (int a = 0; a < LT; ++a)
#pragma unroll
      for (int b = 0; b < LE / 2; ++b) acc2[s4][a][b] = 0ull;

#pragma unroll
  for (int r = 0; r < kRtStages - 1; ++r) issue_w(r);
  load_x(0);
  store_x(xbuf(0));
  cp_async_wait<kRtStages - 2>();
  __syncthreads();
  for (int r = 0; r < rounds; ++r) {
    issue_w(r + kRtStages - 1);
    if (r + 1 < rounds) load_x(r + 1);
    const float *xs = xbuf(r % kRtStages);
    const uint16_t *ws = wbuf(r % kRtStages);
    float xv[2][LT];
    uint4 wv[2];
    // operands of step q = s * 8 + j: slice SW*warp + s, input j of its chunk
    auto ld = [&](int q, int slot) {
      const int c = SW * warp + (q >> 3), j = q & 7;
      const float *xp = xs + c * C::XS + j * C::CT + tl;
      if (LT == 4) {
        *reinterpret_cast<float4 *>(&xv[slot][0]) = *reinterpret_cast<const float4 *>(xp);
      } else if (LT == 2) {
        *reinterpret_cast<float2 *>(&xv[slot][0]) = *reinterpret_cast<const float2 *>(xp);
      } else {
        xv[slot][0] = *xp;
      }
      wv[slot] = *reinterpret_cast<const uint4 *>(ws + c * C::WS + j * CE + el);
    };
    ld(0, 0);
#pragma unroll
    for (int q = 0; q < 8 * SW; ++q) {
      if (q + 1 < 8 * SW) ld(q + 1, (q + 1) & 1);
      const uint4 w = wv[q & 1];
      const uint64_t wp[4] = {bf16x2_to_f32x2(w.x), bf16x2_to_f32x2(w.y), bf16x2_to_f32x2(w.z),
                              bf16x2_to_f32x2(w.w)};
#pragma unroll
      for (int a = 0; a < LT; ++a) {
        uint64_t xd;
        asm("mov.b64 %0, {%1, %1};" : "=l"(xd) : "f"(xv[q & 1][a]));
#pragma unroll
        for (int b = 0; b < LE / 2; ++b)
          asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[q >> 3][a][b]) : "l"(xd), "l"(wp[b]));
      }
    }
    if (r + 1 < rounds) store_x(xbuf((r + 1) % kRtStages));
    cp_async_wait<kRtStages - 2>();
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // exchange: red[slice][o], o = token * CE + expert (tile-relative)
  float *red = reinterpret_cast<float *>(rsm_raw);
#pragma unroll
  for (int s4 = 0; s4 < SW; ++s4)
#pragma unroll
    for (int a = 0; a < LT; ++a)
#pragma unroll
      for (int b = 0; b < LE / 2; ++b) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc2[s4][a][b]));
        float *dst = red + (size_t)(SW * warp + s4) * (C::CT * CE) + (tl + a) * CE + el + 2 * b;
        *reinterpret_cast<float2 *>(dst) = make_float2(lo, hi);
      }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < C::OUT; ++k) {
    const int o = tid + k * NT;
    if (o >= C::CT * CE) break;
    float v[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) v[l] = red[(size_t)l * (C::CT * CE) + o];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
      for (int l = 0; l < off; ++l) v[l] = __fadd_rn(v[l], v[l + off]);
    const int t = t0 + o / CE, e = e0 + o % CE;
    if (t < T && e < E) logits[(size_t)t * E + e] = v[0];
  }
}

// ---------------------------------------------------------------------------
// Small E (W_r fits in shared memory): a persistent kernel keeps all of W_r
// (bf16, d x EP) in shared memory and streams x.  Warp = TT tokens, lane =
// slice, so lane l sums the inputs of its chunks in order, exactly as above;
// the 32 slice sums meet in the xor butterfly.  W row i sits at
// i + (i / 8) rows of 16 bytes (EP = 8) -- one padding row per chunk -- so
// the 32 lanes, which read rows 8 apart, hit distinct banks.
// ---------------------------------------------------------------------------
constexpr int kSmallWarps = 8;
constexpr int kSmallTT = 1;  // tokens per warp
constexpr int kSmallPF = 4;  // rounds of x in flight per lane

template <int EP>
struct SmallCfg {
  static constexpr int ROWB = EP * 2;  // bytes per W row
  static constexpr int CHUNKB = 9 * ROWB;  // 8 rows + 1 padding row per chunk
};

// whole rounds of 32 chunks are staged (zeros past d), so every lane of the
// last round reads inside the buffer
__host__ inline size_t router_small_smem(int d, int EP) {
  const int chunks = (d + 255) / 256 * 32;
  return static_cast<size_t>(chunks) * 9 * EP * 2;
}

template <int EP>
__global__ void __launch_bounds__(kSmallWarps * 32)
    router_logits_small_kernel(const __nv_bfloat16 *__restrict__ x,
                               const uint16_t *__restrict__ w_r, int T, int d, int E,
                               float *__restrict__ logits) {
  pdl_begin();
  using C = SmallCfg<EP>;
  extern __shared__ __align__(16) uint8_t wsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunks = (d + 255) / 256 * 32;
  // stage W_r: chunk c, row j -> wsm + c * CHUNKB + j * ROWB; zeros for
  // experts >= E and inputs >= d
  // one thread per row of 8 experts: aligned full rows are copied
  // asynchronously (all in flight at once), the others through registers
  const bool vec = (E % 8) == 0;
  for (int q = threadIdx.x; q < chunks * 8 * (EP / 8); q += blockDim.x) {
    const int i = q / (EP / 8), e8 = (q % (EP / 8)) * 8;
    uint8_t *dst = wsm + (i >> 3) * C::CHUNKB + (i & 7) * C::ROWB + e8 * 2;
    if (i < d && vec && e8 + 8 <= E) {
      cp_async_16(dst, w_r + (size_t)i * E + e8);
      continue;
    }
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (i < d) {
      {
        uint16_t h[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) h[u] = (e8 + u < E) ? w_r[(size_t)i * E + e8 + u] : 0;
        v = make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                       h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
      }
    }
    *reinterpret_cast<uint4 *>(dst) = v;
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  const int rounds = (d + 255) / 256;
  const int groups = (T + kSmallTT - 1) / kSmallTT;
  for (int grp = blockIdx.x * kSmallWarps + warp; grp < groups;
       grp += gridDim.x * kSmallWarps) {
    const int t0 = grp * kSmallTT;
    float acc[kSmallTT][EP];
#pragma unroll
    for (int a = 0; a < kSmallTT; ++a)
#pragma unroll
      for (int e = 0; e < EP; ++e) acc[a][e] = 0.0f;
    // ring of kSmallPF rounds of this lane's x chunks
    uint4 xr[kSmallPF][kSmallTT];
    auto load = [&](int r, int slot) {
      const int i0 = r * 256 + lane * 8;
#pragma unroll
      for (int a = 0; a < kSmallTT; ++a)
        xr[slot][a] =
            (r < rounds && t0 + a < T && i0 < d)
                ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + a) * d + i0))
                : make_uint4(0u, 0u, 0u, 0u);
    };
#pragma unroll
    for (int u = 0; u < kSmallPF; ++u) load(u, u);
    for (int r0 = 0; r0 < rounds; r0 += kSmallPF) {
#pragma unroll
      for (int u = 0; u < kSmallPF; ++u) {
        const int r = r0 + u;
        if (r < rounds) {
          float xv[kSmallTT][8];
#pragma unroll
          for (int a = 0; a < kSmallTT; ++a) {
            const uint4 v = xr[u][a];
            xv[a][0] = bf16lo(v.x); xv[a][1] = bf16hi(v.x);
            xv[a][2] = bf16lo(v.y); xv[a][3] = bf16hi(v.y);
            xv[a][4] = bf16lo(v.z); xv[a][5] = bf16hi(v.z);
            xv[a][6] = bf16lo(v.w); xv[a][7] = bf16hi(v.w);
          }
          load(r + kSmallPF, u);
          const uint8_t *wc = wsm + (r * 32 + lane) * C::CHUNKB;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float wv[EP];
#pragma unroll
            for (int e8 = 0; e8 < EP / 8; ++e8) {
              const uint4 w = *reinterpret_cast<const uint4 *>(wc + j * C::ROWB + e8 * 16);
              wv[e8 * 8 + 0] = bf16lo(w.x); wv[e8 * 8 + 1] = bf16hi(w.x);
              wv[e8 * 8 + 2] = bf16lo(w.y); wv[e8 * 8 + 3] = bf16hi(w.y);
              wv[e8 * 8 + 4] = bf16lo(w.z); wv[e8 * 8 + 5] = bf16hi(w.z);
              wv[e8 * 8 + 6] = bf16lo(w.w); wv[e8 * 8 + 7] = bf16hi(w.w);
            }
#pragma unroll
            for (int a = 0; a < kSmallTT; ++a)
#pragma unroll
              for (int e = 0; e < EP; ++e) acc[a][e] = __fmaf_rn(xv[a][j], wv[e], acc[a][e]);
          }
        }
      }
    }
#pragma unroll
    for (int a = 0; a < kSmallTT; ++a)
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        float v = acc[a][e];
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
        acc[a][e] = v;
      }
#pragma unroll
    for (int a = 0; a < kSmallTT; ++a)
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (((a * EP + e) & 31) == lane && t0 + a < T && e < E)
          logits[(size_t)(t0 + a) * E + e] = acc[a][e];
  }
}

template <int EP>
cudaError_t run_logits_small(const void *x, const void *w_r, int T, int d, int E,
                             float *logits, cudaStream_t s) {
  const size_t smem = router_small_smem(d, EP);
  auto kern = router_logits_small_kernel<EP>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int groups = (T + kSmallTT - 1) / kSmallTT;
  const int want = (groups + kSmallWarps - 1) / kSmallWarps;
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSmallWarps * 32, smem);
  if (per_sm < 1) per_sm = 1;
  const int cap = num_sms() * per_sm;
  const int grid = want < cap ? want : cap;
  MOE_LAUNCH_PDL(kern, grid, kSmallWarps * 32, smem, s, static_cast<const __nv_bfloat16 *>(x),
                                            static_cast<const uint16_t *>(w_r), T, d, E, logits);
  return cudaGetLastError();
}

template <int LT, int LE, int CE, int NT>
cudaError_t run_logits(const void *x, const uint16_t *wpad, int T, int d, int E, float *logits,
                       cudaStream_t s) {
  using C = RtCfg<LT, LE, CE, NT>;
  auto kern = router_logits_kernel<LT, LE, CE, NT>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  dim3 grid((T + C::CT - 1) / C::CT, (E + CE - 1) / CE);
  MOE_LAUNCH_PDL(kern, grid, NT, C::SMEM, s, static_cast<const __nv_bfloat16 *>(x), wpad, T, d, E, logits);
  return cudaGetLastError();
}

constexpr int kSelWarps = 8;

// One warp per token.  Lane l holds experts l, l+32, ... (E <= 1024).
__global__ void __launch_bounds__(kSelWarps * 32)
    router_select_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T,
                         int E, int G, int topk_group, int k, int score, float bias_scale,
                         int mode, int32_t *__restrict__ ids, float *__restrict__ weights,
                         const int32_t *__restrict__ list, const int32_t *__restrict__ count) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
  if (list) {
    if (t >= *count) return;
    t = list[t];
  }
  if (t >= T) return;
  const float *lt = logits + (size_t)t * E;
  const int per = (E + 31) >> 5;
  const float kNegInf = -__int_as_float(0x7f800000);

  float s[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    s[m] = kNegInf;
    const int e = lane + 32 * m;
    if (m < per && e < E) {
      const float l = lt[e];
      if (mode == 1 || score == MOE_SCORE_SOFTMAX)
        s[m] = l;
      else
        s[m] = __fadd_rn(canon_sigmoid(l), __fmul_rn(bias_scale, bias[e]));
    }
  }

  // eligibility from the group step
  uint32_t eligible = 0;
  if (G > 1) {
    const int gs = E / G;
    float gval = kNegInf;
    for (int g = 0; g < G; ++g) {
      float m1 = kNegInf, m2 = kNegInf;
#pragma unroll
      for (int m = 0; m < 32; ++m) {
        const int e = lane + 32 * m;
        if (m < per && e < E && e >= g * gs && e < (g + 1) * gs) {
          const float v = s[m];
          if (v > m1) {
            m2 = m1;
            m1 = v;
          } else if (v > m2) {
            m2 = v;
          }
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const float o1 = __shfl_xor_sync(0xffffffffu, m1, off);
        const float o2 = __shfl_xor_sync(0xffffffffu, m2, off);
        if (m1 >= o1) {
          m2 = fmaxf(m2, o1);
        } else {
          m2 = fmaxf(m1, o2);
          m1 = o1;
        }
      }
      const float gsum = (gs >= 2) ? __fadd_rn(m1, m2) : m1;
      if (lane == g) gval = gsum;
    }
    uint32_t kept = 0;
    bool mine_kept = false;
    for (int r = 0; r < topk_group; ++r) {
      float v = (lane < G && !mine_kept) ? gval : kNegInf;
      int idx = (lane < G && !mine_kept) ? lane : 0x7fffffff;
      warp_argmax(v, idx);
      if (lane == idx) mine_kept = true;
      kept |= 1u << idx;
    }
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      const int e = lane + 32 * m;
      if (m < per && e < E && ((kept >> (e / gs)) & 1u)) eligible |= 1u << m;
    }
  } else {
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      const int e = lane + 32 * m;
      if (m < per && e < E) eligible |= 1u << m;
    }
  }

  // top-k among eligible experts
  int my_id = -1;
  for (int j = 0; j < k; ++j) {
    float bv = kNegInf;
    int bi = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      if ((eligible >> m) & 1u) {
        if (s[m] > bv || bi == 0x7fffffff) {
          bv = s[m];
          bi = lane + 32 * m;
        }
      }
    }
    warp_argmax(bv, bi);
    if ((bi & 31) == lane) eligible &= ~(1u << (bi >> 5));
    if (lane == j) my_id = bi;
  }

  if (lane < k) ids[(size_t)t * k + lane] = my_id;
  if (mode == 1) return;

  // weights: renormalised sigmoid (bias excluded) or renormalised softmax
  const float l0 = __shfl_sync(0xffffffffu, (lane < k) ? lt[my_id] : 0.0f, 0);
  float v = 0.0f;
  if (lane < k) {
    const float l = lt[my_id];
    v = (score == MOE_SCORE_SOFTMAX) ? canon_exp(__fsub_rn(l, l0)) : canon_sigmoid(l);
  }
  float sum = __shfl_sync(0xffffffffu, v, 0);
  for (int j = 1; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, v, j));
  if (lane < k) weights[(size_t)t * k + lane] = __fdiv_rn(v, sum);
}

// Fast path of the selection: lane l holds the PER consecutive experts
// l*PER .. l*PER+PER-1, so a group of gs experts spans gs/PER lanes and all
// groups' top-2 reduce at once; a group's rank (how many groups beat it,
// ties to the lower index) comes from G independent broadcasts.  Same
// decisions as router_select_kernel; requires G == 1 or gs a power-of-two
// multiple of PER.
template <int PER>
__global__ void __launch_bounds__(kSelWarps * 32)
    router_select_fast_kernel(const float *__restrict__ logits, const float *__restrict__ bias,
                              int T, int E, int G, int topk_group, int k, int score,
                              float bias_scale, int mode, int32_t *__restrict__ ids,
                              float *__restrict__ weights, const int32_t *__restrict__ list,
                              const int32_t *__restrict__ count) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
  if (list) {
    if (t >= *count) return;
    t = list[t];
  }
  if (t >= T) return;
  const float *lt = logits + (size_t)t * E;
  const float kNegInf = -__int_as_float(0x7f800000);
  const int e0 = lane * PER;

  float s[PER];
#pragma unroll
  for (int m = 0; m < PER; ++m) {
    const int e = e0 + m;
    s[m] = kNegInf;
    if (e < E) {
      const float l = lt[e];
      if (mode == 1 || score == MOE_SCORE_SOFTMAX)
        s[m] = l;
      else
        s[m] = __fadd_rn(canon_sigmoid(l), __fmul_rn(bias_scale, bias[e]));
    }
  }
  uint32_t eligible = 0;
#pragma unroll
  for (int m = 0; m < PER; ++m)
    if (e0 + m < E) eligible |= 1u << m;

  if (G > 1) {
    const int gs = E / G;
    const int lpg = gs / PER;  // lanes per group (power of two)
    float m1 = kNegInf, m2 = kNegInf;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const float v = s[m];
      if (v > m1) {
        m2 = m1;
        m1 = v;
      } else if (v > m2) {
        m2 = v;
      }
    }
    for (int off = 1; off < lpg; off <<= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, m1, off);
      const float o2 = __shfl_xor_sync(0xffffffffu, m2, off);
      if (m1 >= o1) {
        m2 = fmaxf(m2, o1);
      } else {
        m2 = fmaxf(m1, o2);
        m1 = o1;
      }
    }
    const float mine = (gs >= 2) ? __fadd_rn(m1, m2) : m1;
    const int my_group = (e0 < E) ? e0 / gs : G;
    int rank = 0;
    for (int g = 0; g < G; ++g) {
      const float o = __shfl_sync(0xffffffffu, mine, g * lpg);
      rank += (o > mine || (o == mine && g < my_group)) ? 1 : 0;
    }
    if (my_group >= G || rank >= topk_group) eligible = 0;
  }

  int my_id = -1;
  for (int j = 0; j < k; ++j) {
    float bv = kNegInf;
    int bi = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      if ((eligible >> m) & 1u) {
        if (s[m] > bv || bi == 0x7fffffff) {
          bv = s[m];
          bi = e0 + m;
        }
      }
    }
    warp_argmax(bv, bi);
    if (bi != 0x7fffffff && bi / PER == lane) eligible &= ~(1u << (bi - e0));
    if (lane == j) my_id = bi;
  }

  if (lane < k) ids[(size_t)t * k + lane] = my_id;
  if (mode == 1) return;
  const float l0 = __shfl_sync(0xffffffffu, (lane < k) ? lt[my_id] : 0.0f, 0);
  float v = 0.0f;
  if (lane < k) {
    const float l = lt[my_id];
    v = (score == MOE_SCORE_SOFTMAX) ? canon_exp(__fsub_rn(l, l0)) : canon_sigmoid(l);
  }
  float sum = __shfl_sync(0xffffffffu, v, 0);
  for (int j = 1; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, v, j));
  if (lane < k) weights[(size_t)t * k + lane] = __fdiv_rn(v, sum);
}

}  // namespace

// experts per lane of the fast selection (0: the general kernel is needed)
int router_select_per(int E, int G) {
  int per = 1;
  while (per * 32 < E) per *= 2;
  if (per > 32) return 0;
  if (G > 1) {
    const int gs = E / G;
    const int lpg = gs / per;
    if (!(gs % per == 0 && lpg >= 1 && lpg <= 32 && (lpg & (lpg - 1)) == 0)) return 0;
  }
  return per;
}

size_t router_scratch_bytes(int T, int d, int E) {
  const size_t pad = static_cast<size_t>(router_d_pad(d)) * router_e_pad(E) * sizeof(uint16_t);
  const size_t scr = screened_scratch_bytes(T, d, E);
  return pad > scr ? pad : scr;
}

// W_r resident in shared memory when it fits
constexpr size_t kSmallSmemMax = 200 * 1024;
bool router_resident(int d, int E) {
  return (E <= 8 && router_small_smem(d, 8) <= kSmallSmemMax) ||
         (E <= 16 && router_small_smem(d, 16) <= kSmallSmemMax);
}

int router_logits_launches(int d, int E) { return router_resident(d, E) ? 1 : 2; }

cudaError_t launch_router_logits(const void *x, const void *w_r, int T, int d, int E,
                                 float *logits, void *w_scratch, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (E <= 8 && router_small_smem(d, 8) <= kSmallSmemMax)
    return run_logits_small<8>(x, w_r, T, d, E, logits, s);
  if (E <= 16 && router_small_smem(d, 16) <= kSmallSmemMax)
    return run_logits_small<16>(x, w_r, T, d, E, logits, s);
  const int64_t n = static_cast<int64_t>(router_d_pad(d)) * router_e_pad(E);
  const int64_t want = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  uint16_t *wpad = static_cast<uint16_t *>(w_scratch);
  MOE_LAUNCH_PDL(router_pad_kernel, static_cast<unsigned>(want < cap ? want : cap), 256, 0, s, 
      static_cast<const uint16_t *>(w_r), d, E, wpad);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // tile shapes (tokens x experts): E <= 8: 32 x 8; <= 16: 32 x 16;
  // <= 32: 32 x 32; otherwise 16 x 64; 16 warps, 2 slices per warp
  if (E <= 8) return run_logits<1, 8, 8, 512>(x, wpad, T, d, E, logits, s);
  if (E <= 16) return run_logits<2, 8, 16, 512>(x, wpad, T, d, E, logits, s);
  if (E <= 32) return run_logits<4, 8, 32, 512>(x, wpad, T, d, E, logits, s);
  return run_logits<4, 8, 64, 512>(x, wpad, T, d, E, logits, s);
}

namespace {
cudaError_t select_impl(const float *logits, const float *bias, int T, int E, int G,
                        int topk_group, int k, int score, float bias_scale, int mode,
                        int32_t *ids, float *weights, const int32_t *list, const int32_t *count,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = (T + kSelWarps - 1) / kSelWarps;
  const int per = router_select_per(E, G);
  if (per != 0) {
#define MOE_SELECT_FAST(P)                                                                  \
  case P:                                                                                   \
    MOE_LAUNCH_PDL(router_select_fast_kernel<P>, grid, kSelWarps * 32, 0, s,                            \
        logits, bias, T, E, G, topk_group, k, score, bias_scale, mode, ids, weights, list,  \
        count);                                                                             \
    return cudaGetLastError();
    switch (per) {
      MOE_SELECT_FAST(1)
      MOE_SELECT_FAST(2)
      MOE_SELECT_FAST(4)
      MOE_SELECT_FAST(8)
      MOE_SELECT_FAST(16)
      MOE_SELECT_FAST(32)
      default:
        break;
    }
#undef MOE_SELECT_FAST
  }
  MOE_LAUNCH_PDL(router_select_kernel, grid, kSelWarps * 32, 0, s, logits, bias, T, E, G, topk_group, k,
                                                       score, bias_scale, mode, ids, weights,
                                                       list, count);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_router_select(const float *logits, const float *bias, int T, int E, int G,
                                 int topk_group, int k, int score, float bias_scale, int mode,
                                 int32_t *ids, float *weights, cudaStream_t s) {
  return select_impl(logits, bias, T, E, G, topk_group, k, score, bias_scale, mode, ids, weights,
                     nullptr, nullptr, s);
}


}  // namespace moe

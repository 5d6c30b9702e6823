// route_screen.cu -- screened routing: the router logits come from the tensor
// cores, every score is known to lie in an interval around its tensor-core
// estimate, and only the experts whose selection those intervals leave open
// get their logit in the fixed fp32 order.  The ids and weights equal those
// of the fixed-order router (router.cu) by construction.
//
// "第十五章：多节点大模型推理" section 4.1 (the gating picks the top-k
// experts) and the "ep-deploy" handbook page, section "EPLB 与路由约束"
// (groups of experts scored by the sum of their two best scores, the best
// groups kept, the top-k experts chosen inside them) define the selection;
// its logits are sums of exact bf16 x bf16 products whose order the fixed
// path pins down.
//
// The bound.  For a token t and expert e let S = sum_i |x_ti w_ie| <=
// ||x_t||_2 ||w_e||_2 (Cauchy-Schwarz).
//   * Tensor cores.  The logits GEMM restarts its TMEM accumulator every
//     kRsPK k-blocks, so every accumulation chain is n = 4 * kRsPK MMAs of 16
//     products; the chains are summed in fp32 (round to nearest) in a fixed
//     order.  The hardware's rounding inside an MMA is not documented; the
//     bound assumes only that one MMA adds its 16 exact products to its
//     accumulator with an error of at most beta = 2^-17 times the sum of the
//     magnitudes involved (|accumulator| + the 16 |products|) -- 64 units in
//     the last place of the largest of them, far above what any alignment-
//     and-truncate adder loses.  A chain then errs by at most
//     n beta (1 + beta)^n S_chain, and summing the c chains adds
//     gamma_{c-1} (gamma_m = m u / (1 - m u), u = 2^-24).
//   * Fixed order.  Each lane sums at most 8 ceil(d/256) products (the first
//     exactly), then 5 butterfly additions: gamma_{8 ceil(d/256) + 4} S.
//   So |l_tc - l_fixed| <= Lambda = alpha ||x_t|| ||w_e|| (alpha on the host,
//   with a factor 1 + 2^-8 for the rounding of the two norms).
// Scores: a sigmoid score moves by at most a quarter of its logit's move
// (the fixed exp/sigmoid evaluation adds at most 2^-18, its bias addition one
// rounding); a softmax score is the logit.  With eta the score half-width,
// [s_tc - eta, s_tc + eta] (directed rounding) holds the fixed-order score.
//
// Decisions from the intervals (one warp per token):
//   * group bounds: the sum of the two largest lower (upper) ends in the
//     group, rounded down (up) -- they hold the fixed-order group score,
//     which is the rounded sum of the group's two best scores;
//   * a group is certainly kept when fewer than topk_group other groups can
//     reach its lower bound, certainly dropped when topk_group others are
//     certainly above its upper bound, else ambiguous;
//   * the experts to refine: in each ambiguous group, every expert whose
//     upper end reaches the group's second-largest lower end (the group's
//     two best are among them); and every expert of a group not certainly
//     dropped whose upper end reaches theta, the k-th largest lower end
//     among experts of certainly kept groups (-inf if there are fewer).
// Then every expert that can be selected is refined, the group scores of
// ambiguous groups are exact, and the fixed-order selection is: the
// certainly kept groups plus the best ambiguous groups by exact score, then
// the top-k refined experts of the kept groups by exact score (ties to the
// lower index).  No second round is ever needed.
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "route_common.cuh"

namespace moe {
namespace {

// 2D bf16 tensor [rows, inner] row-major; box = box_rows x 64 elements,
// 128-byte swizzle, rows past the end read as zero.  cuTensorMapEncodeTiled
// is looked up through the runtime (the library does not link libcuda).
using RsEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
bool rs_make_tmap(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                  uint32_t box_rows) {
  static RsEncodeFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<RsEncodeFn>(p);
    return static_cast<RsEncodeFn>(nullptr);
  }();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kRsBM = 128;
constexpr int kRsBK = 64;
constexpr int kRsPK = 2;             // k-blocks per accumulation chain
constexpr double kTcBeta = 0x1p-17;  // per-MMA error model, see above
constexpr int kRsTargetItems = 128;  // GEMM work items aimed at (K split below it)
constexpr int kRsStageBudget = 196608;
constexpr int kRsRecHead = 4;  // need record: n, kept mask, ambiguous mask, spare

// ---------------------------------------------------------------------------
// scratch layout (inside the router scratch of the workspace)
// ---------------------------------------------------------------------------
size_t al256(size_t v) { return (v + 255) / 256 * 256; }

int rs_bn(int E) { return E % 256 == 0 ? 256 : E % 128 == 0 ? 128 : 64; }

int rs_ksplit(int T, int d, int E) {
  const int64_t mt = (T + kRsBM - 1) / kRsBM;
  const int64_t tiles = mt * (E / rs_bn(E));
  const int kb = d / kRsBK;
  int ks = 1;
  if (tiles < kRsTargetItems) {
    const int64_t by_items = kRsTargetItems / tiles;
    const int64_t by_k = kb / 8;  // at least 8 k-blocks (4 chains) per item
    ks = static_cast<int>(by_items < by_k ? by_items : by_k);
    if (ks < 1) ks = 1;
  }
  return ks;
}

struct RsLayout {
  size_t wt, wn, cnt, part, xn2, rec, end;
};

RsLayout rs_layout(int T, int d, int E) {
  RsLayout L;
  const int ks = rs_ksplit(T, d, E);
  size_t off = 0;
  L.wt = off;
  off = al256(off + static_cast<size_t>(E) * d * 2);
  L.wn = off;
  off = al256(off + static_cast<size_t>(E) * 4);
  L.cnt = off;
  off = al256(off + 16);
  L.part = off;
  off = al256(off + static_cast<size_t>(ks) * T * E * 4);
  L.xn2 = off;
  off = al256(off + static_cast<size_t>(ks) * T * 4);
  L.rec = off;
  off = al256(off + static_cast<size_t>(T) * (E + kRsRecHead) * 4);
  L.end = off;
  return L;
}

// gamma_m = m u / (1 - m u), u = 2^-24
double gamma_n(double m) {
  const double u = 0x1p-24;
  return m * u / (1.0 - m * u);
}

// alpha of the bound |l_tc - l_fixed| <= alpha ||x_t|| ||w_e||
double rs_alpha(int T, int d, int E) {
  const int kb = d / kRsBK;
  const int ks = rs_ksplit(T, d, E);
  int64_t chains = 0;
  for (int g = 0; g < ks; ++g) {
    const int lo = g * kb / ks, hi = (g + 1) * kb / ks;
    chains += (hi - lo + kRsPK - 1) / kRsPK;
  }
  const double n = 4.0 * kRsPK;  // MMAs per chain (K = 16 each)
  const double a_chain = n * kTcBeta * std::pow(1.0 + kTcBeta, n);
  const double a_tc = a_chain + gamma_n(static_cast<double>(chains - 1)) * (1.0 + a_chain);
  const double nch = d / 8.0;
  const double a_fixed = gamma_n(8.0 * std::ceil(nch / 32.0) + 4.0);
  return (a_tc + a_fixed) * (1.0 + 0x1p-8);
}

// ---------------------------------------------------------------------------
// prep: W_r [d, E] -> wt [E, d] (64 x 64 tiles through shared memory), then
// the squared norms of the rows of wt, one warp per expert (fixed order)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    rs_transpose_kernel(const uint16_t *__restrict__ w_r, int d, int E,
                        uint16_t *__restrict__ wt) {
  pdl_begin();
  __shared__ __align__(16) uint16_t tile[64][72];
  const int e0 = blockIdx.x * 64, i0 = blockIdx.y * 64;
  const int tid = threadIdx.x;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int q = tid + 256 * r;
    const int il = q >> 3, ch = q & 7;
    *reinterpret_cast<uint4 *>(&tile[il][ch * 8]) =
        __ldg(reinterpret_cast<const uint4 *>(w_r + (size_t)(i0 + il) * E + e0 + ch * 8));
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int q = tid + 256 * r;
    const int el = q & 63, ch = q >> 6;
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      h[j] = static_cast<uint32_t>(tile[ch * 8 + 2 * j][el]) |
             (static_cast<uint32_t>(tile[ch * 8 + 2 * j + 1][el]) << 16);
    *reinterpret_cast<uint4 *>(wt + (size_t)(e0 + el) * d + i0 + ch * 8) =
        make_uint4(h[0], h[1], h[2], h[3]);
  }
}

__global__ void __launch_bounds__(256)
    rs_wnorm_kernel(const uint16_t *__restrict__ wt, int d, int E, float *__restrict__ wn) {
  pdl_begin();
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (e >= E) return;
  const uint4 *row = reinterpret_cast<const uint4 *>(wt + (size_t)e * d);
  float acc = 0.0f;
  for (int c = lane; c < d / 8; c += 32) {
    float f[8];
    bf16x8_to_f32(__ldg(row + c), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = __fmaf_rn(f[i], f[i], acc);
  }
  acc = butterfly_sum(acc);
  if (lane == 0) wn[e] = __fsqrt_rn(acc);
}

// ---------------------------------------------------------------------------
// tensor-core logits.  Persistent CTAs over items (m-tile, n-tile, K group);
// warp 0: TMA producer (128 x 64 x-tile + BN x 64 wt-tile per stage, 128-byte
// swizzle); warp 1: MMA issuer (M = 128, N = BN, K = 16, two TMEM
// accumulators, a fresh accumulation every kRsPK k-blocks); warps 2-3: the
// squared norms of the tile's 128 x rows, read from the staged tiles (a
// stage is released when the MMAs and both norm warps are done with it);
// warps 4-11: epilogue, each a 32-lane quadrant x BN/2 columns, adding the
// chains in order in registers.  Each item stores its sums to its own K-group
// slice of part and xn2 (no atomics: the need kernel adds the slices in
// order).
// ---------------------------------------------------------------------------
constexpr int kRsThreads = 12 * 32;

template <int BN>
struct RsCfg {
  static constexpr int A_BYTES = kRsBM * kRsBK * 2;
  static constexpr int B_BYTES = BN * kRsBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = kRsStageBudget / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int COLS = BN / 2;  // columns per epilogue warp
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
  static_assert(STAGES >= 3, "pipeline depth");
  static_assert(TMEM_COLS <= 512, "TMEM columns");
};

struct RsArgs {
  int T, d, E, n_tiles, ksplit, items;
  float *part;   // [ksplit][T][E]
  float *xn2;    // [ksplit][T]
  int32_t *cnt;  // refined-pair counter of the call, zeroed here
  uint32_t *status;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ bool rs_wait_drain(uint64_t *bar, uint32_t parity,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

template <int BN>
__global__ void __launch_bounds__(kRsThreads, 1)
    rs_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const RsArgs args) {
  pdl_begin();
  using C = RsCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smem + C::STAGES * C::A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *tmem_full = bars + 2 * C::STAGES;
  uint64_t *tmem_empty = tmem_full + 2;
  uint64_t *drain = tmem_full + 4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) *args.cnt = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 3);  // MMA commit + the two norm warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 8);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (static_cast<int>(blockIdx.x) >= args.items) return;  // uniform across the CTA
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int kblocks = args.d / kRsBK;
  const int ks = args.ksplit;
  // item u: K group u % ks of tile u / ks; tile: n fastest
  auto item_m = [&](int u) { return (u / ks) / args.n_tiles; };
  auto item_n = [&](int u) { return (u / ks) % args.n_tiles; };
  auto kb_lo = [&](int u) { return (u % ks) * kblocks / ks; };
  auto kb_hi = [&](int u) { return (u % ks + 1) * kblocks / ks; };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      bool issued[C::STAGES];
      uint32_t issued_phase[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) issued[s] = false;
      for (int u = blockIdx.x; u < args.items && !*abort_flag; u += gridDim.x) {
        const int row0 = item_m(u) * kRsBM, b0 = item_n(u) * BN;
        for (int kb = kb_lo(u); kb < kb_hi(u); ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status,
                                 args.wait_limit_ns))
            break;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(smA + stage * C::A_BYTES, &tmA, &full[stage], kb * kRsBK, row0);
          tma_load_2d(smB + stage * C::B_BYTES, &tmB, &full[stage], kb * kRsBK, b0);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < C::STAGES; ++s)
        if (issued[s]) rs_wait_drain(&full[s], issued_phase[s], args.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = mma_idesc_bf16_f32(kRsBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool any_mma = false, ok = true;
      for (int u = blockIdx.x; u < args.items && ok && !*abort_flag; u += gridDim.x) {
        const int k0 = kb_lo(u), k1 = kb_hi(u);
        for (int c0 = k0; c0 < k1 && ok; c0 += kRsPK) {
          const int c1 = min(c0 + kRsPK, k1);
          if (!mbar_wait_bounded(&tmem_empty[acc], acc_phase ^ 1u, abort_flag, args.status,
                                 args.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
          for (int kb = c0; kb < c1; ++kb) {
            if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.status,
                                   args.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = sw128_kmajor_desc(smem_u32(smA + stage * C::A_BYTES));
            const uint64_t bd = sw128_kmajor_desc(smem_u32(smB + stage * C::B_BYTES));
#pragma unroll
            for (int kk = 0; kk < kRsBK / 16; ++kk)
              mma_bf16_ss(d_tmem, ad + 2u * kk, bd + 2u * kk, kIdesc,
                          (kb != c0 || kk != 0) ? 1u : 0u);
            any_mma = true;
            mma_commit(&empty[stage]);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(&tmem_full[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      if (any_mma) {
        mma_commit(drain);
        rs_wait_drain(drain, 0, args.wait_limit_ns);
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------- squared norms of the x rows ----------------
    // norm warp w covers rows 64 (w-2) .. +63: one 16-byte load of the warp
    // reads 4 whole rows (lanes 8 j .. 8 j + 7: row 4 i + j, its 8 chunks in
    // their swizzled order), so the loads are conflict-free; lane l keeps the
    // partial sums of its 16 rows, the 8 lanes of a row are added at the end
    // of the item (any order serves: the bound inflates the norm)
    const int rbase = (warp - 2) * 64 + (lane >> 3);
    const int chunk = lane & 7;
    int stage = 0;
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < args.items; u += gridDim.x) {
      float sq[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) sq[i] = 0.0f;
      bool ok = true;
      for (int kb = kb_lo(u); kb < kb_hi(u); ++kb) {
        const bool got = mbar_wait_bounded(&full[stage], phase, abort_flag, args.status,
                                           args.wait_limit_ns);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint4 *a = reinterpret_cast<const uint4 *>(smA + stage * C::A_BYTES);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float f[8];
          bf16x8_to_f32(a[(rbase + 4 * i) * 8 + chunk], f);
#pragma unroll
          for (int j = 0; j < 8; ++j) sq[i] = __fmaf_rn(f[j], f[j], sq[i]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        sq[i] = __fadd_rn(sq[i], __shfl_xor_sync(0xffffffffu, sq[i], 1));
        sq[i] = __fadd_rn(sq[i], __shfl_xor_sync(0xffffffffu, sq[i], 2));
        sq[i] = __fadd_rn(sq[i], __shfl_xor_sync(0xffffffffu, sq[i], 4));
      }
      if (item_n(u) == 0 && chunk == 0) {
        float *dst = args.xn2 + static_cast<int64_t>(u % ks) * args.T;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t g = static_cast<int64_t>(item_m(u)) * kRsBM + rbase + 4 * i;
          if (g < args.T) dst[g] = sq[i];
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 4..11) ----------------
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;
    const int row = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < args.items && ok; u += gridDim.x) {
      // the chains' sums in order (adding the first one to +0 is exact)
      float sum[C::COLS];
#pragma unroll
      for (int i = 0; i < C::COLS; ++i) sum[i] = 0.0f;
      const int k0 = kb_lo(u), k1 = kb_hi(u);
      for (int c0 = k0; c0 < k1; c0 += kRsPK) {
        const bool waited = mbar_wait_bounded(&tmem_full[acc], acc_phase, abort_flag,
                                              args.status, args.wait_limit_ns);
        if (!__all_sync(0xffffffffu, waited)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                            static_cast<uint32_t>(acc * BN + half * C::COLS);
#pragma unroll
        for (int c = 0; c < C::COLS / 16; ++c) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tb + c * 16, v);
          tmem_ld_wait();
          tmem_regs_fence16(v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            sum[c * 16 + i] = __fadd_rn(sum[c * 16 + i], __uint_as_float(v[i]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tmem_empty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) break;
      const int64_t grow = static_cast<int64_t>(item_m(u)) * kRsBM + row;
      if (grow < args.T) {
        float *dst = args.part + (static_cast<int64_t>(u % ks) * args.T + grow) * args.E +
                     item_n(u) * BN + half * C::COLS;
#pragma unroll
        for (int i = 0; i < C::COLS / 4; ++i)
          reinterpret_cast<float4 *>(dst)[i] =
              make_float4(sum[4 * i], sum[4 * i + 1], sum[4 * i + 2], sum[4 * i + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// selection with refinement: a need kernel (one warp per token) decides from
// the intervals which experts to refine; a refine kernel (one CTA per token)
// computes their fixed-order logits and makes the selection.
// ---------------------------------------------------------------------------

// decide which experts of token t to refine (warp-wide; lane owns experts
// lane*PER .. lane*PER+PER-1); writes the sorted list to need_out and
// returns its length; *kept_out / *amb_out get the group masks
template <int PER>
__device__ __forceinline__ int rs_decide(const float *__restrict__ part, float xnorm,
                                         const float *__restrict__ wn,
                                         const float *__restrict__ bias, int t, int T, int E,
                                         int G, int topk_group, int k, int score,
                                         float bias_scale, int ksplit, float alpha, int lane,
                                         int16_t *need_out, uint32_t *kept_out,
                                         uint32_t *amb_out) {
  const float kInf = __int_as_float(0x7f800000);
  const bool sig = score == MOE_SCORE_SIGMOID_BIAS;
  const int e0 = lane * PER;

  float lo[PER], hi[PER], lg[PER];
  // the K-group slices, added in order; four slices' values load together
#pragma unroll
  for (int m = 0; m < PER; ++m) lg[m] = (e0 + m < E) ? part[(size_t)t * E + e0 + m] : 0.0f;
  for (int g0 = 1; g0 < ksplit; g0 += 4) {
    float v[4][PER];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float *pg = part + ((size_t)(g0 + q) * T + t) * E;
#pragma unroll
      for (int m = 0; m < PER; ++m) v[q][m] = (g0 + q < ksplit && e0 + m < E) ? pg[e0 + m] : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (g0 + q < ksplit)
#pragma unroll
        for (int m = 0; m < PER; ++m) lg[m] = __fadd_rn(lg[m], v[q][m]);
  }
  const float ax = __fmul_ru(alpha, xnorm);
#pragma unroll
  for (int m = 0; m < PER; ++m) {
    const int e = e0 + m;
    lo[m] = -kInf;
    hi[m] = -kInf;
    if (e < E) {
      const float l = lg[m];
      const float lam = __fmaf_ru(ax, wn[e], 0x1p-40f);
      float sc, eta;
      if (sig) {
        const float c = __fmul_rn(bias_scale, bias[e]);
        sc = __fadd_rn(canon_sigmoid(l), c);
        eta = __fmaf_ru(0.25f, lam, __fmul_ru(0x1p-17f, __fadd_ru(1.0f, fabsf(c))));
      } else {
        sc = l;
        eta = __fadd_ru(lam, 0x1p-40f);
      }
      if (isfinite(sc) && isfinite(eta)) {
        lo[m] = __fsub_rd(sc, eta);
        hi[m] = __fadd_ru(sc, eta);
      } else {
        lo[m] = -kInf;  // an interval that holds every value: always refined
        hi[m] = kInf;
      }
    }
  }

  uint32_t possible = 0, certain = 0;  // experts (bits m) in groups not dropped / kept
  uint32_t need = 0;
  uint32_t kept_mask = 0, amb_mask = 0;
  if (G > 1) {
    const int gs = E / G;
    const int lpg = gs / PER;
    // the two largest lower and upper ends of the group
    float l1 = -kInf, l2 = -kInf, h1 = -kInf, h2 = -kInf;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      if (lo[m] > l1) {
        l2 = l1;
        l1 = lo[m];
      } else if (lo[m] > l2) {
        l2 = lo[m];
      }
      if (hi[m] > h1) {
        h2 = h1;
        h1 = hi[m];
      } else if (hi[m] > h2) {
        h2 = hi[m];
      }
    }
    for (int off = 1; off < lpg; off <<= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, l1, off);
      const float o2 = __shfl_xor_sync(0xffffffffu, l2, off);
      const float p1 = __shfl_xor_sync(0xffffffffu, h1, off);
      const float p2 = __shfl_xor_sync(0xffffffffu, h2, off);
      if (l1 >= o1) {
        l2 = fmaxf(l2, o1);
      } else {
        l2 = fmaxf(l1, o2);
        l1 = o1;
      }
      if (h1 >= p1) {
        h2 = fmaxf(h2, p1);
      } else {
        h2 = fmaxf(h1, p2);
        h1 = p1;
      }
    }
    const float glo = (gs >= 2) ? __fadd_rd(l1, l2) : l1;
    const float ghi = (gs >= 2) ? __fadd_ru(h1, h2) : h1;
    const int my_group = e0 / gs;
    int reach = 0, above = 0;  // groups that can reach my lower end / are surely above my upper end
    for (int g = 0; g < G; ++g) {
      const float olo = __shfl_sync(0xffffffffu, glo, g * lpg);
      const float ohi = __shfl_sync(0xffffffffu, ghi, g * lpg);
      if (g != my_group) {
        reach += (ohi >= glo) ? 1 : 0;
        above += (olo > ghi) ? 1 : 0;
      }
    }
    const bool ck = reach < topk_group;
    const bool cd = above >= topk_group;
    const uint32_t ck_bal = __ballot_sync(0xffffffffu, ck);
    const uint32_t amb_bal = __ballot_sync(0xffffffffu, !ck && !cd);
    for (int g = 0; g < G; ++g) {
      if ((ck_bal >> (g * lpg)) & 1u) kept_mask |= 1u << g;
      if ((amb_bal >> (g * lpg)) & 1u) amb_mask |= 1u << g;
    }
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      if (e0 + m >= E) continue;
      if (!cd) possible |= 1u << m;
      if (ck) certain |= 1u << m;
      // ambiguous group: every expert that can be one of its two best
      if (!ck && !cd && hi[m] >= ((gs >= 2) ? l2 : l1)) need |= 1u << m;
    }
  } else {
#pragma unroll
    for (int m = 0; m < PER; ++m)
      if (e0 + m < E) {
        possible |= 1u << m;
        certain |= 1u << m;
      }
    kept_mask = 1u;
  }

  // theta: the k-th largest lower end among experts of certainly kept groups
  float theta = -kInf;
  {
    uint32_t left = certain;
    for (int j = 0; j < k; ++j) {
      float bv = -kInf;
      int bi = 0x7fffffff;
#pragma unroll
      for (int m = 0; m < PER; ++m)
        if ((left >> m) & 1u) {
          if (lo[m] > bv || bi == 0x7fffffff) {
            bv = lo[m];
            bi = e0 + m;
          }
        }
      warp_argmax(bv, bi);
      if (bi == 0x7fffffff) {  // fewer than k certainly eligible experts
        theta = -kInf;
        break;
      }
      if (bi / PER == lane) left &= ~(1u << (bi - e0));
      theta = bv;
    }
  }
#pragma unroll
  for (int m = 0; m < PER; ++m)
    if (((possible >> m) & 1u) && hi[m] >= theta) need |= 1u << m;

  // the list: ids in increasing order (lane order is expert order)
  const int mine = __popc(need);
  int before = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, before, off);
    if (lane >= off) before += o;
  }
  const int total = __shfl_sync(0xffffffffu, before, 31);
  before -= mine;
  int w = before;
#pragma unroll
  for (int m = 0; m < PER; ++m)
    if ((need >> m) & 1u) need_out[w++] = static_cast<int16_t>(e0 + m);
  *kept_out = kept_mask;
  *amb_out = amb_mask;
  return total;
}

// need: one warp per token: the token's norm (its K-group slices of the
// squared norm added in order), rs_decide, and the record [n, certainly kept
// group mask, ambiguous group mask, 0, the n expert ids in increasing order].
constexpr int kNeedWarps = 8;

template <int PER>
__global__ void __launch_bounds__(kNeedWarps * 32)
    rs_need_kernel(const float *__restrict__ part, const float *__restrict__ xn2, int ksplit,
                   const float *__restrict__ wn, const float *__restrict__ bias, int T, int E,
                   int G, int topk_group, int k, int score, float bias_scale, float alpha,
                   int32_t *__restrict__ rec, int32_t *__restrict__ cnt) {
  pdl_begin();
  __shared__ int sh_total;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) sh_total = 0;
  __syncthreads();
  const int t = blockIdx.x * kNeedWarps + (threadIdx.x >> 5);
  if (t < T) {
    // the K-group slices of the squared norm: one load per lane, added in
    // slice order
    float xsq = 0.0f;
    for (int g0 = 0; g0 < ksplit; g0 += 32) {
      const float v = (g0 + lane < ksplit) ? xn2[(size_t)(g0 + lane) * T + t] : 0.0f;
      const int m = min(32, ksplit - g0);
      for (int g = 0; g < m; ++g) xsq = __fadd_rn(xsq, __shfl_sync(0xffffffffu, v, g));
    }
    int32_t *r = rec + (size_t)t * (E + kRsRecHead);
    uint32_t kept = 0, amb = 0;
    const int n = rs_decide<PER>(part, __fsqrt_rn(xsq), wn, bias, t, T, E, G, topk_group, k,
                                 score, bias_scale, ksplit, alpha, lane,
                                 reinterpret_cast<int16_t *>(r + kRsRecHead), &kept, &amb);
    if (lane == 0) {
      r[0] = n;
      r[1] = static_cast<int32_t>(kept);
      r[2] = static_cast<int32_t>(amb);
      r[3] = 0;
      atomicAdd(&sh_total, n);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh_total > 0) atomicAdd(cnt, sh_total);  // refined pairs of the call
}

// Fixed-order logits of B experts of one token at once: lane l sums its
// chunks l, l+32, ... in order for each expert; the x chunk (shared memory)
// is unpacked once for all B, and pairs of experts share one packed
// fma.rn.f32x2 (two IEEE fp32 fused multiply-adds, each rounded as a scalar
// fma.rn).
template <int B>
__device__ __forceinline__ void canon_dot_batch(const uint4 *xs, const uint16_t *__restrict__ wt,
                                                const int *es, int d, int lane, float (&out)[4]) {
  const int nch = d / 8;
  const uint4 *wr[B];
#pragma unroll
  for (int b = 0; b < B; ++b) wr[b] = reinterpret_cast<const uint4 *>(wt + (size_t)es[b] * d);
  uint64_t acc2[B / 2 + 1];  // (one spare: B / 2 may be 0)
  float acc1 = 0.0f;
#pragma unroll
  for (int b = 0; b < B / 2 + 1; ++b) acc2[b] = 0;
  int c = lane;
  uint4 wv[2][B];
  if (c < nch) {  // rows of fewer than 32 chunks (d < 256) leave lanes idle
#pragma unroll
    for (int b = 0; b < B; ++b) wv[0][b] = __ldg(wr[b] + c);
  }
  for (int it = 0; c < nch; ++it, c += 32) {
    const int cur = it & 1;
    if (c + 32 < nch) {
#pragma unroll
      for (int b = 0; b < B; ++b) wv[cur ^ 1][b] = __ldg(wr[b] + c + 32);
    }
    const uint4 xv = xs[c];
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float x0 = bf16lo(xw[h]), x1 = bf16hi(xw[h]);
      uint64_t xd0, xd1;
      asm("mov.b64 %0, {%1, %1};" : "=l"(xd0) : "f"(x0));
      asm("mov.b64 %0, {%1, %1};" : "=l"(xd1) : "f"(x1));
#pragma unroll
      for (int b = 0; b + 1 < B; b += 2) {
        const uint32_t wa = (&wv[cur][b].x)[h], wb = (&wv[cur][b + 1].x)[h];
        uint64_t w0, w1;
        asm("{\n\t.reg .b32 a, b;\n\tshl.b32 a, %1, 16;\n\tshl.b32 b, %2, 16;\n\t"
            "mov.b64 %0, {a, b};\n\t}"
            : "=l"(w0)
            : "r"(wa), "r"(wb));
        asm("{\n\t.reg .b32 a, b;\n\tand.b32 a, %1, 0xFFFF0000;\n\tand.b32 b, %2, 0xFFFF0000;\n\t"
            "mov.b64 %0, {a, b};\n\t}"
            : "=l"(w1)
            : "r"(wa), "r"(wb));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[b / 2]) : "l"(xd0), "l"(w0));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[b / 2]) : "l"(xd1), "l"(w1));
      }
      if (B & 1) {
        const uint32_t wa = (&wv[cur][B - 1].x)[h];
        acc1 = __fmaf_rn(x0, bf16lo(wa), acc1);
        acc1 = __fmaf_rn(x1, bf16hi(wa), acc1);
      }
    }
  }
#pragma unroll
  for (int b = 0; b + 1 < B; b += 2) {
    float a0, a1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc2[b / 2]));
    out[b] = butterfly_sum(a0);
    out[b + 1] = butterfly_sum(a1);
  }
  if (B & 1) out[B - 1] = butterfly_sum(acc1);
}

// refine: one CTA per token.  The token's row is staged in shared memory;
// then either (BATCH, small T: fewer passes matter most) 4 warps, warp w
// taking record entries 4 w .. 4 w + 3, 4 w + 16 .., four experts at a time,
// or (large T: the many weight rows in flight matter most) 8 warps, warp w
// taking entries w, w + 8, ... one at a time; then warp 0 takes the kept
// groups (certain ones plus the best ambiguous ones by exact group score)
// and the top-k refined experts in them, their output order (score desc,
// index asc) and weights.
template <bool BATCH>
struct RefCfg {
  static constexpr int WARPS = BATCH ? 4 : 8;
};
constexpr int kRefBatchMaxT = 4096;

template <int PER, bool BATCH>
__global__ void __launch_bounds__(RefCfg<BATCH>::WARPS * 32)
    rs_refine_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ wt,
                     const float *__restrict__ bias, const int32_t *__restrict__ rec, int T,
                     int d, int E, int G, int topk_group, int k, int score, float bias_scale,
                     int32_t *__restrict__ ids, float *__restrict__ weights) {
  pdl_begin();
  extern __shared__ uint4 sh_x[];  // d / 8 chunks, then E floats (exact logits by expert)
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nch = d / 8;
  float *sh_l = reinterpret_cast<float *>(sh_x + nch);
  const int32_t *r = rec + (size_t)t * (E + kRsRecHead);
  const int16_t *need = reinterpret_cast<const int16_t *>(r + kRsRecHead);
  const int n = r[0];
  const uint32_t kept_mask = static_cast<uint32_t>(r[1]);
  const uint32_t amb_mask = static_cast<uint32_t>(r[2]);
  constexpr int kWarps = RefCfg<BATCH>::WARPS;
  const uint4 *xg = reinterpret_cast<const uint4 *>(x + (size_t)t * d);
  for (int c = threadIdx.x; c < nch; c += kWarps * 32) sh_x[c] = __ldg(xg + c);
  for (int e = threadIdx.x; e < E; e += kWarps * 32) sh_l[e] = __int_as_float(0x7fc00000);
  __syncthreads();
  if (!BATCH) {
    for (int j = warp; j < n; j += kWarps) {
      const int e = min(max(static_cast<int>(need[j]), 0), E - 1);  // guards the load
      const float v = canon_dot(sh_x, reinterpret_cast<const uint4 *>(wt + (size_t)e * d), nch,
                                lane);
      if (lane == 0) sh_l[e] = v;
    }
  }
  for (int first = 4 * warp; BATCH && first < n; first += 4 * kWarps) {
    const int B = min(4, n - first);
    int es[4];
#pragma unroll
    for (int b = 0; b < 4; ++b)  // always in range; guards the loads
      es[b] = min(max(static_cast<int>(need[first + (b < B ? b : 0)]), 0), E - 1);
    float v[4];
    switch (B) {
      case 4: canon_dot_batch<4>(sh_x, wt, es, d, lane, v); break;
      case 3: canon_dot_batch<3>(sh_x, wt, es, d, lane, v); break;
      case 2: canon_dot_batch<2>(sh_x, wt, es, d, lane, v); break;
      default: canon_dot_batch<1>(sh_x, wt, es, d, lane, v); break;
    }
    if (lane == 0)
      for (int b = 0; b < B; ++b) sh_l[es[b]] = v[b];
  }
  __syncthreads();
  if (warp != 0) return;

  const float *lt = sh_l;
  const float kInf = __int_as_float(0x7f800000);
  const bool sig = score == MOE_SCORE_SIGMOID_BIAS;
  const int e0 = lane * PER;
  // exact scores of the refined experts (NaN marks "not refined")
  float sc[PER];
  uint32_t refined = 0;
#pragma unroll
  for (int m = 0; m < PER; ++m) {
    const int e = e0 + m;
    sc[m] = -kInf;
    if (e < E) {
      const float l = lt[e];
      if (!isnan(l)) {
        refined |= 1u << m;
        sc[m] = sig ? __fadd_rn(canon_sigmoid(l), __fmul_rn(bias_scale, bias[e])) : l;
      }
    }
  }
  uint32_t kept = kept_mask;
  if (G > 1 && amb_mask != 0) {
    // exact group scores of the ambiguous groups (their two best are refined)
    const int gs = E / G;
    const int lpg = gs / PER;
    float m1 = -kInf, m2 = -kInf;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const float v = ((refined >> m) & 1u) ? sc[m] : -kInf;
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
    const float gsc = (gs >= 2) ? __fadd_rn(m1, m2) : m1;
    const int free_slots = topk_group - __popc(kept_mask);
    uint32_t left = amb_mask;
    for (int j = 0; j < free_slots; ++j) {
      // lane g bids group g's score (computed at lane g * lpg)
      const float gv = __shfl_sync(0xffffffffu, gsc, (lane < G ? lane : 0) * lpg);
      const bool bid = lane < G && ((left >> lane) & 1u);
      float bv = bid ? gv : -kInf;
      int bi = bid ? lane : 0x7fffffff;
      warp_argmax(bv, bi);
      if (bi == 0x7fffffff) break;
      kept |= 1u << bi;
      left &= ~(1u << bi);
    }
  }
  uint32_t eligible = 0;
  {
    const int gs = (G > 1) ? E / G : E;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = e0 + m;
      if (e < E && ((refined >> m) & 1u) && ((G <= 1) || ((kept >> (e / gs)) & 1u)))
        eligible |= 1u << m;
    }
  }
  // top-k refined experts of the kept groups; output order is the pick order
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -kInf;
    int bi = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < PER; ++m)
      if ((eligible >> m) & 1u) {
        if (sc[m] > bv || bi == 0x7fffffff) {
          bv = sc[m];
          bi = e0 + m;
        }
      }
    warp_argmax(bv, bi);
    if (bi != 0x7fffffff && bi / PER == lane) eligible &= ~(1u << (bi - e0));
    if (lane == j) my_id = bi;
  }
  const bool act = lane < k;
  const int id = act ? min(max(my_id, 0), E - 1) : 0;
  const float my_l = act ? lt[id] : 0.0f;
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float v = act ? (sig ? canon_sigmoid(my_l) : canon_exp(__fsub_rn(my_l, l0))) : 0.0f;
  float sum = __shfl_sync(0xffffffffu, v, 0);
  for (int j = 1; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, v, j));
  if (act) {
    ids[(size_t)t * k + lane] = my_id;
    weights[(size_t)t * k + lane] = __fdiv_rn(v, sum);
  }
}

// host: router weights with a caller-owned prepared copy (transposed
// weight + column norms), registered by moe_router_prepare
struct Prepared {
  const void *w_r;
  int d, E;
  void *prep;
};
std::mutex g_prep_mu;
Prepared g_prep[64];
int g_prep_n = 0;

void *find_prepared(const void *w_r, int d, int E) {
  std::lock_guard<std::mutex> lock(g_prep_mu);
  for (int i = 0; i < g_prep_n; ++i)
    if (g_prep[i].w_r == w_r && g_prep[i].d == d && g_prep[i].E == E) return g_prep[i].prep;
  return nullptr;
}

}  // namespace

size_t router_prep_bytes(int d, int E) {
  return al256(static_cast<size_t>(E) * d * 2) + al256(static_cast<size_t>(E) * 4);
}

bool router_register_prepared(const void *w_r, int d, int E, void *prep) {
  std::lock_guard<std::mutex> lock(g_prep_mu);
  for (int i = 0; i < g_prep_n; ++i)
    if (g_prep[i].w_r == w_r) {
      g_prep[i] = {w_r, d, E, prep};
      return true;
    }
  if (g_prep_n == 64) return false;
  g_prep[g_prep_n++] = {w_r, d, E, prep};
  return true;
}

bool router_release_prepared(const void *w_r) {
  std::lock_guard<std::mutex> lock(g_prep_mu);
  for (int i = 0; i < g_prep_n; ++i)
    if (g_prep[i].w_r == w_r) {
      g_prep[i] = g_prep[--g_prep_n];
      return true;
    }
  return false;
}

size_t screened_scratch_bytes(int T, int d, int E) {
  if (d % 64 != 0 || E % 64 != 0) return 0;
  return rs_layout(T, d, E).end;
}

bool router_screened(int T, int d, int E, int G, int k) {
  // the refine kernel keeps the token row and E logits in shared memory
  return T > 0 && d % 64 == 0 && d <= 16384 && E % 64 == 0 && E <= 1024 && k <= 32 &&
         router_select_per(E, G) != 0;
}

int router_launches(int T, int d, int E, int G, int k) {
  // screened: transposed copy and norms (not launched for a prepared
  // weight), GEMM, need, refine
  if (router_screened(T, d, E, G, k)) return 5;
  return router_logits_launches(d, E) + 1;
}

const int32_t *router_refined_count(const void *w_scratch, int T, int d, int E, int G, int k) {
  if (!router_screened(T, d, E, G, k)) return nullptr;
  return reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(w_scratch) +
                                           rs_layout(T, d, E).cnt);
}

cudaError_t launch_router_prepare(const void *w_r, int d, int E, void *prep, cudaStream_t s) {
  uint8_t *base = static_cast<uint8_t *>(prep);
  uint16_t *wt = reinterpret_cast<uint16_t *>(base);
  MOE_LAUNCH_PDL(rs_transpose_kernel, dim3(E / 64, d / 64), 256, 0, s,
                 static_cast<const uint16_t *>(w_r), d, E, wt);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  MOE_LAUNCH_PDL(rs_wnorm_kernel, (E + 7) / 8, 256, 0, s, static_cast<const uint16_t *>(wt), d,
                 E, reinterpret_cast<float *>(base + al256(static_cast<size_t>(E) * d * 2)));
  return cudaGetLastError();
}

cudaError_t launch_router(const void *x, const void *w_r, const float *bias, int T, int d, int E,
                          int G, int topk_group, int k, int score, float bias_scale,
                          float *logits, int32_t *ids, float *weights, void *w_scratch,
                          uint32_t *status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (!router_screened(T, d, E, G, k)) {
    cudaError_t err = launch_router_logits(x, w_r, T, d, E, logits, w_scratch, s);
    if (err != cudaSuccess) return err;
    return launch_router_select(logits, bias, T, E, G, topk_group, k, score, bias_scale, 0, ids,
                                weights, s);
  }
  const RsLayout L = rs_layout(T, d, E);
  uint8_t *base = static_cast<uint8_t *>(w_scratch);
  int32_t *cnt = reinterpret_cast<int32_t *>(base + L.cnt);
  float *part = reinterpret_cast<float *>(base + L.part);
  float *xn2 = reinterpret_cast<float *>(base + L.xn2);
  int32_t *rec = reinterpret_cast<int32_t *>(base + L.rec);
  cudaError_t err;
  // the prepared copy of this weight, or one made now in the scratch
  uint8_t *prep = static_cast<uint8_t *>(find_prepared(w_r, d, E));
  if (!prep) {
    prep = base + L.wt;
    err = launch_router_prepare(w_r, d, E, prep, s);
    if (err != cudaSuccess) return err;
  }
  const uint16_t *wt = reinterpret_cast<const uint16_t *>(prep);
  const float *wn = reinterpret_cast<const float *>(prep + al256(static_cast<size_t>(E) * d * 2));

  // tensor-core logits and the token norms
  const int bn = rs_bn(E);
  const int ks = rs_ksplit(T, d, E);
  CUtensorMap tmA, tmB;
  if (!rs_make_tmap(&tmA, x, d, T, kRsBM) || !rs_make_tmap(&tmB, wt, d, E, bn))
    return cudaErrorInvalidValue;
  RsArgs a;
  a.T = T;
  a.d = d;
  a.E = E;
  a.n_tiles = E / bn;
  a.ksplit = ks;
  a.items = ((T + kRsBM - 1) / kRsBM) * a.n_tiles * ks;
  a.part = part;
  a.xn2 = xn2;
  a.cnt = cnt;
  a.status = status;
  a.wait_limit_ns = kDefaultWaitLimitNs;
  int nsm = 0, dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  const int grid = a.items < nsm ? a.items : nsm;
#define MOE_RS_GEMM(BN_)                                                                     \
  case BN_: {                                                                                \
    using C = RsCfg<BN_>;                                                                    \
    err = cudaFuncSetAttribute(rs_gemm_kernel<BN_>,                                          \
                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);  \
    if (err != cudaSuccess) return err;                                                      \
    MOE_LAUNCH_PDL(rs_gemm_kernel<BN_>, grid, kRsThreads, C::SMEM_BYTES, s, tmA, tmB, a);    \
    break;                                                                                   \
  }
  switch (bn) {
    MOE_RS_GEMM(256)
    MOE_RS_GEMM(128)
    MOE_RS_GEMM(64)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_RS_GEMM
  if ((err = cudaGetLastError()) != cudaSuccess) return err;

  const float alpha = static_cast<float>(rs_alpha(T, d, E));
  const int per = router_select_per(E, G);
  const unsigned ngrid = static_cast<unsigned>((T + kNeedWarps - 1) / kNeedWarps);
  const size_t rsmem = static_cast<size_t>(d) * 2 + static_cast<size_t>(E) * 4;
#define MOE_RS_REFINE(P, BATCH)                                                                \
  do {                                                                                         \
    if (rsmem > 48 * 1024) {                                                                   \
      err = cudaFuncSetAttribute(rs_refine_kernel<P, BATCH>,                                   \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,                  \
                                 static_cast<int>(rsmem));                                     \
      if (err != cudaSuccess) return err;                                                      \
    }                                                                                          \
    MOE_LAUNCH_PDL(rs_refine_kernel<P, BATCH>, T, RefCfg<BATCH>::WARPS * 32, rsmem, s,         \
                   static_cast<const uint16_t *>(x), wt, bias,                                 \
                   static_cast<const int32_t *>(rec), T, d, E, G, topk_group, k, score,        \
                   bias_scale, ids, weights);                                                  \
  } while (0)
  switch (per) {
#define MOE_RS_SEL(P)                                                                          \
  case P:                                                                                      \
    MOE_LAUNCH_PDL(rs_need_kernel<P>, ngrid, kNeedWarps * 32, 0, s,                            \
                   static_cast<const float *>(part), static_cast<const float *>(xn2), ks, wn,  \
                   bias, T, E, G, topk_group, k, score, bias_scale, alpha, rec, cnt);          \
    if ((err = cudaGetLastError()) != cudaSuccess) return err;                                 \
    if (T <= kRefBatchMaxT) {                                                                  \
      MOE_RS_REFINE(P, true);                                                                  \
    } else {                                                                                   \
      MOE_RS_REFINE(P, false);                                                                 \
    }                                                                                          \
    break;
    MOE_RS_SEL(2)
    MOE_RS_SEL(4)
    MOE_RS_SEL(8)
    MOE_RS_SEL(16)
    MOE_RS_SEL(32)
#undef MOE_RS_SEL
#undef MOE_RS_REFINE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace moe

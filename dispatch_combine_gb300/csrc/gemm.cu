// gemm.cu -- grouped expert GEMMs on the 5th-generation tensor cores.
//
// The expert FFN of the MoE-TP/EP comparison on "推理INFRA方法论-02-parallelism"
// is a grouped GEMM over experts with gate and up fused into one weight
// ("DeepGEMM masked, gate_up fused"); experts that received no token are
// skipped ("fused_moe" skips unhit experts), and the masked variant gives each
// expert a padded slab with a valid-row count.  This file rebuilds that for
// sm_103a:
//
//   * persistent kernel, one CTA per SM, static round-robin over tiles
//     (expert, n-tile, m-tile) with m fastest, so the CTAs working at the same
//     time share the expert's weight tile through L2;
//   * warp 0 (one lane): TMA producer, 128x64 A tile + two 64-column halves of
//     the B tile per stage, 128-byte swizzle, multi-stage mbarrier ring;
//   * warp 1 (one lane): issues tcgen05.mma (M=128, N=BN, K=16, bf16 in, fp32
//     accumulator in TMEM), two TMEM accumulators so the epilogue of one tile
//     overlaps the main loop of the next;
//   * warps 2-5: epilogue, tcgen05.ld of their 32-lane quadrant; gate_up
//     tiles hold gate columns [0,BN/2) and the matching up columns
//     [BN/2,BN) of the same intermediate indices, so SwiGLU
//     h = silu(g) * u is applied in registers and only h (bf16) is written;
//     down tiles are written as fp32.
//
// Every wait is bounded (MOE_ERR_TIMEOUT in the status word, then the CTA
// drains its in-flight copies and MMAs, frees TMEM and returns).
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // 64 bf16 = one 128-byte swizzle row
constexpr int kGemmThreads = 192;
constexpr int kStageBudget = 196608;
constexpr int kMaxE = 1024;

template <int BN, bool SWIGLU>
struct Cfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = kStageBudget / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BN_OUT = SWIGLU ? BN / 2 : BN;
  static constexpr int HALF = BN / 2;  // rows of B per TMA load
  // [A stages][B stages][barriers: full, empty, tmem_full x2, tmem_empty x2,
  // drain][tmem slot][abort][mtile_base copy]
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int MT_OFF = MISC_OFF + 16;
  static constexpr int SMEM_BYTES = MT_OFF + (kMaxE + 1) * 4 + 1024;  // + alignment slack
  static_assert(STAGES >= 2, "need at least two stages");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "bad BN");
  static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
};

struct Tile {
  int e, m, n;
  int row0;        // first row of the tile in A / out
  int rows_valid;  // valid rows in the tile (<= 128)
};

struct KArgs {
  int E, K, n_tiles, layout, M_max, b_rows, up_off;
  int ksplit;   // 1-CTA down form: K pieces per tile, summed into a zeroed out (1: none)
  int m_block;  // m-tiles per rasterization block (A rows of a block stay in L2)
  int out_v8;   // output base 32-byte aligned: 32-byte stores
  int out_tma;  // pair down form: fp32 output through the tmY tensor map (TMA stores)
  uint32_t *split_flags;  // pair down form: flags of the split last wave (nullptr: no split)
  uint32_t split_epoch;   // nonzero value this launch raises the flags to
  // pair down form, compact output (y16): out holds the fp16 values
  // [rows, ldo] and out_codes the code bytes [rows, ldo / 32]; a split tile's
  // first K half leaves its fp32 sums in split_part (256 x 256 floats per
  // split slot, split_part_slots slots).  nullptr: fp32 output.
  uint8_t *out_codes;
  float *split_part;
  int split_part_slots;
  float *out_h_scales;  // FP8 gate_up: h quantized in the epilogue (nullptr: bf16 h)
  int64_t rows_total;
  const int32_t *seg;
  const int32_t *seg2;  // kLayoutTwoSeg: overflow offsets [E+1]
  const int32_t *mtile_base;
  void *out;
  int64_t ldo;
  uint32_t *status;
  uint64_t wait_limit_ns;
};

template <int TILE_M = kBM>
__device__ __forceinline__ Tile decode_tile(const KArgs &a, const int32_t *mt, int u,
                                            const int32_t *sg = nullptr) {
  // sg: a shared-memory copy of a.seg (the row offsets / counts), or nullptr
  const int32_t *seg = sg ? sg : a.seg;
  Tile t;
  const int q = u / a.n_tiles;
  int lo = 0, hi = a.E - 1;  // largest e with mt[e] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mt[mid] <= q)
      lo = mid;
    else
      hi = mid - 1;
  }
  t.e = lo;
  // Inside an expert, tiles go in blocks of m_block m-tiles; inside a block
  // the m-tile index runs fastest, then n.  CTAs working at the same time
  // then share the block's A rows and each B tile through L2, and A is read
  // from HBM once however many n-tiles there are.
  const int mt_e = mt[lo + 1] - mt[lo];
  const int local = u - mt[lo] * a.n_tiles;
  const int full = mt_e / a.m_block;
  const int blk = local / (a.m_block * a.n_tiles);
  const int mb = (blk < full) ? a.m_block : mt_e - full * a.m_block;
  const int within = local - blk * a.m_block * a.n_tiles;
  t.n = within / mb;
  t.m = blk * a.m_block + (within - t.n * mb);
  int rows, start, m = t.m;
  if (a.layout == MOE_LAYOUT_CONTIGUOUS) {
    start = seg[t.e];
    rows = seg[t.e + 1] - start;
  } else {
    start = t.e * a.M_max;
    rows = min(max(seg[t.e], 0), a.M_max);
    if (a.layout == kLayoutTwoSeg) {
      // the slab's tiles, then the overflow rows' tiles
      const int tiles1 = (rows + TILE_M - 1) / TILE_M;
      if (m >= tiles1) {
        m -= tiles1;
        start = a.E * a.M_max + a.seg2[t.e];
        rows = a.seg2[t.e + 1] - a.seg2[t.e];
      }
    }
  }
  t.row0 = start + m * TILE_M;
  t.rows_valid = min(TILE_M, rows - m * TILE_M);
  return t;
}

// Wait bounded by time only (used to drain after an abort).
__device__ __forceinline__ bool wait_drain(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

template <int BN, bool SWIGLU>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const KArgs args) {
  pdl_begin();
  using C = Cfg<BN, SWIGLU>;
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
  int32_t *mt = reinterpret_cast<int32_t *>(smem + C::MT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) mt[i] = args.mtile_base[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int ksplit = SWIGLU ? 1 : args.ksplit;
  const int total = mt[args.E] * args.n_tiles * ksplit;
  if (static_cast<int>(blockIdx.x) >= total) return;  // uniform across the CTA

  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int kblocks = args.K / kBK;
  // k-blocks [kb_lo, kb_hi) of piece u % ksplit
  auto kb_lo = [&](int u) { return (u % ksplit) * kblocks / ksplit; };
  auto kb_hi = [&](int u) { return (u % ksplit + 1) * kblocks / ksplit; };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[C::STAGES];
      bool issued[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) issued[s] = false;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        const Tile t = decode_tile(args, mt, u / ksplit);
        int b0, b1;
        if (SWIGLU) {
          b0 = t.e * args.b_rows + t.n * C::HALF;
          b1 = t.e * args.b_rows + args.up_off + t.n * C::HALF;
        } else {
          b0 = t.e * args.b_rows + t.n * BN;
          b1 = b0 + C::HALF;
        }
        for (int kb = kb_lo(u); kb < kb_hi(u); ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status,
                                 args.wait_limit_ns))
            break;
          uint8_t *a_dst = smA + stage * C::A_BYTES;
          uint8_t *b_dst = smB + stage * C::B_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(a_dst, &tmA, &full[stage], kb * kBK, t.row0);
          tma_load_2d(b_dst, &tmB, &full[stage], kb * kBK, b0);
          tma_load_2d(b_dst + C::HALF * 128, &tmB, &full[stage], kb * kBK, b1);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every issued copy must have landed before the CTA exits
      for (int s = 0; s < C::STAGES; ++s)
        if (issued[s]) wait_drain(&full[s], issued_phase[s], args.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t kIdesc = mma_idesc_bf16_f32(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool any_mma = false;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        if (!mbar_wait_bounded(&tmem_empty[acc], acc_phase ^ 1u, abort_flag, args.status,
                               args.wait_limit_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        const int kb0 = kb_lo(u);
        for (int kb = kb0; kb < kb_hi(u); ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.status,
                                 args.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(smA + stage * C::A_BYTES));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(smB + stage * C::B_BYTES));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // +32 bytes along K inside the 128-byte swizzle row
            mma_bf16_ss(d_tmem, ad + 2u * kk, bd + 2u * kk, kIdesc,
                        (kb != kb0 || kk != 0) ? 1u : 0u);
          }
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
      if (any_mma) {
        mma_commit(drain);
        wait_drain(drain, 0, args.wait_limit_ns);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quad = warp & 3;  // TMEM lanes quad*32 .. +31
    const int row = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Tile t = decode_tile(args, mt, u / ksplit);
      const bool waited = mbar_wait_bounded(&tmem_full[acc], acc_phase, abort_flag,
                                            args.status, args.wait_limit_ns);
      // the tcgen05.ld below is warp-collective: leave together if any lane gave up
      if (!__all_sync(0xffffffffu, waited)) break;
      tc_fence_after();
      const uint32_t tb =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      const int64_t grow = static_cast<int64_t>(t.row0) + row;
      // rows_total guards against caller offsets that overrun the buffers
      const bool ok = row < t.rows_valid && grow >= 0 && grow < args.rows_total;
      if (SWIGLU) {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(args.out) + grow * args.ldo +
                             static_cast<int64_t>(t.n) * C::BN_OUT;
#pragma unroll 1
        for (int c = 0; c < C::BN_OUT / 32; ++c) {
          uint32_t g[32], v[32];
          tmem_ld_32x32b_x32(tb + c * 32, g);
          tmem_ld_32x32b_x32(tb + C::HALF + c * 32, v);
          tmem_ld_wait();
          tmem_regs_fence(g);
          tmem_regs_fence(v);
          if (ok) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float u0 = __uint_as_float(v[2 * i]), u1 = __uint_as_float(v[2 * i + 1]);
              const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
              const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
              packed[i] = pack_bf16x2(h0, h1);
            }
            if (args.out_v8) {
              // each lane writes whole 32-byte sectors of its row
              uint32_t w8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w8[i] = packed[i];
              st_global_v8(dst + c * 32, w8);
#pragma unroll
              for (int i = 0; i < 8; ++i) w8[i] = packed[8 + i];
              st_global_v8(dst + c * 32 + 16, w8);
            } else {
              uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                   packed[4 * i + 3]);
            }
          }
        }
      } else if (args.out_codes != nullptr) {
        // compact output (BN = 256, no K pieces): 32 fp16 values and one code
        // per 32-column chunk, the row's 8 codes of the tile in one store
        __half *dst = static_cast<__half *>(args.out) + grow * args.ldo +
                      static_cast<int64_t>(t.n) * BN;
        uint64_t codes = 0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c * 32, v);
          tmem_ld_wait();
          tmem_regs_fence(v);
          if (ok) {
            uint32_t hw[16];
            const uint32_t cc = y16_encode32(v, hw);
            uint32_t w8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) w8[q] = hw[q];
            st_global_v8(dst + c * 32, w8);
#pragma unroll
            for (int q = 0; q < 8; ++q) w8[q] = hw[8 + q];
            st_global_v8(dst + c * 32 + 16, w8);
            codes |= static_cast<uint64_t>(cc) << (8 * c);
          }
        }
        if (ok)
          *reinterpret_cast<uint64_t *>(args.out_codes + grow * (args.ldo / 32) +
                                        static_cast<int64_t>(t.n) * (BN / 32)) = codes;
      } else {
        float *dst = static_cast<float *>(args.out) + grow * args.ldo +
                     static_cast<int64_t>(t.n) * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c * 32, v);
          tmem_ld_wait();
          tmem_regs_fence(v);
          if (ok && ksplit > 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              red_add_v4(dst + c * 32 + 4 * i, __uint_as_float(v[4 * i]),
                         __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                         __uint_as_float(v[4 * i + 3]));
          } else if (ok) {
            if (args.out_v8) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t w8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) w8[j] = v[8 * i + j];
                st_global_v8(dst + c * 32 + 8 * i, w8);
              }
            } else {
              float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Pair variant (cta_group::2): a cluster of two CTAs on two SMs computes a
// 256-row tile.  Each CTA loads its own 128 rows of A and half (BN/2 rows) of
// the B tile; the even CTA issues the pair MMAs (M=256, N=BN), which read A
// and B from both CTAs' shared memory and leave rows 0-127 of the
// accumulator in its TMEM and rows 128-255 in the peer's.  Per SM this halves
// the B bytes per FLOP and, with 32 KB stages, gives a 6-stage ring.  The
// down form stores its fp32 output with TMA: an epilogue warp whose 32 rows
// are all valid stages each 32-column chunk in the two 16-column halves of a
// swizzled shared-memory box and issues one tensor store per half, so the
// output leaves as whole 64-byte row pieces instead of per-row sector writes
// (other warps store directly).
//   full[s]       in the even CTA, completed by both CTAs' TMA bytes;
//   empty[s]      in both CTAs, the pair MMA commit arrives on both;
//   tmem_full[b]  in both CTAs, the pair MMA commit arrives on both;
//   tmem_empty[b] in the even CTA, all 8 epilogue warps of the pair arrive.
// ---------------------------------------------------------------------------
// k-blocks per ring stage of the pair kernel (one barrier round trip each)
constexpr int kPairKPS = 2;

template <int BN, bool SWIGLU>
struct Cfg2 {
  static constexpr int A_BYTES = 128 * kBK * 2;        // one k-block of this CTA's A
  static constexpr int B_BYTES = (BN / 2) * kBK * 2;   // one k-block of its B half
  static constexpr int KPS = kPairKPS;
  static constexpr int A_STAGE = KPS * A_BYTES;
  static constexpr int B_STAGE = KPS * B_BYTES;
  static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
  static constexpr int STAGES = kStageBudget / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BN_OUT = SWIGLU ? BN / 2 : BN;
  static constexpr int HALF = BN / 2;
  // down: one 32-row x 32-column fp32 staging box per epilogue warp for the
  // TMA stores of the output (128-byte swizzle, 1024-byte aligned)
  static constexpr int OUT_OFF = STAGES * STAGE_BYTES;
  static constexpr int OUT_BOX_BYTES = 32 * 32 * 4;
  static constexpr int OUT_BYTES = SWIGLU ? 0 : 4 * OUT_BOX_BYTES;
  static constexpr int BAR_OFF = OUT_OFF + OUT_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int MT_OFF = MISC_OFF + 16;
  // a copy of the row offsets / counts, so tile decoding reads no global memory
  static constexpr int SEG_OFF = MT_OFF + (kMaxE + 1) * 4;
  static constexpr int SMEM_BYTES = SEG_OFF + (kMaxE + 1) * 4 + 1024;
  static_assert(BN == 256 || BN == 128, "pair tile width");
  static_assert(STAGES * KPS >= 4, "pipeline depth");
  static_assert(OUT_OFF % 1024 == 0, "swizzled staging alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// An expert's last 256-row tile that holds at most 128 rows runs swapped
// (BN = 256 only): the 256 weight rows of the n-tile are the pair MMA's M
// side (128 per CTA, in the A slots), the tile's token rows are its N side
// (N = rows rounded up to 16, N/2 rows per CTA from a 64-row box, in the B
// slots).  The tile then costs the weight bytes plus its own rows instead
// of a full 256-row tile.  For gate_up each CTA's 128 M rows are 4 groups of
// [16 gate rows, the 16 matching up rows] (a 4-D tensor map), so a warp's
// 32 TMEM lanes hold both factors of 16 intermediate columns.
constexpr int kSwapBoxRows = 64;
__device__ __forceinline__ int pair_swap_n(const Tile &t) {
  return (t.rows_valid <= 2 * kSwapBoxRows) ? ((t.rows_valid + 15) & ~15) : 0;
}
// A swapped tail is paced by its loads, so each CTA loads only the token
// rows it needs: boxes of 8, 16, 32 or 64 rows (the smallest >= N / 2).
struct SwapXMaps {
  CUtensorMap m[4];  // box rows 8, 16, 32, 64
};
__device__ __forceinline__ int swap_box_index(int sn) {
  const int half = sn >> 1;
  return half <= 8 ? 0 : half <= 16 ? 1 : half <= 32 ? 2 : 3;
}

// One work item of a CTA pair: a whole tile, or (split last wave of the down
// form) one K half of a tile.  Items n_full + j, j < 2 * rem, are a half of
// tile n_full + j % rem; pair c takes items c, c + ncl, ..., so the two
// halves of a tile normally run at the same time on pairs j % rem and
// j % rem + rem.  Which half stores and which adds is decided at run time
// (the first to reach its epilogue stores), so neither depends on the other
// pair being scheduled.
struct PairWork {
  int u;         // tile index
  int kb0, kb1;  // k-blocks [kb0, kb1)
  int piece;     // -1 whole tile, 0 first K half, 1 second K half
  int slot;      // split tile j % rem (16 flag words each)
};
__device__ __forceinline__ PairWork pair_work(int w, int n_full, int rem, int kblocks) {
  PairWork pw;
  if (w < n_full) {
    pw.u = w;
    pw.kb0 = 0;
    pw.kb1 = kblocks;
    pw.piece = -1;
    pw.slot = 0;
  } else {
    const int j = w - n_full;
    pw.slot = j % rem;
    pw.piece = (j < rem) ? 1 : 0;
    pw.u = n_full + pw.slot;
    pw.kb0 = pw.piece ? kblocks / 2 : 0;
    pw.kb1 = pw.piece ? kblocks : kblocks / 2;
  }
  return pw;
}

template <int BN, bool SWIGLU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ SwapXMaps tmX,
                             const __grid_constant__ CUtensorMap tmW,
                             const __grid_constant__ CUtensorMap tmY, const KArgs args) {
  pdl_begin();
  using C = Cfg2<BN, SWIGLU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smem + C::STAGES * C::A_STAGE;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *tmem_full = bars + 2 * C::STAGES;
  uint64_t *tmem_empty = tmem_full + 2;
  uint64_t *drain = tmem_full + 4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
  int32_t *mt = reinterpret_cast<int32_t *>(smem + C::MT_OFF);
  int32_t *sg = reinterpret_cast<int32_t *>(smem + C::SEG_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);

  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) {
    mt[i] = args.mtile_base[i];
    // offsets [E+1] (contiguous) or counts [E] (masked, two-segment)
    sg[i] = (args.layout == MOE_LAYOUT_CONTIGUOUS || i < args.E) ? args.seg[i] : 0;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 8);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  cluster_sync_all();  // both CTAs' barriers exist before any remote use
  const int total = mt[args.E] * args.n_tiles;
  const int kblocks = args.K / kBK;
  // split of a short last wave (down form): the last rem tiles as K halves
  int n_full = total, rem = 0;
  if (!SWIGLU && args.split_flags != nullptr && kblocks >= 2) {
    const int r = total % ncl;
    if (r > 0 && 2 * r <= ncl && r <= kPairSplitSlots && total / ncl <= kPairSplitMaxWaves &&
        (args.out_codes == nullptr || r <= args.split_part_slots)) {
      n_full = total - r;
      rem = r;
    }
  }
  const int items = n_full + 2 * rem;
  if (cid >= items) return;  // uniform across the pair

  if (warp == 1) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[C::STAGES];
      bool issued[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) issued[s] = false;
#pragma unroll
      for (int i = 0; i < 4; ++i) tma_prefetch_desc(&tmX.m[i]);
      if (SWIGLU) tma_prefetch_desc(&tmW);
      for (int w = cid; w < items && !*abort_flag; w += ncl) {
        const PairWork pw = pair_work(w, n_full, rem, kblocks);
        const Tile t = decode_tile<256>(args, mt, pw.u, sg);
        const int sn = (BN == 256) ? pair_swap_n(t) : 0;
        const int a_row = t.row0 + 128 * static_cast<int>(rank);
        int b_row;
        if (SWIGLU)  // even CTA: gate rows, odd CTA: the matching up rows
          b_row = t.e * args.b_rows + (even ? 0 : args.up_off) + t.n * C::HALF;
        else
          b_row = t.e * args.b_rows + t.n * BN + static_cast<int>(rank) * C::HALF;
        // swapped tile: this CTA's token rows, and (gate_up) its 16-row group
        // index in the 4-D weight map
        const int x_row = t.row0 + static_cast<int>(rank) * (sn >> 1);
        const int w_grp = (t.e * args.b_rows + t.n * C::BN_OUT + static_cast<int>(rank) * 64) >> 4;
        const int xbox = sn ? swap_box_index(sn) : 0;
        // TMA bytes of one k-block (both CTAs)
        const uint32_t tx =
            sn ? 2u * (C::A_BYTES + (8u << xbox) * kBK * 2u) : 2u * (C::A_BYTES + C::B_BYTES);
        for (int kb = pw.kb0; kb < pw.kb1; kb += C::KPS) {
          const int nk = min(C::KPS, pw.kb1 - kb);  // k-blocks in this stage
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status,
                                 args.wait_limit_ns))
            break;
          if (even) mbar_arrive_expect_tx(&full[stage], tx * static_cast<uint32_t>(nk));
          const uint32_t fbar = mapa_shared(&full[stage], 0);
          for (int i = 0; i < nk; ++i) {
            uint8_t *a_dst = smA + stage * C::A_STAGE + i * C::A_BYTES;
            uint8_t *b_dst = smB + stage * C::B_STAGE + i * C::B_BYTES;
            const int kc = (kb + i) * kBK;
            if (sn == 0) {
              tma_load_2d_pair(a_dst, &tmA, fbar, kc, a_row);
              tma_load_2d_pair(b_dst, &tmB, fbar, kc, b_row);
            } else {
              if (SWIGLU)
                tma_load_4d_pair(a_dst, &tmW, fbar, kc, 0, 0, w_grp);
              else
                tma_load_2d_pair(a_dst, &tmB, fbar, kc, b_row);
              tma_load_2d_pair(b_dst, &tmX.m[xbox], fbar, kc, x_row);
            }
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: the even CTA sees its full barriers; the odd CTA knows its
      // copies landed once the pair MMA that read them released the slot
      for (int s = 0; s < C::STAGES; ++s)
        if (issued[s]) {
          if (even)
            wait_drain(&full[s], issued_phase[s], args.wait_limit_ns);
          else
            wait_drain(&empty[s], issued_phase[s], args.wait_limit_ns);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && even) {
      // ---------------- pair MMA issuer (even CTA) ----------------
      constexpr uint32_t kIdesc = mma_idesc_bf16_f32(256, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool any_mma = false;
      for (int w = cid; w < items && !*abort_flag; w += ncl) {
        const PairWork pw = pair_work(w, n_full, rem, kblocks);
        const int sn = (BN == 256) ? pair_swap_n(decode_tile<256>(args, mt, pw.u, sg)) : 0;
        // swapped: the A slots hold weight rows (M) and the B slots token rows (N)
        const uint32_t idesc = sn ? mma_idesc_bf16_f32(256, sn) : kIdesc;
        if (!mbar_wait_bounded(&tmem_empty[acc], acc_phase ^ 1u, abort_flag, args.status,
                               args.wait_limit_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int kb = pw.kb0; kb < pw.kb1; kb += C::KPS) {
          const int nk = min(C::KPS, pw.kb1 - kb);
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.status,
                                 args.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int i = 0; i < nk; ++i) {
            const uint64_t ad =
                sw128_kmajor_desc(smem_u32(smA + stage * C::A_STAGE + i * C::A_BYTES));
            const uint64_t bd =
                sw128_kmajor_desc(smem_u32(smB + stage * C::B_STAGE + i * C::B_BYTES));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16_ss_pair(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc,
                               (kb + i != pw.kb0 || kk != 0) ? 1u : 0u);
          }
          any_mma = true;
          mma_commit_pair(&empty[stage], 0x3);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(&tmem_full[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (any_mma) {
        mma_commit_pair(drain, 0x1);
        wait_drain(drain, 0, args.wait_limit_ns);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5, both CTAs) ----------------
    const int quad = warp & 3;
    const int row = quad * 32 + lane;               // TMEM lane = row in this CTA's half
    const int prow = static_cast<int>(rank) * 128 + row;  // row within the 256-row tile
    const uint32_t empty_even = mapa_shared(&tmem_empty[0], 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = cid; w < items; w += ncl) {
      const PairWork pw = pair_work(w, n_full, rem, kblocks);
      const Tile t = decode_tile<256>(args, mt, pw.u, sg);
      const bool waited = mbar_wait_bounded(&tmem_full[acc], acc_phase, abort_flag,
                                            args.status, args.wait_limit_ns);
      if (!__all_sync(0xffffffffu, waited)) break;
      tc_fence_after();
      // split tile: this warp's part of the tile (its 32 TMEM lanes) has a
      // ticket word and a ready word, shared with the same part of the other
      // K half.  The half whose warp takes the ticket first stores its sums
      // and raises ready; the other waits for ready and adds its sums with
      // one fp32 reduction per element.  Either order gives fl(s0 + s1), and
      // the waiting half waits only for a warp already past its ticket, whose
      // stores wait on nothing, so no pair has to be resident at any time.
      uint32_t *ticket = (!SWIGLU && pw.piece >= 0)
                             ? args.split_flags + pw.slot * 16 +
                                   (static_cast<int>(rank) * 4 + quad) * 2
                             : nullptr;
      bool add = false;
      if (ticket != nullptr) {
        uint32_t prev = 0;
        if (lane == 0) prev = atomicExch(ticket, args.split_epoch);
        add = __shfl_sync(0xffffffffu, prev, 0) == args.split_epoch;
        if (add) {
          bool up = true;
          if (lane == 0)
            up = flag_wait_bounded(ticket + 1, args.split_epoch, abort_flag, args.status,
                                   args.wait_limit_ns);
          if (!__shfl_sync(0xffffffffu, up ? 1 : 0, 0)) break;
          (void)ld_acquire_gpu(ticket + 1);  // every lane acquires the stored sums
          __syncwarp();
          if (lane == 0) {  // both words cleared for the next launch (or replay)
            ticket[0] = 0;
            ticket[1] = 0;
          }
        }
      }
      const uint32_t tb =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      const int64_t grow = static_cast<int64_t>(t.row0) + prow;
      const bool ok = prow < t.rows_valid && grow >= 0 && grow < args.rows_total;
      const int sn = (BN == 256) ? pair_swap_n(t) : 0;
      // compact output: a split tile's halves meet in split_part (the first
      // stores its fp32 sums there, the second adds them to its own and
      // writes the tile), so every value is rounded to fp16 once
      const bool f16 = !SWIGLU && args.out_codes != nullptr;
      float *part = (f16 && ticket != nullptr)
                        ? args.split_part + static_cast<size_t>(pw.slot) * 256 * 256
                        : nullptr;
      const bool part_store = part != nullptr && !add;  // first half: partial sums only
      if (sn > 0) {
        // swapped tile: TMEM lane = weight row of this CTA's half, column =
        // token row of the tile
#pragma unroll 1
        for (int c0 = 0; c0 < sn; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tb + c0, v);
          tmem_ld_wait();
          tmem_regs_fence16(v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int r = c0 + i;
            const int64_t gr = static_cast<int64_t>(t.row0) + r;
            const bool rok = r < t.rows_valid && gr >= 0 && gr < args.rows_total;
            if (SWIGLU) {
              // lanes 0-15: gate of intermediate column j, lanes 16-31: its up
              const float mine = __uint_as_float(v[i]);
              const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
              if (lane < 16 && rok) {
                const int j = t.n * C::BN_OUT + static_cast<int>(rank) * 64 + quad * 16 + lane;
                const float h = __fdividef(mine, 1.0f + __expf(-mine)) * other;
                static_cast<__nv_bfloat16 *>(args.out)[gr * args.ldo + j] =
                    __float2bfloat16_rn(h);
              }
            } else if (rok) {  // rok is the same for the whole warp
              const int cl = static_cast<int>(rank) * 128 + quad * 32 + lane;
              const int col = t.n * BN + cl;
              float val = __uint_as_float(v[i]);
              if (f16) {
                if (part != nullptr) {
                  float *pp = part + static_cast<size_t>(r) * 256 + cl;
                  if (part_store)
                    *pp = val;
                  else
                    val = __fadd_rn(val, *pp);
                }
                if (!part_store) {
                  // the group is the warp's 32 consecutive columns of row r;
                  // non-negative floats order like their bit patterns
                  const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(val)));
                  const uint32_t cc = y16_code(__uint_as_float(mb));
                  static_cast<__half *>(args.out)[gr * args.ldo + col] =
                      __float2half_rn(val * y16_enc_mul(cc));
                  if (lane == 0) args.out_codes[gr * (args.ldo / 32) + col / 32] =
                      static_cast<uint8_t>(cc);
                }
              } else {
                float *o = static_cast<float *>(args.out) + gr * args.ldo + col;
                if (add)
                  red_add_f32(o, val);
                else
                  *o = val;
              }
            }
          }
        }
      } else if (SWIGLU) {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(args.out) + grow * args.ldo +
                             static_cast<int64_t>(t.n) * C::BN_OUT;
#pragma unroll 1
        for (int c = 0; c < C::BN_OUT / 32; ++c) {
          uint32_t g[32], v[32];
          tmem_ld_32x32b_x32(tb + c * 32, g);
          tmem_ld_32x32b_x32(tb + C::HALF + c * 32, v);
          tmem_ld_wait();
          tmem_regs_fence(g);
          tmem_regs_fence(v);
          if (ok) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float u0 = __uint_as_float(v[2 * i]), u1 = __uint_as_float(v[2 * i + 1]);
              const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
              const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
              packed[i] = pack_bf16x2(h0, h1);
            }
            if (args.out_v8) {
              // each lane writes whole 32-byte sectors of its row
              uint32_t w8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w8[i] = packed[i];
              st_global_v8(dst + c * 32, w8);
#pragma unroll
              for (int i = 0; i < 8; ++i) w8[i] = packed[8 + i];
              st_global_v8(dst + c * 32 + 16, w8);
            } else {
              uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                   packed[4 * i + 3]);
            }
          }
        }
      } else if (!SWIGLU && !f16 && pw.piece < 0 && args.out_tma &&
                 quad * 32 + static_cast<int>(rank) * 128 + 32 <=
                                                     t.rows_valid &&
                 grow - lane >= 0 && grow - lane + 32 <= args.rows_total) {
        // every row of this warp's 32-row slab is valid: each 32-column
        // chunk leaves as two TMA stores of 16 columns, each staged in one
        // half of the warp's box (row = lane, 16-byte pieces placed by the
        // 64-byte swizzle), so one half is filled while the other is stored
        uint8_t *box = smem + C::OUT_OFF + quad * C::OUT_BOX_BYTES;
        const int row_g = static_cast<int>(grow - lane);
        const uint32_t swz = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c * 32, v);
          tmem_ld_wait();
          tmem_regs_fence(v);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint8_t *hb = box + h * (C::OUT_BOX_BYTES / 2);
            const uint32_t rbase = smem_u32(hb) + static_cast<uint32_t>(lane) * 64u;
            if (lane == 0) bulk_wait_read_1();  // this half's previous store has read it
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(rbase + ((static_cast<uint32_t>(q) ^ swz) * 16u), v[16 * h + 4 * q],
                           v[16 * h + 4 * q + 1], v[16 * h + 4 * q + 2], v[16 * h + 4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmY, hb, t.n * BN + c * 32 + 16 * h, row_g);
              bulk_commit();
            }
          }
        }
      } else if (f16 && pw.piece < 0 && args.out_tma &&
                 quad * 32 + static_cast<int>(rank) * 128 + 32 <= t.rows_valid &&
                 grow - lane >= 0 && grow - lane + 32 <= args.rows_total) {
        // compact output, every row of this warp's 32-row slab valid: each
        // 32-column chunk becomes 32 fp16 values per row, staged as a 32 x 32
        // box (64-byte rows, 64-byte swizzle) in one half of the warp's
        // staging area and written by one TMA store, the halves alternating;
        // the lane writes its row's 8 code bytes of the tile at the end
        uint8_t *box = smem + C::OUT_OFF + quad * C::OUT_BOX_BYTES;
        const int row_g = static_cast<int>(grow - lane);
        const uint32_t swz = static_cast<uint32_t>((lane >> 1) & 3);
        uint64_t codes = 0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c * 32, v);
          tmem_ld_wait();
          tmem_regs_fence(v);
          uint32_t hw[16];
          const uint32_t cc = y16_encode32(v, hw);
          codes |= static_cast<uint64_t>(cc) << (8 * c);
          uint8_t *hb = box + (c & 1) * (C::OUT_BOX_BYTES / 2);
          const uint32_t rbase = smem_u32(hb) + static_cast<uint32_t>(lane) * 64u;
          if (lane == 0) bulk_wait_read_1();  // this half's previous store has read it
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_shared_v4(rbase + ((static_cast<uint32_t>(q) ^ swz) * 16u), hw[4 * q],
                         hw[4 * q + 1], hw[4 * q + 2], hw[4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmY, hb, t.n * BN + c * 32, row_g);
            bulk_commit();
          }
        }
        *reinterpret_cast<uint64_t *>(args.out_codes + grow * (args.ldo / 32) +
                                      static_cast<int64_t>(t.n) * (BN / 32)) = codes;
      } else if (f16) {
        // compact output: 32 fp16 values (64 bytes) and one code per chunk
        __half *dst = static_cast<__half *>(args.out) + grow * args.ldo +
                      static_cast<int64_t>(t.n) * BN;
        uint64_t codes = 0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c * 32, v);
          tmem_ld_wait();
          tmem_regs_fence(v);
          float4 *pp = part != nullptr ? reinterpret_cast<float4 *>(
                                             part + static_cast<size_t>(prow) * 256 + c * 32)
                                       : nullptr;
          if (ok && part_store) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              pp[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                  __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
          } else if (ok) {
            if (pp != nullptr) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 o = pp[q];
                v[4 * q] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * q]), o.x));
                v[4 * q + 1] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * q + 1]), o.y));
                v[4 * q + 2] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * q + 2]), o.z));
                v[4 * q + 3] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * q + 3]), o.w));
              }
            }
            uint32_t hw[16];
            const uint32_t cc = y16_encode32(v, hw);
            uint32_t w8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) w8[q] = hw[q];
            st_global_v8(dst + c * 32, w8);
#pragma unroll
            for (int q = 0; q < 8; ++q) w8[q] = hw[8 + q];
            st_global_v8(dst + c * 32 + 16, w8);
            codes |= static_cast<uint64_t>(cc) << (8 * c);
          }
        }
        if (ok && !part_store) {
          uint8_t *cd = args.out_codes + grow * (args.ldo / 32) + static_cast<int64_t>(t.n) * (BN / 32);
          if (BN / 32 == 8)
            *reinterpret_cast<uint64_t *>(cd) = codes;
          else
            for (int c = 0; c < BN / 32; ++c) cd[c] = static_cast<uint8_t>(codes >> (8 * c));
        }
      } else {
        float *dst = static_cast<float *>(args.out) + grow * args.ldo +
                     static_cast<int64_t>(t.n) * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c * 32, v);
          tmem_ld_wait();
          tmem_regs_fence(v);
          if (ok) {
            if (add) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                red_add_v4(dst + c * 32 + 4 * i, __uint_as_float(v[4 * i]),
                           __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                           __uint_as_float(v[4 * i + 3]));
            } else if (args.out_v8) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t w8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) w8[j] = v[8 * i + j];
                st_global_v8(dst + c * 32 + 8 * i, w8);
              }
            } else {
              float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            }
          }
        }
      }
      if (ticket != nullptr && !add) {
        // the first K half to arrive: its sums are stored; raise ready
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(ticket + 1, args.split_epoch);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (even)
          mbar_arrive(&tmem_empty[acc]);
        else
          mbar_arrive_remote(empty_even + static_cast<uint32_t>(acc) * 8u);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!SWIGLU && lane == 0) bulk_wait_all();  // output stores written before exit
  }

  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while its peer may still use its memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// FP8 (e4m3) grouped GEMM with power-of-two block scales applied by the
// tensor cores.  A rows carry one scale per 128 columns, B (weights) one per
// 128 x 128 block; a k-block is 128 columns: one scale block, one 128-byte
// swizzle row and four block-scaled MMAs (kind::mxf8f6f4, M=128, N=128,
// K=32) that take both scales from TMEM as 8-bit exponents and accumulate
// the whole K loop in one TMEM accumulator (two, alternating between tiles,
// so a tile's epilogue overlaps the next tile's MMAs).
// The exponents sit in a ring of 8-column TMEM slots, each serving four
// consecutive k-blocks of a tile: columns 0-3 hold row m's A exponent at
// lane m, column m / 32; columns 4-7 hold tile column n's B exponent at lane
// 32q + n % 32 in every lane quadrant q, column 4 + n / 32 (gate_up: columns
// 0-63 of the tile are gate rows, 64-127 up rows, each with its own weight
// block); byte j of a cell is k-block 4g + j's exponent, which the MMAs of
// that k-block select with scale factor id j.
// Roles: warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 scale writers
// (one per TMEM lane quadrant), warps 6-13 epilogue (two per quadrant, each
// half of the tile's columns).
//   full/empty[s]    stage ring (producer and scale writers <-> MMA);
//   sfull/sempty[g]  scale slot g written (four scale warps) / read by the
//                    MMAs of its k-blocks;
//   afull/aempty[b]  accumulator b (MMA <-> eight epilogue warps).
// ---------------------------------------------------------------------------
constexpr int kF8BK = 128;  // e4m3 per k-block = bytes per swizzle row
constexpr int kF8BN = 128;
constexpr int kF8Stages = 6;
constexpr int kF8Threads = 448;
constexpr int kF8ScaleCol = 2 * kF8BN;  // first TMEM column of the scale slots
constexpr int kF8ScaleSlots = 4;        // 8-column slots, each holding 4 k-blocks' exponents
constexpr int kF8TmemCols = 512;

template <bool SWIGLU>
struct CfgF8 {
  static constexpr int A_BYTES = kBM * kF8BK;
  static constexpr int B_BYTES = kF8BN * kF8BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = kF8Stages;
  static constexpr int BN_OUT = SWIGLU ? kF8BN / 2 : kF8BN;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * kF8ScaleSlots + 4 + 1;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int MT_OFF = MISC_OFF + 16;
  static constexpr int SMEM_BYTES = MT_OFF + (kMaxE + 1) * 4 + 1024;
  static_assert(SMEM_BYTES <= 232448, "227 KB of shared memory per CTA");
  static_assert(kF8ScaleCol + 8 * kF8ScaleSlots <= kF8TmemCols,
                "scale slots fit the TMEM allocation");
};

struct F8Args {
  KArgs k;              // tiles, layout, output (k.K = reduction length)
  const float *a_scale;  // [rows_total, K/128]
  const float *b_scale;  // [E, b_rows/128, K/128]
};

// A tile of fewer than 128 rows loads only ceil(rows / 32) boxes of 32 rows;
// the shared-memory rows past them are stale and only feed accumulator rows
// that are never written.
constexpr int kF8SubRows = 32;

// The UE8M0 byte (the biased exponent) of a power-of-two scale in
// [2^-127, 2^127]; false for any other value.
__device__ __forceinline__ bool ue8m0_of(float s, uint32_t &byte) {
  const uint32_t b = __float_as_uint(s);
  byte = (b >> 23) & 0xffu;
  return ((b & 0x807fffffu) == 0u && byte != 0u && byte != 0xffu) || b == 0x00400000u;
}

// One epilogue thread's part of an FP8 tile row: acc holds two 32-column
// runs of the accumulator, written at output column col of row grow.
// gate_up: 32 gate columns, then their up columns -> 32 values of h (bf16,
// SwiGLU); down: 64 consecutive columns -> compact rows or fp32.
template <bool SWIGLU>
__device__ __forceinline__ void f8_store_tile_row(const KArgs &args, int64_t grow, int64_t col,
                                                  const float (&acc)[64]) {
  if (SWIGLU) {
    // gate acc[0..31], up acc[32..63]
    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(args.out) + grow * args.ldo + col;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t w8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = c * 16 + 2 * i;
        const float g0 = acc[j], g1 = acc[j + 1];
        const float u0 = acc[32 + j], u1 = acc[32 + j + 1];
        w8[i] = pack_bf16x2(__fdividef(g0, 1.0f + __expf(-g0)) * u0,
                            __fdividef(g1, 1.0f + __expf(-g1)) * u1);
      }
      if (args.out_v8) {
        st_global_v8(dst + c * 16, w8);
      } else {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 16);
        d4[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
        d4[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
      }
    }
  } else if (args.out_codes != nullptr) {
    // compact output: the thread's 64 columns are two 32-column groups,
    // 128 bytes of fp16 values and two code bytes
    __half *dst = static_cast<__half *>(args.out) + grow * args.ldo + col;
    uint32_t codes = 0;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      uint32_t vv[32], hw[16];
#pragma unroll
      for (int i = 0; i < 32; ++i) vv[i] = __float_as_uint(acc[32 * g + i]);
      codes |= y16_encode32(vv, hw) << (8 * g);
      uint32_t w8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w8[i] = hw[i];
      st_global_v8(dst + 32 * g, w8);
#pragma unroll
      for (int i = 0; i < 8; ++i) w8[i] = hw[8 + i];
      st_global_v8(dst + 32 * g + 16, w8);
    }
    *reinterpret_cast<uint16_t *>(args.out_codes + grow * (args.ldo / 32) + col / 32) =
        static_cast<uint16_t>(codes);
  } else {
    float *dst = static_cast<float *>(args.out) + grow * args.ldo + col;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t w8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w8[i] = __float_as_uint(acc[c * 8 + i]);
      if (args.out_v8) {
        st_global_v8(dst + c * 8, w8);
      } else {
        float4 *d4 = reinterpret_cast<float4 *>(dst + c * 8);
        d4[0] = make_float4(acc[c * 8], acc[c * 8 + 1], acc[c * 8 + 2], acc[c * 8 + 3]);
        d4[1] = make_float4(acc[c * 8 + 4], acc[c * 8 + 5], acc[c * 8 + 6], acc[c * 8 + 7]);
      }
    }
  }
}

// SwiGLU of a thread's 32 gate values v and their up values w, rounded to
// bf16 (h's storage format), two per register in column order.
__device__ __forceinline__ void f8_swiglu_bf16(const uint32_t (&v)[32], const uint32_t (&w)[32],
                                               uint32_t (&hb)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float g0 = __uint_as_float(v[2 * i]), g1 = __uint_as_float(v[2 * i + 1]);
    const float u0 = __uint_as_float(w[2 * i]), u1 = __uint_as_float(w[2 * i + 1]);
    hb[i] = pack_bf16x2(__fdividef(g0, 1.0f + __expf(-g0)) * u0,
                        __fdividef(g1, 1.0f + __expf(-g1)) * u1);
  }
}

__device__ __forceinline__ float f8_bf16x2_absmax(const uint32_t (&hb)[16], float m) {
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fmaxf(fabsf(bf16lo(hb[i])), fabsf(bf16hi(hb[i]))));
  return m;
}

// 32 bf16 values of h -> their e4m3 codes at dst (32 bytes, 32-byte aligned),
// times the exact reciprocal of the power-of-two scale: the codes of the
// row quantizer.
__device__ __forceinline__ void f8_store_codes32(uint8_t *dst, const uint32_t (&hb)[16],
                                                 float inv) {
  uint32_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = hb[2 * i], b = hb[2 * i + 1];
    q[i] = static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16lo(a), inv), __fmul_rn(bf16hi(a), inv))) |
           (static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16lo(b), inv), __fmul_rn(bf16hi(b), inv)))
            << 16);
  }
  st_global_v8(dst, q);
}

// The fused h quantization of one tile row (gate_up, 256-column tiles): the
// row's 128 h columns, one scale block, are held by two threads (parts 0 and
// 1, warps w and w + 4 of one lane quadrant) as two 32-column runs each
// (halves 0 and 1).  Each warp posts its rows' partial maxima in xch
// (double-buffered by use), arrives on the quadrant's barrier, waits for
// the other warp (bounded) and quantizes its runs with the row's scale.
// Returns false if the wait ran out.
__device__ __forceinline__ bool f8_quantize_row(const KArgs &args, const Tile &t, int64_t grow,
                                                bool rok, int row, int part, uint32_t use,
                                                const uint32_t (&h0)[16], const uint32_t (&h1)[16],
                                                float *xch, uint64_t *xbar,
                                                volatile int *abort_flag) {
  const int lane = threadIdx.x & 31;
  float m = rok ? f8_bf16x2_absmax(h1, f8_bf16x2_absmax(h0, 0.0f)) : 0.0f;
  float *buf = xch + (use & 1u) * 256;
  buf[part * 128 + row] = m;
  __syncwarp();
  if (lane == 0) mbar_arrive(xbar);
  const bool waited = mbar_wait_bounded(xbar, use & 1u, abort_flag, args.status,
                                        args.wait_limit_ns);
  if (!__all_sync(0xffffffffu, waited)) return false;
  m = fmaxf(m, buf[(1 - part) * 128 + row]);
  if (rok) {
    const float sc = fp8_block_scale(m);
    const float inv = __frcp_rn(sc);  // exact: sc is a power of two
    uint8_t *dst = static_cast<uint8_t *>(args.out) + grow * args.ldo +
                   static_cast<int64_t>(t.n) * 128 + 32 * part;
    f8_store_codes32(dst, h0, inv);
    f8_store_codes32(dst + 64, h1, inv);
    if (part == 0) args.out_h_scales[grow * (args.ldo / 128) + t.n] = sc;
  }
  return true;
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kF8Threads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmA32,
                            const __grid_constant__ CUtensorMap tmB, const F8Args fa) {
  pdl_begin();
  using C = CfgF8<SWIGLU>;
  const KArgs &args = fa.k;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smem + C::STAGES * C::A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *sfull = bars + 2 * C::STAGES;
  uint64_t *sempty = sfull + kF8ScaleSlots;
  uint64_t *afull = sempty + kF8ScaleSlots;
  uint64_t *aempty = afull + 2;
  uint64_t *drain = aempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
  int32_t *mt = reinterpret_cast<int32_t *>(smem + C::MT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) mt[i] = args.mtile_base[i];
  if (threadIdx.x == 0) {
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    for (int g = 0; g < kF8ScaleSlots; ++g) {
      mbar_init(&sfull[g], 4);
      mbar_init(&sempty[g], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 8);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int total = mt[args.E] * args.n_tiles;
  if (blockIdx.x >= total) return;
  if (warp == 1) tmem_alloc(tmem_slot, kF8TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int kblocks = args.K / kF8BK;
  const int kbs = kblocks;  // scale blocks along K
  const int b_blocks = args.b_rows / 128;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA32);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[C::STAGES];
      bool issued[C::STAGES];
#pragma unroll
      for (int st = 0; st < C::STAGES; ++st) issued[st] = false;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        const Tile t = decode_tile(args, mt, u);
        const int subs = (t.rows_valid + kF8SubRows - 1) / kF8SubRows;  // 1..4
        const uint32_t tx = C::B_BYTES + (subs < kBM / kF8SubRows ? subs * kF8SubRows * kF8BK
                                                                  : C::A_BYTES);
        int b0, b1;
        if (SWIGLU) {
          b0 = t.e * args.b_rows + t.n * C::BN_OUT;
          b1 = t.e * args.b_rows + args.up_off + t.n * C::BN_OUT;
        } else {
          b0 = t.e * args.b_rows + t.n * kF8BN;
          b1 = b0 + kF8BN / 2;
        }
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status,
                                 args.wait_limit_ns))
            break;
          uint8_t *a_dst = smA + stage * C::A_BYTES;
          uint8_t *b_dst = smB + stage * C::B_BYTES;
          mbar_arrive_expect_tx(&full[stage], tx);
          if (subs < kBM / kF8SubRows) {
            for (int i = 0; i < subs; ++i)
              tma_load_2d(a_dst + i * kF8SubRows * kF8BK, &tmA32, &full[stage], kb * kF8BK,
                          t.row0 + i * kF8SubRows);
          } else {
            tma_load_2d(a_dst, &tmA, &full[stage], kb * kF8BK, t.row0);
          }
          tma_load_2d(b_dst, &tmB, &full[stage], kb * kF8BK, b0);
          tma_load_2d(b_dst + (kF8BN / 2) * kF8BK, &tmB, &full[stage], kb * kF8BK, b1);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int st = 0; st < C::STAGES; ++st)
        if (issued[st]) wait_drain(&full[st], issued_phase[st], args.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t kIdesc = mma_idesc_mxf8_f32(kBM, kF8BN);
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t sphase = 0;
      uint32_t tcount = 0;  // tiles issued: accumulator tcount % 2, its use tcount / 2
      bool any_mma = false;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok && !*abort_flag; u += gridDim.x, ++tcount) {
        const uint32_t b = tcount & 1u;
        if (!mbar_wait_bounded(&aempty[b], ((tcount >> 1) & 1u) ^ 1u, abort_flag, args.status,
                               args.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kF8BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          const int j = kb & 3;  // byte of the slot's cells with this k-block's exponents
          if ((j == 0 && !mbar_wait_bounded(&sfull[slot], sphase, abort_flag, args.status,
                                            args.wait_limit_ns)) ||
              !mbar_wait_bounded(&full[stage], phase, abort_flag, args.status,
                                 args.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(smA + stage * C::A_BYTES));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(smB + stage * C::B_BYTES));
          const uint32_t sfa = tmem_base + static_cast<uint32_t>(kF8ScaleCol + 8 * slot);
          const uint32_t idesc =
              kIdesc | (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
#pragma unroll
          for (int kk = 0; kk < kF8BK / 32; ++kk)  // +32 bytes = 32 e4m3 along K
            mma_mxf8_ss(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, sfa, sfa + 4u,
                        (kb != 0 || kk != 0) ? 1u : 0u);
          any_mma = true;
          mma_commit(&empty[stage]);
          if (j == 3 || kb == kblocks - 1) {
            mma_commit(&sempty[slot]);
            if (++slot == kF8ScaleSlots) {
              slot = 0;
              sphase ^= 1u;
            }
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&afull[b]);
      }
      if (any_mma) {
        mma_commit(drain);
        wait_drain(drain, 0, args.wait_limit_ns);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------- scale writers (warps 2..5) ----------------
    // The warp of lane quadrant q writes, per four k-blocks, lanes
    // 32q..32q+31 of a scale slot: its rows' A exponents (columns 0-3) and
    // the tile's B exponents (columns 4-7: two gate, two up for gate_up).
    // Scales are loaded a group of four k-blocks ahead.
    const int quad = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int row = quad * 32 + lane;
    int slot = 0;
    uint32_t sphase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok && !*abort_flag; u += gridDim.x) {
      const Tile t = decode_tile(args, mt, u);
      const int64_t grow = static_cast<int64_t>(t.row0) + row;
      const bool rok = row < t.rows_valid && grow >= 0 && grow < args.rows_total;
      const float *as = fa.a_scale + (rok ? grow : 0) * kbs;
      const float *bs0, *bs1;
      if (SWIGLU) {
        bs0 = fa.b_scale + (static_cast<int64_t>(t.e) * b_blocks + (t.n * C::BN_OUT) / 128) * kbs;
        bs1 = fa.b_scale +
              (static_cast<int64_t>(t.e) * b_blocks + (args.up_off + t.n * C::BN_OUT) / 128) * kbs;
      } else {
        bs0 = bs1 = fa.b_scale + (static_cast<int64_t>(t.e) * b_blocks + t.n) * kbs;
      }
      float ca[4], cg[4], cu[4];
      auto load4 = [&](int kb0, float(&a)[4], float(&g)[4], float(&uu)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kb = kb0 + i;
          const bool in = kb < kblocks;
          a[i] = (in && rok) ? __ldg(as + kb) : 1.0f;
          g[i] = in ? __ldg(bs0 + kb) : 1.0f;
          uu[i] = in ? __ldg(bs1 + kb) : 1.0f;
        }
      };
      load4(0, ca, cg, cu);
      for (int kb0 = 0; kb0 < kblocks && ok; kb0 += 4) {
        float na[4], ng[4], nu[4];
        load4(kb0 + 4, na, ng, nu);
        // byte i of each cell: k-block kb0 + i (past the tile's last k-block: 2^0)
        uint32_t va = 0, vg = 0, vu = 0;
        bool valid = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t ba, bg, bu;
          valid = valid & ue8m0_of(ca[i], ba) & ue8m0_of(cg[i], bg) & ue8m0_of(cu[i], bu);
          va |= ba << (8 * i);
          vg |= bg << (8 * i);
          vu |= bu << (8 * i);
        }
        if (!valid) set_status(args.status, kStatusBadId);
        const bool waited = mbar_wait_bounded(&sempty[slot], sphase ^ 1u, abort_flag,
                                              args.status, args.wait_limit_ns);
        if (!__all_sync(0xffffffffu, waited)) {
          ok = false;
          break;
        }
        const uint32_t v[8] = {va, va, va, va, vg, vg, vu, vu};
        tmem_st_32x32b_x8(tmem_base + lane_off + static_cast<uint32_t>(kF8ScaleCol + 8 * slot), v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[slot]);
        if (++slot == kF8ScaleSlots) {
          slot = 0;
          sphase ^= 1u;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ca[i] = na[i];
          cg[i] = ng[i];
          cu[i] = nu[i];
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 6..13) ----------------
    // Warp w handles TMEM lane quadrant w % 4 and column half h = (w - 6) / 4:
    // gate_up: gate columns 32h .. 32h+31 and the matching up columns
    // 64 + 32h .. (so SwiGLU stays in the thread); down: columns 64h .. 64h+63.
    const int quad = warp & 3;
    const int half = (warp - 6) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int col0 = SWIGLU ? 32 * half : 64 * half;            // first TMEM column
    const int col1 = SWIGLU ? kF8BN / 2 + 32 * half : col0 + 32;  // second 32-column run
    uint32_t tcount = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++tcount) {
      const Tile t = decode_tile(args, mt, u);
      const int64_t grow = static_cast<int64_t>(t.row0) + row;
      const bool rok = row < t.rows_valid && grow >= 0 && grow < args.rows_total;
      const uint32_t b = tcount & 1u;
      const bool waited = mbar_wait_bounded(&afull[b], (tcount >> 1) & 1u, abort_flag,
                                            args.status, args.wait_limit_ns);
      if (!__all_sync(0xffffffffu, waited)) break;
      tc_fence_after();
      // a warp whose 32 rows are all past the tile's rows only releases
      const bool warp_rows = quad * 32 < t.rows_valid;
      uint32_t v[32], w[32];
      if (warp_rows) {
        const uint32_t tp = tmem_base + lane_off + b * kF8BN;
        tmem_ld_32x32b_x32(tp + col0, v);
        tmem_ld_32x32b_x32(tp + col1, w);
        tmem_ld_wait();
        tmem_regs_fence(v);
        tmem_regs_fence(w);
      }
      // the accumulator is released as soon as its values are in registers
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[b]);
      if (!warp_rows || !rok) continue;
      float acc[64];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        acc[c] = __uint_as_float(v[c]);
        acc[32 + c] = __uint_as_float(w[c]);
      }
      f8_store_tile_row<SWIGLU>(
          args, grow,
          SWIGLU ? static_cast<int64_t>(t.n) * (kF8BN / 2) + 32 * half
                 : static_cast<int64_t>(t.n) * kF8BN + 64 * half,
          acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kF8TmemCols);
}

// ---------------------------------------------------------------------------
// The same FP8 GEMM on a cluster of two CTAs (cta_group::2 block-scaled
// MMAs) with 256 x 256 tiles: one M=256 x N=256 MMA per K step, the even
// CTA's 128 B rows giving accumulator columns 0-127 (half 0) and the odd
// CTA's columns 128-255 (half 1).  (Two N=128 MMAs per step would read the A
// tile from shared memory twice; shared-memory bandwidth, not the tensor
// core, then sets the pace.)  The accumulator windows alternate between
// TMEM columns [0, 256) (even tiles) and [128, 384) (odd tiles), three
// 128-column slots in all; the epilogue reads the middle slot first and
// releases it, so the next tile's MMAs wait only for that read, and a
// slot's other user is two tiles back.  Each CTA loads 128 A rows and 128 B
// rows per stage (32 KB, 6 stages).  gate_up: the even CTA loads gate rows
// i0 .. i0+63 and their up rows, the odd CTA gate rows i0+64 .. i0+127 and
// theirs (i0 = 128 t.n), so each half holds 64 gate columns and their 64 up
// columns; down: CTA r loads output rows c0 + 128r .. c0 + 128r + 127.
// Each CTA's MMA half reads its exponents from its own TMEM in the 1-CTA
// layout (N = 256: B column n's exponent at lane 32q + n % 32, column
// n / 32); a scale slot has 16 columns: A (0-3), B (4-11).  An expert's
// last tile may leave the odd CTA without A rows: it then loads only its B
// rows.  The down form's compact rows leave through TMA tensor stores: each
// epilogue warp whose 32 rows are all valid stages a 32 x 32 fp16 box
// (64-byte swizzle) in its own 2 KB of shared memory per 32-column group
// (per-thread 32-byte global stores kept the load/store queue full).
//   full[s]          even CTA: both CTAs' copies of stage s landed;
//   empty[s]         both CTAs: the pair MMAs that read stage s completed;
//   sfull[g]         even CTA: both CTAs' exponents of scale slot g are in TMEM;
//   sempty[g]        both CTAs: the pair MMAs that read slot g completed;
//   hfull[b]         both CTAs: TMEM slot b holds a complete tile half;
//   hempty[b]        even CTA: both CTAs' epilogue warps have read slot b.
// ---------------------------------------------------------------------------
constexpr int kF8PairStages = 6;
constexpr int kF8PairBN = 256;
constexpr int kF8PairSlotCols = 16;
constexpr int kF8PairScaleCol = 3 * 128;  // after the three accumulator slots

template <bool SWIGLU>
struct CfgF8P {
  static constexpr int A_BYTES = kBM * kF8BK;
  static constexpr int B_BYTES = (kF8PairBN / 2) * kF8BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = kF8PairStages;
  static constexpr int BN_OUT = SWIGLU ? kF8PairBN / 2 : kF8PairBN;
  // down: one 32 x 32 fp16 staging box per epilogue warp (compact rows);
  // gate_up: the row maxima exchanged by the fused h quantization
  static constexpr int OUT_OFF = STAGES * STAGE_BYTES;
  static constexpr int OUT_BOX_BYTES = 32 * 32 * 2;
  static constexpr int OUT_BYTES = SWIGLU ? 2 * 2 * 128 * 4 : 8 * OUT_BOX_BYTES;
  static constexpr int BAR_OFF = OUT_OFF + OUT_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * kF8ScaleSlots + 2 * 3 + 1 + 4;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int MT_OFF = MISC_OFF + 16;
  static constexpr int SEG_OFF = MT_OFF + (kMaxE + 1) * 4;
  static constexpr int SMEM_BYTES = SEG_OFF + (kMaxE + 1) * 4 + 1024;
  static_assert(SMEM_BYTES <= 232448, "227 KB of shared memory per CTA");
  static_assert(OUT_OFF % 2048 == 0, "swizzled staging alignment");
  static_assert(kF8PairScaleCol + kF8PairSlotCols * kF8ScaleSlots <= kF8TmemCols,
                "scale slots fit the TMEM allocation");
};

// D (M=256: rows 0-127 in this CTA's TMEM, 128-255 in the peer's) (+)=
// block-scaled e4m3 A (128 rows per CTA) * B^T (N/2 rows per CTA); each CTA's
// half reads its exponents from its own TMEM at sfa_tmem / sfb_tmem.
__device__ __forceinline__ void mma_mxf8_ss_pair(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Whole warp: thread i writes v[j] to lane (base lane + i), column col + j.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

// TMA bytes of A that one CTA of the pair loads for a tile with rows_valid
// rows (its 128-row half: none, 32-row boxes, or one 128-row box)
__device__ __forceinline__ uint32_t f8_pair_a_bytes(int rows_valid, int rank) {
  const int here = min(max(rows_valid - 128 * rank, 0), 128);
  const int subs = (here + kF8SubRows - 1) / kF8SubRows;
  return static_cast<uint32_t>(subs) * kF8SubRows * kF8BK;
}

template <bool SWIGLU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kF8Threads, 1)
    grouped_gemm_fp8_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                                 const __grid_constant__ CUtensorMap tmA32,
                                 const __grid_constant__ CUtensorMap tmB,
                                 const __grid_constant__ CUtensorMap tmY, const F8Args fa) {
  pdl_begin();
  using C = CfgF8P<SWIGLU>;
  const KArgs &args = fa.k;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smem + C::STAGES * C::A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *sfull = bars + 2 * C::STAGES;
  uint64_t *sempty = sfull + kF8ScaleSlots;
  uint64_t *hfull = sempty + kF8ScaleSlots;
  uint64_t *hempty = hfull + 3;
  uint64_t *drain = hempty + 3;
  uint64_t *xbar = drain + 1;  // per lane quadrant: the fused h quantization's exchange
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
  int32_t *mt = reinterpret_cast<int32_t *>(smem + C::MT_OFF);
  int32_t *sg = reinterpret_cast<int32_t *>(smem + C::SEG_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) {
    mt[i] = args.mtile_base[i];
    sg[i] = (args.layout == MOE_LAYOUT_CONTIGUOUS || i < args.E) ? args.seg[i] : 0;
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    for (int g = 0; g < kF8ScaleSlots; ++g) {
      mbar_init(&sfull[g], 8);
      mbar_init(&sempty[g], 1);
    }
    for (int b = 0; b < 3; ++b) {
      mbar_init(&hfull[b], 1);
      mbar_init(&hempty[b], 16);
    }
    mbar_init(drain, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&xbar[q], 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  cluster_sync_all();  // both CTAs' barriers exist before any remote use
  const int total = mt[args.E] * args.n_tiles;
  if (cid >= total) return;  // uniform across the pair
  if (warp == 1) tmem_alloc_pair(tmem_slot, kF8TmemCols);
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int kblocks = args.K / kF8BK;
  const int kbs = kblocks;
  const int b_blocks = args.b_rows / 128;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA32);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[C::STAGES];
      bool issued[C::STAGES];
#pragma unroll
      for (int st = 0; st < C::STAGES; ++st) issued[st] = false;
      for (int u = cid; u < total && !*abort_flag; u += ncl) {
        const Tile t = decode_tile<256>(args, mt, u, sg);
        const uint32_t a_here = f8_pair_a_bytes(t.rows_valid, static_cast<int>(rank));
        // both CTAs' bytes of one k-block, expected on the even CTA's barrier
        const uint32_t tx = 2u * C::B_BYTES + f8_pair_a_bytes(t.rows_valid, 0) +
                            f8_pair_a_bytes(t.rows_valid, 1);
        const int a_row = t.row0 + 128 * static_cast<int>(rank);
        int b_row0, b_row1;  // this CTA's B rows for smem rows 0-63 and 64-127
        if (SWIGLU) {
          b_row0 = t.e * args.b_rows + t.n * C::BN_OUT + 64 * static_cast<int>(rank);
          b_row1 = b_row0 + args.up_off;
        } else {
          b_row0 = t.e * args.b_rows + t.n * kF8PairBN + 128 * static_cast<int>(rank);
          b_row1 = b_row0 + 64;
        }
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status,
                                 args.wait_limit_ns))
            break;
          if (even) mbar_arrive_expect_tx(&full[stage], tx);
          const uint32_t fbar = mapa_shared(&full[stage], 0);
          uint8_t *a_dst = smA + stage * C::A_BYTES;
          uint8_t *b_dst = smB + stage * C::B_BYTES;
          if (a_here == static_cast<uint32_t>(C::A_BYTES)) {
            tma_load_2d_pair(a_dst, &tmA, fbar, kb * kF8BK, a_row);
          } else {
            for (uint32_t i = 0; i * kF8SubRows * kF8BK < a_here; ++i)
              tma_load_2d_pair(a_dst + i * kF8SubRows * kF8BK, &tmA32, fbar, kb * kF8BK,
                               a_row + static_cast<int>(i) * kF8SubRows);
          }
          tma_load_2d_pair(b_dst, &tmB, fbar, kb * kF8BK, b_row0);
          tma_load_2d_pair(b_dst + 64 * kF8BK, &tmB, fbar, kb * kF8BK, b_row1);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: the even CTA sees its full barriers; the odd CTA knows its
      // copies landed once the pair MMA that read them released the slot
      for (int st = 0; st < C::STAGES; ++st)
        if (issued[st]) {
          if (even)
            wait_drain(&full[st], issued_phase[st], args.wait_limit_ns);
          else
            wait_drain(&empty[st], issued_phase[st], args.wait_limit_ns);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && even) {
      // ---------------- pair MMA issuer (even CTA) ----------------
      constexpr uint32_t kIdesc = mma_idesc_mxf8_f32(256, kF8PairBN);
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t sphase = 0;
      uint32_t tcount = 0;
      uint32_t hpar = 0;  // bit b: parity of slot b's next use
      bool any_mma = false;
      bool ok = true;
      for (int u = cid; u < total && ok && !*abort_flag; u += ncl, ++tcount) {
        const uint32_t h0 = tcount & 1u, h1 = h0 + 1u;  // the tile's two slots
        if (!mbar_wait_bounded(&hempty[h0], ((hpar >> h0) & 1u) ^ 1u, abort_flag, args.status,
                               args.wait_limit_ns) ||
            !mbar_wait_bounded(&hempty[h1], ((hpar >> h1) & 1u) ^ 1u, abort_flag, args.status,
                               args.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + 128u * h0;
        for (int kb = 0; kb < kblocks; ++kb) {
          const int j = kb & 3;  // byte of the slot's cells with this k-block's exponents
          if ((j == 0 && !mbar_wait_bounded(&sfull[slot], sphase, abort_flag, args.status,
                                            args.wait_limit_ns)) ||
              !mbar_wait_bounded(&full[stage], phase, abort_flag, args.status,
                                 args.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(smA + stage * C::A_BYTES));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(smB + stage * C::B_BYTES));
          const uint32_t sfa =
              tmem_base + static_cast<uint32_t>(kF8PairScaleCol + kF8PairSlotCols * slot);
          const uint32_t idesc =
              kIdesc | (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
#pragma unroll
          for (int kk = 0; kk < kF8BK / 32; ++kk) {
            mma_mxf8_ss_pair(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, sfa, sfa + 4u,
                             (kb != 0 || kk != 0) ? 1u : 0u);
          }
          any_mma = true;
          mma_commit_pair(&empty[stage], 0x3);
          if (j == 3 || kb == kblocks - 1) {
            mma_commit_pair(&sempty[slot], 0x3);
            if (++slot == kF8ScaleSlots) {
              slot = 0;
              sphase ^= 1u;
            }
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(&hfull[h0], 0x3);
        mma_commit_pair(&hfull[h1], 0x3);
        hpar ^= (1u << h0) | (1u << h1);
      }
      if (any_mma) {
        mma_commit_pair(drain, 0x1);
        wait_drain(drain, 0, args.wait_limit_ns);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------- scale writers (warps 2..5, both CTAs) ----------------
    // Per four k-blocks, lanes 32q..32q+31 of a slot: this CTA's rows' A
    // exponents (columns 0-3) and both halves' B exponents (4-7, 8-11;
    // gate_up: two gate, two up columns each, down: one block per half).
    const int quad = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int prow = static_cast<int>(rank) * 128 + quad * 32 + lane;  // row in the 256-row tile
    int slot = 0;
    uint32_t sphase = 0;
    bool ok = true;
    for (int u = cid; u < total && ok && !*abort_flag; u += ncl) {
      const Tile t = decode_tile<256>(args, mt, u, sg);
      const int64_t grow = static_cast<int64_t>(t.row0) + prow;
      const bool rok = prow < t.rows_valid && grow >= 0 && grow < args.rows_total;
      const float *as = fa.a_scale + (rok ? grow : 0) * kbs;
      // gate_up: gate and up blocks (both halves); down: half 0's and half 1's blocks
      const float *bs0, *bs1;
      if (SWIGLU) {
        bs0 = fa.b_scale + (static_cast<int64_t>(t.e) * b_blocks + (t.n * C::BN_OUT) / 128) * kbs;
        bs1 = fa.b_scale +
              (static_cast<int64_t>(t.e) * b_blocks + (args.up_off + t.n * C::BN_OUT) / 128) * kbs;
      } else {
        bs0 = fa.b_scale + (static_cast<int64_t>(t.e) * b_blocks + 2 * t.n) * kbs;
        bs1 = bs0 + kbs;
      }
      float ca[4], c0[4], c1[4];
      auto load4 = [&](int kb0, float(&a)[4], float(&b0)[4], float(&b1)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kb = kb0 + i;
          const bool in = kb < kblocks;
          a[i] = (in && rok) ? __ldg(as + kb) : 1.0f;
          b0[i] = in ? __ldg(bs0 + kb) : 1.0f;
          b1[i] = in ? __ldg(bs1 + kb) : 1.0f;
        }
      };
      load4(0, ca, c0, c1);
      for (int kb0 = 0; kb0 < kblocks && ok; kb0 += 4) {
        float na[4], n0[4], n1[4];
        load4(kb0 + 4, na, n0, n1);
        // byte i of each cell: k-block kb0 + i (past the tile's last k-block: 2^0)
        uint32_t va = 0, v0 = 0, v1 = 0;
        bool valid = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t ba, b0, b1;
          valid = valid & ue8m0_of(ca[i], ba) & ue8m0_of(c0[i], b0) & ue8m0_of(c1[i], b1);
          va |= ba << (8 * i);
          v0 |= b0 << (8 * i);
          v1 |= b1 << (8 * i);
        }
        if (!valid) set_status(args.status, kStatusBadId);
        const bool waited = mbar_wait_bounded(&sempty[slot], sphase ^ 1u, abort_flag,
                                              args.status, args.wait_limit_ns);
        if (!__all_sync(0xffffffffu, waited)) {
          ok = false;
          break;
        }
        // gate_up: each half's B columns 0-63 gate (v0), 64-127 up (v1);
        // down: half 0 all v0, half 1 all v1
        const uint32_t h0a = v0, h0b = SWIGLU ? v1 : v0;
        const uint32_t h1a = SWIGLU ? v0 : v1, h1b = v1;
        const uint32_t v[16] = {va, va, va, va, h0a, h0a, h0b, h0b,
                                h1a, h1a, h1b, h1b, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu,
                                0x7f7f7f7fu};
        tmem_st_32x32b_x16(
            tmem_base + lane_off + static_cast<uint32_t>(kF8PairScaleCol + kF8PairSlotCols * slot),
            v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(mapa_shared(&sfull[slot], 0));
        if (++slot == kF8ScaleSlots) {
          slot = 0;
          sphase ^= 1u;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ca[i] = na[i];
          c0[i] = n0[i];
          c1[i] = n1[i];
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 6..13, both CTAs) ----------------
    // For each half of a tile in turn (the one in the middle slot first,
    // releasing it for the next tile's MMAs): warp w takes TMEM lane
    // quadrant w % 4 and part p = (w - 6) / 4 of the half.  gate_up: gate columns 32p..32p+31 of the
    // half and their up columns 64 + 32p.. -> h columns t.n * 128 + 64 * half
    // + 32p; down: columns 64p..64p+63 -> output columns t.n * 256 +
    // 128 * half + 64p.
    const int quad = warp & 3;
    const int part = (warp - 6) >> 2;
    const int prow = static_cast<int>(rank) * 128 + quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int col0 = SWIGLU ? 32 * part : 64 * part;
    const int col1 = SWIGLU ? 64 + 32 * part : 64 * part + 32;
    uint32_t tcount = 0;
    uint32_t hpar = 0;  // bit b: parity of slot b's next completion
    const bool fuse = SWIGLU && args.out_h_scales != nullptr;
    float *xch = reinterpret_cast<float *>(smem + C::OUT_OFF);
    uint32_t xuse = 0;  // uses of this quadrant's exchange barrier
    bool ok = true;
    for (int u = cid; u < total && ok; u += ncl, ++tcount) {
      const Tile t = decode_tile<256>(args, mt, u, sg);
      const int64_t grow = static_cast<int64_t>(t.row0) + prow;
      const bool rok = prow < t.rows_valid && grow >= 0 && grow < args.rows_total;
      const bool warp_rows = static_cast<int>(rank) * 128 + quad * 32 < t.rows_valid;
      uint32_t hq0[16], hq1[16];  // fused quantization: this thread's h runs of the tile
      for (int it = 0; it < 2; ++it) {
        // even tiles: slots 0, 1 (half 1 in the middle slot); odd: slots 1, 2
        const int half = (tcount & 1u) ? it : 1 - it;
        const uint32_t b = (tcount & 1u) + static_cast<uint32_t>(half);
        const bool waited = mbar_wait_bounded(&hfull[b], (hpar >> b) & 1u, abort_flag,
                                              args.status, args.wait_limit_ns);
        if (!__all_sync(0xffffffffu, waited)) {
          ok = false;
          break;
        }
        hpar ^= 1u << b;
        tc_fence_after();
        uint32_t v[32], w[32];
        if (warp_rows) {
          const uint32_t tp = tmem_base + lane_off + 128u * b;
          tmem_ld_32x32b_x32(tp + col0, v);
          tmem_ld_32x32b_x32(tp + col1, w);
          tmem_ld_wait();
          tmem_regs_fence(v);
          tmem_regs_fence(w);
        }
        // the half is released as soon as its values are in registers
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(mapa_shared(&hempty[b], 0));
        if (!warp_rows) continue;
        if (fuse) {
          if (half == 0)
            f8_swiglu_bf16(v, w, hq0);
          else
            f8_swiglu_bf16(v, w, hq1);
          continue;
        }
        if (!SWIGLU && args.out_tma &&
            static_cast<int>(rank) * 128 + quad * 32 + 32 <= t.rows_valid &&
            grow - lane >= 0 && grow - lane + 32 <= args.rows_total) {
          // compact rows by TMA: per 32-column group the warp's 32 rows of
          // fp16 values as one box, then the lane's two code bytes
          uint8_t *box = smem + C::OUT_OFF + (warp - 6) * C::OUT_BOX_BYTES;
          const int row_g = static_cast<int>(grow - lane);
          const uint32_t swz = static_cast<uint32_t>((lane >> 1) & 3);
          const uint32_t rbase = smem_u32(box) + static_cast<uint32_t>(lane) * 64u;
          const int64_t col = static_cast<int64_t>(t.n) * kF8PairBN + 128 * half + 64 * part;
          uint32_t codes = 0;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t hw[16];
            codes |= y16_encode32(g ? w : v, hw) << (8 * g);
            if (lane == 0) bulk_wait_read_0();  // the previous store has read the box
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(rbase + ((static_cast<uint32_t>(q) ^ swz) * 16u), hw[4 * q],
                           hw[4 * q + 1], hw[4 * q + 2], hw[4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmY, box, static_cast<int32_t>(col + 32 * g), row_g);
              bulk_commit();
            }
          }
          *reinterpret_cast<uint16_t *>(args.out_codes + grow * (args.ldo / 32) + col / 32) =
              static_cast<uint16_t>(codes);
          continue;
        }
        if (!rok) continue;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          acc[i] = __uint_as_float(v[i]);
          acc[32 + i] = __uint_as_float(w[i]);
        }
        f8_store_tile_row<SWIGLU>(
            args, grow,
            SWIGLU ? static_cast<int64_t>(t.n) * C::BN_OUT + 64 * half + 32 * part
                   : static_cast<int64_t>(t.n) * kF8PairBN + 128 * half + 64 * part,
            acc);
      }
      if (fuse && ok && warp_rows &&
          !f8_quantize_row(args, t, grow, rok, quad * 32 + lane, part, xuse++, hq0, hq1, xch,
                           &xbar[quad], abort_flag))
        ok = false;
    }
  }

  if (!SWIGLU && warp >= 6 && lane == 0) bulk_wait_all();  // output stores written
  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while its peer may still use its memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kF8TmemCols);
}

// ---------------------------------------------------------------------------
// The FP8 GEMM's 1-CTA form with 128 x 256 tiles (used where the routed rows
// are few per expert, so the weights are the bound): one M=128 x N=256
// block-scaled MMA per K step, the accumulator windows alternating over
// three 128-column TMEM slots as in the pair form.  A stage holds 128 A rows and
// 256 B rows (48 KB, 4 stages): 32 KB of weights per stage and 128 KB in
// flight.  gate_up: smem B rows 0-63 gate i0.., 64-127 up i0.., 128-191
// gate i0+64.., 192-255 up i0+64.. (i0 = 128 t.n), so each half holds 64 gate
// columns and their up columns; down: rows c0 .. c0+255 (c0 = 256 t.n).
// The exponent slots are the pair form's (16 columns: A in 0-3, B in 4-11,
// B column n's exponent at lane 32q + n % 32, column 4 + n / 32).
// ---------------------------------------------------------------------------
constexpr int kF8WideStages = 4;

template <bool SWIGLU>
struct CfgF8W {
  static constexpr int A_BYTES = kBM * kF8BK;
  static constexpr int B_BYTES = kF8PairBN * kF8BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = kF8WideStages;
  static constexpr int BN_OUT = SWIGLU ? kF8PairBN / 2 : kF8PairBN;
  // gate_up: the row maxima exchanged by the fused h quantization
  static constexpr int XCH_OFF = STAGES * STAGE_BYTES;
  static constexpr int XCH_BYTES = SWIGLU ? 2 * 2 * 128 * 4 : 0;
  static constexpr int BAR_OFF = XCH_OFF + XCH_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * kF8ScaleSlots + 2 * 3 + 1 + 4;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int MT_OFF = MISC_OFF + 16;
  static constexpr int SMEM_BYTES = MT_OFF + (kMaxE + 1) * 4 + 1024;
  static_assert(SMEM_BYTES <= 232448, "227 KB of shared memory per CTA");
  static_assert(kF8PairScaleCol + kF8PairSlotCols * kF8ScaleSlots <= kF8TmemCols,
                "scale slots fit the TMEM allocation");
};

template <bool SWIGLU>
__global__ void __launch_bounds__(kF8Threads, 1)
    grouped_gemm_fp8_wide_kernel(const __grid_constant__ CUtensorMap tmA,
                                 const __grid_constant__ CUtensorMap tmA32,
                                 const __grid_constant__ CUtensorMap tmB, const F8Args fa) {
  pdl_begin();
  using C = CfgF8W<SWIGLU>;
  const KArgs &args = fa.k;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smem + C::STAGES * C::A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::STAGES;
  uint64_t *sfull = bars + 2 * C::STAGES;
  uint64_t *sempty = sfull + kF8ScaleSlots;
  uint64_t *hfull = sempty + kF8ScaleSlots;
  uint64_t *hempty = hfull + 3;
  uint64_t *drain = hempty + 3;
  uint64_t *xbar = drain + 1;  // per lane quadrant: the fused h quantization's exchange
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
  int32_t *mt = reinterpret_cast<int32_t *>(smem + C::MT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) mt[i] = args.mtile_base[i];
  if (threadIdx.x == 0) {
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    for (int g = 0; g < kF8ScaleSlots; ++g) {
      mbar_init(&sfull[g], 4);
      mbar_init(&sempty[g], 1);
    }
    for (int b = 0; b < 3; ++b) {
      mbar_init(&hfull[b], 1);
      mbar_init(&hempty[b], 8);
    }
    mbar_init(drain, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&xbar[q], 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int total = mt[args.E] * args.n_tiles;
  if (blockIdx.x >= total) return;
  if (warp == 1) tmem_alloc(tmem_slot, kF8TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int kblocks = args.K / kF8BK;
  const int kbs = kblocks;
  const int b_blocks = args.b_rows / 128;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA32);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[C::STAGES];
      bool issued[C::STAGES];
#pragma unroll
      for (int st = 0; st < C::STAGES; ++st) issued[st] = false;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        const Tile t = decode_tile(args, mt, u);
        const int subs = (t.rows_valid + kF8SubRows - 1) / kF8SubRows;  // 1..4
        const uint32_t tx = C::B_BYTES + (subs < kBM / kF8SubRows ? subs * kF8SubRows * kF8BK
                                                                  : C::A_BYTES);
        // the four 64-row B boxes of a stage (smem rows 0, 64, 128, 192)
        int b_row[4];
        if (SWIGLU) {
          const int g0 = t.e * args.b_rows + t.n * C::BN_OUT;
          b_row[0] = g0;
          b_row[1] = g0 + args.up_off;
          b_row[2] = g0 + 64;
          b_row[3] = g0 + args.up_off + 64;
        } else {
          const int c0 = t.e * args.b_rows + t.n * kF8PairBN;
#pragma unroll
          for (int q = 0; q < 4; ++q) b_row[q] = c0 + 64 * q;
        }
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status,
                                 args.wait_limit_ns))
            break;
          uint8_t *a_dst = smA + stage * C::A_BYTES;
          uint8_t *b_dst = smB + stage * C::B_BYTES;
          mbar_arrive_expect_tx(&full[stage], tx);
          if (subs < kBM / kF8SubRows) {
            for (int i = 0; i < subs; ++i)
              tma_load_2d(a_dst + i * kF8SubRows * kF8BK, &tmA32, &full[stage], kb * kF8BK,
                          t.row0 + i * kF8SubRows);
          } else {
            tma_load_2d(a_dst, &tmA, &full[stage], kb * kF8BK, t.row0);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            tma_load_2d(b_dst + q * 64 * kF8BK, &tmB, &full[stage], kb * kF8BK, b_row[q]);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int st = 0; st < C::STAGES; ++st)
        if (issued[st]) wait_drain(&full[st], issued_phase[st], args.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t kIdesc = mma_idesc_mxf8_f32(kBM, kF8PairBN);
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t sphase = 0;
      uint32_t tcount = 0;
      uint32_t hpar = 0;  // bit b: parity of slot b's next use
      bool any_mma = false;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok && !*abort_flag; u += gridDim.x, ++tcount) {
        const uint32_t h0 = tcount & 1u, h1 = h0 + 1u;  // the tile's two slots
        if (!mbar_wait_bounded(&hempty[h0], ((hpar >> h0) & 1u) ^ 1u, abort_flag, args.status,
                               args.wait_limit_ns) ||
            !mbar_wait_bounded(&hempty[h1], ((hpar >> h1) & 1u) ^ 1u, abort_flag, args.status,
                               args.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + 128u * h0;
        for (int kb = 0; kb < kblocks; ++kb) {
          const int j = kb & 3;  // byte of the slot's cells with this k-block's exponents
          if ((j == 0 && !mbar_wait_bounded(&sfull[slot], sphase, abort_flag, args.status,
                                            args.wait_limit_ns)) ||
              !mbar_wait_bounded(&full[stage], phase, abort_flag, args.status,
                                 args.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(smA + stage * C::A_BYTES));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(smB + stage * C::B_BYTES));
          const uint32_t sfa =
              tmem_base + static_cast<uint32_t>(kF8PairScaleCol + kF8PairSlotCols * slot);
          const uint32_t idesc =
              kIdesc | (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
#pragma unroll
          for (int kk = 0; kk < kF8BK / 32; ++kk) {
            mma_mxf8_ss(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, sfa, sfa + 4u,
                        (kb != 0 || kk != 0) ? 1u : 0u);
          }
          any_mma = true;
          mma_commit(&empty[stage]);
          if (j == 3 || kb == kblocks - 1) {
            mma_commit(&sempty[slot]);
            if (++slot == kF8ScaleSlots) {
              slot = 0;
              sphase ^= 1u;
            }
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&hfull[h0]);
        mma_commit(&hfull[h1]);
        hpar ^= (1u << h0) | (1u << h1);
      }
      if (any_mma) {
        mma_commit(drain);
        wait_drain(drain, 0, args.wait_limit_ns);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------- scale writers (warps 2..5) ----------------
    // Per four k-blocks, lanes 32q..32q+31 of a slot: the rows' A exponents
    // (columns 0-3) and both halves' B exponents (4-7, 8-11; gate_up: two
    // gate, two up columns each, down: one block per half).
    const int quad = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int row = quad * 32 + lane;
    int slot = 0;
    uint32_t sphase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok && !*abort_flag; u += gridDim.x) {
      const Tile t = decode_tile(args, mt, u);
      const int64_t grow = static_cast<int64_t>(t.row0) + row;
      const bool rok = row < t.rows_valid && grow >= 0 && grow < args.rows_total;
      const float *as = fa.a_scale + (rok ? grow : 0) * kbs;
      const float *bs0, *bs1;
      if (SWIGLU) {
        bs0 = fa.b_scale + (static_cast<int64_t>(t.e) * b_blocks + (t.n * C::BN_OUT) / 128) * kbs;
        bs1 = fa.b_scale +
              (static_cast<int64_t>(t.e) * b_blocks + (args.up_off + t.n * C::BN_OUT) / 128) * kbs;
      } else {
        bs0 = fa.b_scale + (static_cast<int64_t>(t.e) * b_blocks + 2 * t.n) * kbs;
        bs1 = bs0 + kbs;
      }
      float ca[4], c0[4], c1[4];
      auto load4 = [&](int kb0, float(&a)[4], float(&b0)[4], float(&b1)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kb = kb0 + i;
          const bool in = kb < kblocks;
          a[i] = (in && rok) ? __ldg(as + kb) : 1.0f;
          b0[i] = in ? __ldg(bs0 + kb) : 1.0f;
          b1[i] = in ? __ldg(bs1 + kb) : 1.0f;
        }
      };
      load4(0, ca, c0, c1);
      for (int kb0 = 0; kb0 < kblocks && ok; kb0 += 4) {
        float na[4], n0[4], n1[4];
        load4(kb0 + 4, na, n0, n1);
        uint32_t va = 0, v0 = 0, v1 = 0;
        bool valid = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t ba, b0, b1;
          valid = valid & ue8m0_of(ca[i], ba) & ue8m0_of(c0[i], b0) & ue8m0_of(c1[i], b1);
          va |= ba << (8 * i);
          v0 |= b0 << (8 * i);
          v1 |= b1 << (8 * i);
        }
        if (!valid) set_status(args.status, kStatusBadId);
        const bool waited = mbar_wait_bounded(&sempty[slot], sphase ^ 1u, abort_flag,
                                              args.status, args.wait_limit_ns);
        if (!__all_sync(0xffffffffu, waited)) {
          ok = false;
          break;
        }
        const uint32_t h0a = v0, h0b = SWIGLU ? v1 : v0;
        const uint32_t h1a = SWIGLU ? v0 : v1, h1b = v1;
        const uint32_t v[16] = {va, va, va, va, h0a, h0a, h0b, h0b,
                                h1a, h1a, h1b, h1b, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu,
                                0x7f7f7f7fu};
        tmem_st_32x32b_x16(
            tmem_base + lane_off + static_cast<uint32_t>(kF8PairScaleCol + kF8PairSlotCols * slot),
            v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[slot]);
        if (++slot == kF8ScaleSlots) {
          slot = 0;
          sphase ^= 1u;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ca[i] = na[i];
          c0[i] = n0[i];
          c1[i] = n1[i];
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 6..13) ----------------
    // As in the pair form: each half in turn (the one in the middle slot
    // first), warp w taking lane quadrant w % 4 and part p = (w - 6) / 4 of
    // the half.
    const int quad = warp & 3;
    const int part = (warp - 6) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int col0 = SWIGLU ? 32 * part : 64 * part;
    const int col1 = SWIGLU ? 64 + 32 * part : 64 * part + 32;
    uint32_t tcount = 0;
    uint32_t hpar = 0;
    const bool fuse = SWIGLU && args.out_h_scales != nullptr;
    float *xch = reinterpret_cast<float *>(smem + C::XCH_OFF);
    uint32_t xuse = 0;  // uses of this quadrant's exchange barrier
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++tcount) {
      const Tile t = decode_tile(args, mt, u);
      const int64_t grow = static_cast<int64_t>(t.row0) + row;
      const bool rok = row < t.rows_valid && grow >= 0 && grow < args.rows_total;
      const bool warp_rows = quad * 32 < t.rows_valid;
      uint32_t hq0[16], hq1[16];  // fused quantization: this thread's h runs of the tile
      for (int it = 0; it < 2; ++it) {
        // even tiles: slots 0, 1 (half 1 in the middle slot); odd: slots 1, 2
        const int half = (tcount & 1u) ? it : 1 - it;
        const uint32_t b = (tcount & 1u) + static_cast<uint32_t>(half);
        const bool waited = mbar_wait_bounded(&hfull[b], (hpar >> b) & 1u, abort_flag,
                                              args.status, args.wait_limit_ns);
        if (!__all_sync(0xffffffffu, waited)) {
          ok = false;
          break;
        }
        hpar ^= 1u << b;
        tc_fence_after();
        uint32_t v[32], w[32];
        if (warp_rows) {
          const uint32_t tp = tmem_base + lane_off + 128u * b;
          tmem_ld_32x32b_x32(tp + col0, v);
          tmem_ld_32x32b_x32(tp + col1, w);
          tmem_ld_wait();
          tmem_regs_fence(v);
          tmem_regs_fence(w);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&hempty[b]);
        if (warp_rows && fuse) {
          if (half == 0)
            f8_swiglu_bf16(v, w, hq0);
          else
            f8_swiglu_bf16(v, w, hq1);
          continue;
        }
        if (!warp_rows || !rok) continue;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          acc[i] = __uint_as_float(v[i]);
          acc[32 + i] = __uint_as_float(w[i]);
        }
        f8_store_tile_row<SWIGLU>(
            args, grow,
            SWIGLU ? static_cast<int64_t>(t.n) * C::BN_OUT + 64 * half + 32 * part
                   : static_cast<int64_t>(t.n) * kF8PairBN + 128 * half + 64 * part,
            acc);
      }
      if (fuse && ok && warp_rows &&
          !f8_quantize_row(args, t, grow, rok, quad * 32 + lane, part, xuse++, hq0, hq1, xch,
                           &xbar[quad], abort_flag))
        ok = false;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kF8TmemCols);
}

// ---------------------------------------------------------------------------
// bounded-wait self test: one thread waits on a barrier nobody arrives on
// ---------------------------------------------------------------------------
__global__ void wait_selftest_kernel(uint32_t *status, uint64_t limit_ns) {
  pdl_begin();
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, &abort_flag, status, limit_ns);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Gate/up weights [E * 2 inter, K] seen as 4-D (k, row in group of 16,
// gate|up, group of 16 rows), box 64 x 16 x 2 x 4: one box holds 4 x [16 gate
// rows, the 16 up rows up_off further] of K columns [k, k + 64).  The group
// extent stops up_off rows short, so every element the map can address lies
// inside the weight tensor.
bool make_tmap_gate_up_groups(CUtensorMap *map, const void *base, uint64_t K, uint64_t rows,
                              uint64_t up_off) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= up_off || (rows - up_off) % 16 != 0) return false;
  const cuuint64_t dims[4] = {K, 16, 2, (rows - up_off) / 16};
  const cuuint64_t strides[3] = {K * 2, up_off * K * 2, 16 * K * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(kBK), 16, 2, 4};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D bf16 tensor [rows, inner] row-major; box = box_rows x 64 elements,
// 128-byte swizzle, out-of-bounds rows read as zero.
bool make_tmap(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
               uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp32 tensor [rows, inner] row-major for TMA stores; box = 32 rows x 16
// elements (64 bytes), 64-byte swizzle.  False if the base is not 16-byte
// aligned or a row is not a multiple of 16 bytes.
bool make_tmap_f32_out(CUtensorMap *map, void *base, uint64_t inner, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15u) != 0 || inner % 4 != 0 || rows == 0)
    return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {16, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp16 tensor [rows, inner] row-major for TMA stores of the compact
// output; box = 32 rows x 32 elements (64 bytes), 64-byte swizzle.  False if
// the base is not 16-byte aligned or a row is not a multiple of 16 bytes.
bool make_tmap_f16_out(CUtensorMap *map, void *base, uint64_t inner, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15u) != 0 || inner % 8 != 0 || rows == 0)
    return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D e4m3 (byte) tensor [rows, inner]; box = box_rows x 128 bytes, 128-byte
// swizzle, out-of-bounds rows read as zero.
bool make_tmap_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                  uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kF8BK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool SWIGLU>
cudaError_t run_gemm_fp8(const GemmProblem &p, const float *a_scale, const float *b_scale,
                         int up_off, cudaStream_t s) {
  using C = CfgF8<SWIGLU>;
  CUtensorMap tmA, tmA32, tmB;
  if (!make_tmap_u8(&tmA, p.a, static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.rows_total),
                    kBM) ||
      !make_tmap_u8(&tmA32, p.a, static_cast<uint64_t>(p.K),
                    static_cast<uint64_t>(p.rows_total), kF8SubRows))
    return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tmB, p.b, static_cast<uint64_t>(p.K),
                    static_cast<uint64_t>(p.E) * static_cast<uint64_t>(p.b_rows), kF8BN / 2))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_fp8_kernel<SWIGLU>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  F8Args fa = {};
  KArgs &a = fa.k;
  a.E = p.E;
  a.K = p.K;
  a.n_tiles = p.n_out / C::BN_OUT;
  a.layout = p.layout;
  a.M_max = p.M_max;
  a.b_rows = p.b_rows;
  a.up_off = up_off;
  a.seg = p.seg;
  a.seg2 = p.seg2;
  a.mtile_base = p.mtile_base;
  a.out = p.out;
  a.ldo = p.n_out;
  a.rows_total = p.rows_total;
  a.out_v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
  if (SWIGLU && p.out_h_scales != nullptr) {
    // h quantized in the epilogue: 32-byte stores of e4m3 codes
    if (!a.out_v8 || p.n_out % 128 != 0) return cudaErrorInvalidValue;
    a.out_h_scales = p.out_h_scales;
  }
  if (!SWIGLU && p.out_codes != nullptr) {
    // compact output: 32-byte stores of fp16 values, 2-byte code stores
    if (!a.out_v8 || p.n_out % kF8BN != 0 || (reinterpret_cast<uintptr_t>(p.out_codes) & 1u))
      return cudaErrorInvalidValue;
    a.out_codes = p.out_codes;
  }
  // A rows of one block: about 24 MB (a 128-row tile holds 128*K bytes)
  a.m_block = static_cast<int>((24ll << 20) / (128ll * p.K));
  if (a.m_block < 1) a.m_block = 1;
  a.status = p.status;
  a.wait_limit_ns = p.wait_limit_ns ? p.wait_limit_ns : kDefaultWaitLimitNs;
  a.ksplit = 1;
  fa.a_scale = a_scale;
  fa.b_scale = b_scale;
  if (!p.pair && p.n_out % CfgF8W<SWIGLU>::BN_OUT == 0) {
    // 1-CTA form with 256-column tiles (128-row m-tiles, as mtile_base counts)
    using W = CfgF8W<SWIGLU>;
    err = cudaFuncSetAttribute(grouped_gemm_fp8_wide_kernel<SWIGLU>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, W::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    a.n_tiles = p.n_out / W::BN_OUT;
    MOE_LAUNCH_PDL(grouped_gemm_fp8_wide_kernel<SWIGLU>, num_sms(), kF8Threads, W::SMEM_BYTES, s,
                   tmA, tmA32, tmB, fa);
    return cudaGetLastError();
  }
  if (!p.pair) {
    if (a.out_h_scales != nullptr) return cudaErrorInvalidValue;  // 128-column tiles: bf16 h only
    MOE_LAUNCH_PDL(grouped_gemm_fp8_kernel<SWIGLU>, num_sms(), kF8Threads, C::SMEM_BYTES, s, tmA,
                   tmA32, tmB, fa);
    return cudaGetLastError();
  }
  // CTA pairs on 256-row tiles (mtile_base counts 256-row tiles)
  using P = CfgF8P<SWIGLU>;
  // down, compact rows: fp16 values leave through TMA stores
  CUtensorMap tmY = tmA;
  a.out_tma = 0;
  if (!SWIGLU && a.out_codes != nullptr &&
      make_tmap_f16_out(&tmY, p.out, static_cast<uint64_t>(p.n_out),
                        static_cast<uint64_t>(p.rows_total)))
    a.out_tma = 1;
  err = cudaFuncSetAttribute(grouped_gemm_fp8_pair_kernel<SWIGLU>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  if (p.n_out % P::BN_OUT != 0) return cudaErrorInvalidValue;
  a.n_tiles = p.n_out / P::BN_OUT;
  a.m_block = static_cast<int>((24ll << 20) / (256ll * p.K));
  if (a.m_block < 1) a.m_block = 1;
  int clusters = 0;
  {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.blockDim = dim3(kF8Threads);
    cfg.dynamicSmemBytes = P::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_fp8_pair_kernel<SWIGLU>, &cfg);
    if (err != cudaSuccess) return err;
  }
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  MOE_LAUNCH_PDL(grouped_gemm_fp8_pair_kernel<SWIGLU>, 2 * clusters, kF8Threads, P::SMEM_BYTES, s,
                 tmA, tmA32, tmB, tmY, fa);
  return cudaGetLastError();
}

template <int BN, bool SWIGLU>
cudaError_t run_gemm(const GemmProblem &p, int up_off, cudaStream_t s) {
  using C = Cfg<BN, SWIGLU>;
  CUtensorMap tmA, tmB;
  if (!make_tmap(&tmA, p.a, static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.rows_total),
                 kBM))
    return cudaErrorInvalidValue;
  if (!make_tmap(&tmB, p.b, static_cast<uint64_t>(p.K),
                 static_cast<uint64_t>(p.E) * static_cast<uint64_t>(p.b_rows), C::HALF))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<BN, SWIGLU>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  KArgs a = {};
  a.E = p.E;
  a.K = p.K;
  a.n_tiles = p.n_out / C::BN_OUT;
  a.layout = p.layout;
  a.M_max = p.M_max;
  a.b_rows = p.b_rows;
  a.up_off = up_off;
  a.seg = p.seg;
  a.seg2 = p.seg2;
  a.mtile_base = p.mtile_base;
  a.out = p.out;
  a.ldo = p.n_out;
  a.rows_total = p.rows_total;
  a.out_v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
  // A rows of one block: about 24 MB (a 128-row tile holds 256*K bytes)
  a.m_block = static_cast<int>((24ll << 20) / (256ll * p.K));
  if (a.m_block < 1) a.m_block = 1;
  a.status = p.status;
  a.wait_limit_ns = p.wait_limit_ns ? p.wait_limit_ns : kDefaultWaitLimitNs;
  a.ksplit = (!SWIGLU && p.ksplit > 1) ? p.ksplit : 1;
  if (!SWIGLU && p.out_codes != nullptr) {
    // compact output: whole 256-column tiles, no K pieces, 32-byte stores
    if (BN != 256 || a.ksplit != 1 || p.n_out % 256 != 0 ||
        (reinterpret_cast<uintptr_t>(p.out) & 31u) != 0 ||
        (reinterpret_cast<uintptr_t>(p.out_codes) & 7u) != 0)
      return cudaErrorInvalidValue;
    a.out_codes = p.out_codes;
  }
  MOE_LAUNCH_PDL(grouped_gemm_kernel<BN, SWIGLU>, num_sms(), kGemmThreads, C::SMEM_BYTES, s, tmA, tmB, a);
  return cudaGetLastError();
}

template <int BN, bool SWIGLU>
cudaError_t run_gemm_pair(const GemmProblem &p, int up_off, cudaStream_t s) {
  using C = Cfg2<BN, SWIGLU>;
  CUtensorMap tmA, tmB, tmW, tmY;
  SwapXMaps tmX;
  const uint64_t w_rows = static_cast<uint64_t>(p.E) * static_cast<uint64_t>(p.b_rows);
  if (!make_tmap(&tmA, p.a, static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.rows_total),
                 128))
    return cudaErrorInvalidValue;
  if (!make_tmap(&tmB, p.b, static_cast<uint64_t>(p.K), w_rows, C::HALF))
    return cudaErrorInvalidValue;
  for (int i = 0; i < 4; ++i)
    if (!make_tmap(&tmX.m[i], p.a, static_cast<uint64_t>(p.K),
                   static_cast<uint64_t>(p.rows_total), 8u << i))
      return cudaErrorInvalidValue;
  if (SWIGLU) {
    if (!make_tmap_gate_up_groups(&tmW, p.b, static_cast<uint64_t>(p.K), w_rows,
                                  static_cast<uint64_t>(up_off)))
      return cudaErrorInvalidValue;
  } else {
    tmW = tmB;
  }
  // down: output (fp32, or the compact fp16 values) stored by TMA where its
  // layout allows (else plain stores)
  const bool out_f16 = !SWIGLU && p.out_codes != nullptr;
  if (out_f16 && (p.n_out % 256 != 0 || (reinterpret_cast<uintptr_t>(p.out) & 31u) != 0 ||
                  (reinterpret_cast<uintptr_t>(p.out_codes) & 7u) != 0))
    return cudaErrorInvalidValue;
  const bool out_tma =
      !SWIGLU && (out_f16 ? make_tmap_f16_out(&tmY, p.out, static_cast<uint64_t>(p.n_out),
                                              static_cast<uint64_t>(p.rows_total))
                          : make_tmap_f32_out(&tmY, p.out, static_cast<uint64_t>(p.n_out),
                                              static_cast<uint64_t>(p.rows_total)));
  if (!out_tma) tmY = tmA;
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_pair_kernel<BN, SWIGLU>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  KArgs a = {};
  a.E = p.E;
  a.K = p.K;
  a.n_tiles = p.n_out / C::BN_OUT;
  a.layout = p.layout;
  a.M_max = p.M_max;
  a.b_rows = p.b_rows;
  a.up_off = up_off;
  a.seg = p.seg;
  a.seg2 = p.seg2;
  a.mtile_base = p.mtile_base;
  a.out = p.out;
  a.ldo = p.n_out;
  a.rows_total = p.rows_total;
  a.out_tma = out_tma ? 1 : 0;
  a.out_codes = out_f16 ? p.out_codes : nullptr;
  a.split_part = out_f16 ? p.split_part : nullptr;
  a.split_part_slots = (out_f16 && p.split_part != nullptr) ? p.split_part_slots : 0;
  a.split_flags = SWIGLU ? nullptr : p.split_flags;
  {
    // a different value per launch, so that a flag left raised by an aborted
    // launch, or never cleared, is not taken for this launch's
    static std::atomic<uint32_t> epoch{0};
    uint32_t e = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    if (e == 0) e = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    a.split_epoch = e;
  }
  a.out_v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
  a.m_block = static_cast<int>((24ll << 20) / (512ll * p.K));
  if (a.m_block < 1) a.m_block = 1;
  a.status = p.status;
  a.wait_limit_ns = p.wait_limit_ns ? p.wait_limit_ns : kDefaultWaitLimitNs;
  a.ksplit = 1;
  // persistent grid: as many CTA pairs as can be resident at once
  int clusters = 0;
  {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_pair_kernel<BN, SWIGLU>, &cfg);
    if (err != cudaSuccess) return err;
  }
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  MOE_LAUNCH_PDL(grouped_gemm_pair_kernel<BN, SWIGLU>, 2 * clusters, kGemmThreads, C::SMEM_BYTES, s, 
      tmA, tmB, tmX, tmW, tmY, a);
  return cudaGetLastError();
}

}  // namespace

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  static int cache[64] = {0};
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cache[dev] = n;
  return n;
}

cudaError_t launch_gemm_gate_up_swiglu(const GemmProblem &p, cudaStream_t s) {
  // p.n_out = inter, p.b_rows = 2*inter, K = d
  if (p.pair) {
    if (p.n_out % 128 == 0) return run_gemm_pair<256, true>(p, p.n_out, s);
    return cudaErrorInvalidValue;
  }
  if (p.n_out % 128 == 0) return run_gemm<256, true>(p, p.n_out, s);
  if (p.n_out % 64 == 0) return run_gemm<128, true>(p, p.n_out, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_down(const GemmProblem &p, cudaStream_t s) {
  // p.n_out = d, p.b_rows = d, K = inter
  if (p.pair) {
    if (p.n_out % 256 == 0) return run_gemm_pair<256, false>(p, 0, s);
    return cudaErrorInvalidValue;
  }
  if (p.bn != 0) {
    if (p.n_out % p.bn != 0) return cudaErrorInvalidValue;
    if (p.bn == 256) return run_gemm<256, false>(p, 0, s);
    if (p.bn == 128) return run_gemm<128, false>(p, 0, s);
    if (p.bn == 64) return run_gemm<64, false>(p, 0, s);
    return cudaErrorInvalidValue;
  }
  if (p.n_out % 256 == 0) return run_gemm<256, false>(p, 0, s);
  if (p.n_out % 128 == 0) return run_gemm<128, false>(p, 0, s);
  if (p.n_out % 64 == 0) return run_gemm<64, false>(p, 0, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_fp8_gate_up_swiglu(const GemmProblem &p, const float *a_scale,
                                           const float *b_scale, cudaStream_t s) {
  // p.n_out = inter, p.b_rows = 2*inter, K = d; inter and d multiples of 128
  if (p.n_out % 128 != 0 || p.K % kF8BK != 0) return cudaErrorInvalidValue;
  return run_gemm_fp8<true>(p, a_scale, b_scale, p.n_out, s);
}

cudaError_t launch_gemm_fp8_down(const GemmProblem &p, const float *a_scale,
                                 const float *b_scale, cudaStream_t s) {
  // p.n_out = d, p.b_rows = d, K = inter
  if (p.n_out % kF8BN != 0 || p.K % kF8BK != 0) return cudaErrorInvalidValue;
  return run_gemm_fp8<false>(p, a_scale, b_scale, 0, s);
}

cudaError_t launch_wait_selftest(uint32_t *status, uint64_t limit_ns, cudaStream_t s) {
  MOE_LAUNCH_PDL(wait_selftest_kernel, 1, 32, 0, s, status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe

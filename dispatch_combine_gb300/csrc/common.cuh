// common.cuh -- device helpers shared by the MoE kernels (sm_103a only).
//
// Inline PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and tcgen05
// (TMEM allocation, MMA, commit, loads), the bounded wait used by every
// device-side spin, and the device status word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a only"
#endif

namespace moe {

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization (launch_pdl) and starts with
// pdl_begin(): it waits until the previous kernel of the stream has
// completed and its writes are visible, then lets the next kernel launch.
// So a kernel's launch and set-up overlap its predecessor's tail, and, since
// every kernel waits, completion stays ordered along the whole stream.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// kernel, grid, block, dynamic shared bytes, stream, arguments: launches with
// launch_pdl and returns its error from the enclosing function
#define MOE_LAUNCH_PDL(...)                                  \
  do {                                                       \
    const cudaError_t moe_launch_err_ = ::moe::launch_pdl(__VA_ARGS__); \
    if (moe_launch_err_ != cudaSuccess) return moe_launch_err_; \
  } while (0)

// ---------------------------------------------------------------------------
// status word (first 4 bytes of the workspace)
// ---------------------------------------------------------------------------

// One bit per device-detectable error.
enum : uint32_t {
  kStatusBadId = 1u << MOE_ERR_INVALID_ARG,
  kStatusTimeout = 1u << MOE_ERR_TIMEOUT,
  kStatusOverflow = 1u << MOE_ERR_OVERFLOW,
};

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// Default bound of every device-side wait (nanoseconds of %globaltimer).
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// small bf16 helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16lo(uint32_t packed) {
  return __uint_as_float(packed << 16);
}
__device__ __forceinline__ float bf16hi(uint32_t packed) {
  return __uint_as_float(packed & 0xFFFF0000u);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// ---------------------------------------------------------------------------
// The layer's compact form of the down GEMM's output rows (y16): each group
// of 32 consecutive columns of a row is stored as 32 fp16 values
// q_i = rn(y_i * 2^(14 - E)) and one code byte c = E + 127, E the binary
// exponent of the group's largest |y_i|; y_i = q_i * 2^(c - 141).  The
// scaling is exact, |q_i| < 2^15, and the rounding error is at most 2^-11
// of the group's largest magnitude.  A group whose largest |y_i| is below
// 2^-111 (c < 16) is stored as zero (c = 0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t y16_code(float group_max_abs) {
  const uint32_t c = (__float_as_uint(group_max_abs) >> 23) & 0xffu;
  return c < 16u ? 0u : c;
}
// 2^(141 - c): the scale applied before rounding to fp16
__device__ __forceinline__ float y16_enc_mul(uint32_t c) {
  return c ? __uint_as_float((268u - c) << 23) : 0.0f;
}
// 2^(c - 141): the scale back
__device__ __forceinline__ float y16_dec_mul(uint32_t c) {
  return c ? __uint_as_float((c - 14u) << 23) : 0.0f;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// One group of 32 fp32 values (bit patterns v) to its code (returned) and
// its 16 packed fp16 pairs h (value 2q in the low half of h[q]): the largest
// magnitude by three-input max, the scaling by packed multiplies (exact:
// a power of two).
__device__ __forceinline__ uint32_t y16_encode32(const uint32_t (&v)[32], uint32_t (&h)[16]) {
  float m = 0.0f;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const float a = fabsf(__uint_as_float(v[2 * q])), b = fabsf(__uint_as_float(v[2 * q + 1]));
    asm("max.f32 %0, %0, %1, %2;" : "+f"(m) : "f"(a), "f"(b));
  }
  const uint32_t cc = y16_code(m);
  const float mul = y16_enc_mul(cc);
  uint64_t mm;
  asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(mul));
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    uint64_t pr;
    asm("mov.b64 %0, {%1, %2};" : "=l"(pr) : "r"(v[2 * q]), "r"(v[2 * q + 1]));
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(pr) : "l"(mm));
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(pr));
    h[q] = pack_f16x2(lo, hi);
  }
  return cc;
}

// four fp32 adds to global memory (no return value)
__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void red_add_f32(float *p, float a) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}
// 32-byte global stores (one whole sector per lane); p must be 32-byte aligned
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// ---------------------------------------------------------------------------
// shared-memory addresses
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Gives up when *abort is
// set by another role or when limit_ns elapse; in the latter case it sets
// *abort and records MOE_ERR_TIMEOUT.  Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort, uint32_t *status,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if ((it & 63u) == 63u) {
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        set_status(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// flags in global memory between CTAs of one grid
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Bounded wait until *flag == value (acquire).  Gives up when *abort is set
// or limit_ns elapse; in the latter case it sets *abort and records
// MOE_ERR_TIMEOUT.  Returns true when the flag was seen at value.
__device__ __forceinline__ bool flag_wait_bounded(const uint32_t *flag, uint32_t value,
                                                  volatile int *abort, uint32_t *status,
                                                  uint64_t limit_ns) {
  if (ld_acquire_gpu(flag) == value) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    __nanosleep(64);
    if (ld_acquire_gpu(flag) == value) return true;
    if (*abort) return false;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      set_status(status, kStatusTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled load of the box at (c0 = innermost element index, c1 = row) into
// shared memory, completing `bytes` on bar.  c0 * elem_size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map,
                                            uint64_t *bar, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// ---------------------------------------------------------------------------
// clusters (CTA pairs)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the same variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// all threads of all CTAs of the cluster
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// arrive on an mbarrier of another CTA of the cluster (shared::cluster address)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// The same arrival without release ordering: for an arrival that only
// reports tensor-memory accesses already completed by tcgen05.wait::st or
// tcgen05.wait::ld (and fenced with tcgen05.fence::before_thread_sync).
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// 2D tiled TMA load into this CTA's shared memory whose completion is
// signalled on an mbarrier that may live in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster_addr, int32_t c0,
                                                 int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1)
      : "memory");
}

// 4-D box, same pair form as tma_load_2d_pair.
__device__ __forceinline__ void tma_load_4d_pair(void *smem_dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster_addr, int32_t c0,
                                                 int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

// 2D tiled TMA store of the box at (c0 = innermost element index, c1 = row)
// from this CTA's shared memory, tracked in the issuing thread's bulk group.
// The shared-memory writes it reads must be fenced to the async proxy first
// (fence_proxy_async_smem by each writing thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *smem_src,
                                             int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// all but the most recent of the issuing thread's committed bulk groups have
// finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// all of the issuing thread's committed bulk groups have finished reading
// shared memory
__device__ __forceinline__ void bulk_wait_read_0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// the issuing thread's committed bulk stores are complete (written to global)
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th generation tensor cores, accumulators in TMEM)
// ---------------------------------------------------------------------------

// Whole warp: allocate ncols TMEM columns, address written to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Whole warp, in each CTA of a pair: allocation for pair (cta_group::2) MMAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Whole warp.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzling: rows of 128 bytes, 8-row atoms 1024 bytes apart.
//   bits  0-13  start address >> 4
//   bits 16-29  leading byte offset >> 4 (unused for swizzled K-major; 1)
//   bits 32-45  stride byte offset >> 4  (1024 B between 8-row groups)
//   bits 46-48  0b001 (descriptor version)
//   bits 61-63  swizzle mode, 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  desc |= static_cast<uint64_t>(1u) << 16;
  desc |= static_cast<uint64_t>(1024u >> 4) << 32;
  desc |= static_cast<uint64_t>(1u) << 46;
  desc |= static_cast<uint64_t>(2u) << 61;
  return desc;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A/B (both
// K-major), fp32 accumulator, M x N tile.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15/16 A/B major (0 = K), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t mma_idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// FP8 (e4m3) block quantization, shared by the quantizers and the FP8
// gate_up epilogue.  A block's scale is the power of two s = 2^e with e the
// smallest integer >= -127 such that amax <= 448 * 2^e (1 for an all-zero
// block, 2^127 for a non-finite amax), taken from amax's bits: amax =
// (1 + f) * 2^(E - 127) with E its exponent field, and 448 * 2^(E - 135) =
// 1.75 * 2^(E - 127), so e = E - 135 when f <= 0.75 (mantissa field <=
// 0x600000), else E - 134.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fp8_block_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  const uint32_t b = __float_as_uint(amax);
  const int ef = static_cast<int>((b >> 23) & 0xffu);
  if (ef == 0xff) return __uint_as_float(254u << 23);  // 2^127
  int e = ef - 135 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0);
  if (e <= -127) return __uint_as_float(0x00400000u);  // 2^-127 (an fp32 subnormal)
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// two fp32 -> two e4m3 codes (lo in bits 0-7), round to nearest even,
// saturating to +-448
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// kind::mxf8f6f4 block-scaled descriptor: A and B e4m3 (format 0 in bits
// 7-9 and 10-12), both K-major, N >> 3 at bit 17, scale type UE8M0 (bit 23),
// M >> 4 at bit 24; scale factor ids 0 (bits 4-5 for B, 29-30 for A): each
// MMA reads byte 0 of its scale cells.
__host__ __device__ constexpr uint32_t mma_idesc_mxf8_f32(int M, int N) {
  return (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= (A[smem] * 2^sa) * (B[smem] * 2^sb)^T with e4m3 operands
// (K = 32 per instruction) and one 8-bit exponent per row of A and per row
// of B, read from TMEM at sfa_tmem / sfb_tmem (UE8M0: 2^(byte - 127)); one
// elected thread.  For M = N = 128: row m's A exponent sits at lane m,
// column m / 32 from sfa_tmem; B row n's at lane 32q + n % 32 of every lane
// quadrant q, column n / 32 from sfb_tmem.
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem,
                                            uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Whole warp: thread i writes v[j] to lane (base lane + i), column col + j.
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one elected thread.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair MMA issued by the even CTA of the pair: D (M=256: rows 0-127 in this
// CTA's TMEM, 128-255 in the peer's) (+)= A (128 rows in each CTA's shared
// memory at the same offset) * B^T (N/2 rows in each CTA).
__device__ __forceinline__ void mma_bf16_ss_pair(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at this shared offset in every CTA of
// cta_mask when the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Arrive once on bar when every previously issued tcgen05.mma of this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Whole warp: 32 lanes x 32 consecutive fp32 columns; thread i gets lane
// (base lane + i), register j = column (col + j).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

// Whole warp: 32 lanes x 16 consecutive fp32 columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_regs_fence16(uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The registers written by tcgen05.ld are only valid after tcgen05.wait::ld;
// this empty asm makes every later use depend on a point after the wait.
__device__ __forceinline__ void tmem_regs_fence(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

}  // namespace moe

// quant.cu -- FP8 (e4m3) quantization with block scales.
//
// The MoE path of "ep-deploy" (its cost model: "the dispatch sends FP8 with
// scales", 7168 + 224 bytes per token) and the FP8 grouped GEMM of
// "推理INFRA方法论-02-parallelism" ("DeepGEMM masked, FP8") use e4m3 values
// with fp32 scales: one per (row, 128 columns) of an activation and one per
// 128 x 128 block of a weight.  Here each scale is a power of two, so that
// the tensor cores can apply it themselves (as an 8-bit exponent): s = 2^e
// with e the smallest integer >= -127 such that amax <= 448 * 2^e (1 for an
// all-zero block, 2^127 when amax is not finite); q = e4m3(x / s) rounded to
// nearest even with saturation at 448.  Dividing by a power of two is exact,
// so the codes are reproducible bit for bit.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// A row's 128-column blocks are consecutive in memory (cols is a multiple
// of 128), so block b of the whole array starts at element 128 b and its
// scale is scales[b].  Half a warp per block, 16 bytes (8 values) per lane,
// kQRowsUnroll block pairs per warp in flight; grid-stride over the blocks.
// Dividing by the power-of-two scale is the exact product with its
// reciprocal, so the codes are those of the division.
constexpr int kQRowsUnroll = 4;

__global__ void __launch_bounds__(256)
    quantize_rows_kernel(const __nv_bfloat16 *__restrict__ x, int64_t blocks,
                         uint8_t *__restrict__ q, float *__restrict__ scales) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;  // lane within the half warp
  const int half = lane >> 4;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t base = warp * 2 * kQRowsUnroll; base < blocks;
       base += nwarps * 2 * kQRowsUnroll) {
    uint4 raw[kQRowsUnroll];
#pragma unroll
    for (int j = 0; j < kQRowsUnroll; ++j) {
      const int64_t b = base + 2 * j + half;
      raw[j] = b < blocks ? *reinterpret_cast<const uint4 *>(x + b * 128 + hl * 8)
                          : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kQRowsUnroll; ++j) {
      const int64_t b = base + 2 * j + half;
      const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
      float v[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        v[2 * t] = bf16lo(w[t]);
        v[2 * t + 1] = bf16hi(w[t]);
      }
      float amax = 0.0f;
#pragma unroll
      for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(v[t]));
#pragma unroll
      for (int off = 8; off; off >>= 1)  // within the half warp
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      if (b >= blocks) continue;
      const float sc = fp8_block_scale(amax);
      const float inv = __frcp_rn(sc);  // exact: sc is a power of two
      uint32_t out[2];
#pragma unroll
      for (int t = 0; t < 2; ++t)
        out[t] = static_cast<uint32_t>(e4m3x2(__fmul_rn(v[4 * t], inv), __fmul_rn(v[4 * t + 1], inv))) |
                 (static_cast<uint32_t>(e4m3x2(__fmul_rn(v[4 * t + 2], inv),
                                               __fmul_rn(v[4 * t + 3], inv)))
                  << 16);
      *reinterpret_cast<uint2 *>(q + b * 128 + hl * 8) = make_uint2(out[0], out[1]);
      if (hl == 0) scales[b] = sc;
    }
  }
}

// One CTA of 256 threads per 128 x 128 block: each thread 64 values.
__global__ void __launch_bounds__(256)
    quantize_blocks_kernel(const __nv_bfloat16 *__restrict__ w, int rows, int cols,
                           uint8_t *__restrict__ q, float *__restrict__ scales) {
  pdl_begin();
  __shared__ float red[8];
  const int rb = rows / 128, cb = cols / 128;
  const int64_t blk = blockIdx.x;
  const int64_t m = blk / (static_cast<int64_t>(rb) * cb);
  const int i = static_cast<int>((blk / cb) % rb), j = static_cast<int>(blk % cb);
  const __nv_bfloat16 *base = w + static_cast<size_t>(m) * rows * cols;
  // thread t: row (t / 2) of the block, columns (t % 2) * 64 .. +63
  const int br = threadIdx.x >> 1, bc = (threadIdx.x & 1) * 64;
  const size_t o = static_cast<size_t>(i * 128 + br) * cols + j * 128 + bc;
  uint4 raw[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) raw[u] = *reinterpret_cast<const uint4 *>(base + o + u * 8);
  float amax = 0.0f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
    for (int t = 0; t < 4; ++t) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(wv[t])), fabsf(bf16hi(wv[t]))));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int t = 1; t < 8; ++t) amax = fmaxf(amax, red[t]);
  const float s = fp8_block_scale(amax);
  uint8_t *qo = q + static_cast<size_t>(m) * rows * cols + o;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
    uint32_t out[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t a = wv[2 * t], b = wv[2 * t + 1];
      out[t] = static_cast<uint32_t>(e4m3x2(__fdiv_rn(bf16lo(a), s), __fdiv_rn(bf16hi(a), s))) |
               (static_cast<uint32_t>(e4m3x2(__fdiv_rn(bf16lo(b), s), __fdiv_rn(bf16hi(b), s)))
                << 16);
    }
    *reinterpret_cast<uint2 *>(qo + u * 8) = make_uint2(out[0], out[1]);
  }
  if (threadIdx.x == 0) scales[blk] = s;
}

}  // namespace

cudaError_t launch_quantize_rows_fp8(const void *x, int64_t rows, int cols, void *q,
                                     float *scales, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t nblk = rows * (cols / 128);
  // 8 warps per CTA, 2 * kQRowsUnroll blocks per warp and pass; at most 8
  // CTAs per SM, the rest by the grid-stride loop
  int64_t ctas = (nblk + 8 * 2 * kQRowsUnroll - 1) / (8 * 2 * kQRowsUnroll);
  const int64_t cap = 8ll * num_sms();
  if (ctas > cap) ctas = cap;
  MOE_LAUNCH_PDL(quantize_rows_kernel, static_cast<unsigned>(ctas), 256, 0, s,
                 static_cast<const __nv_bfloat16 *>(x), nblk, static_cast<uint8_t *>(q), scales);
  return cudaGetLastError();
}

cudaError_t launch_quantize_blocks_fp8(const void *w, int mats, int rows, int cols, void *q,
                                       float *scales, cudaStream_t s) {
  const int64_t blocks = static_cast<int64_t>(mats) * (rows / 128) * (cols / 128);
  if (blocks == 0) return cudaSuccess;
  MOE_LAUNCH_PDL(quantize_blocks_kernel, static_cast<unsigned>(blocks), 256, 0, s, 
      static_cast<const __nv_bfloat16 *>(w), rows, cols, static_cast<uint8_t *>(q), scales);
  return cudaGetLastError();
}

}  // namespace moe

// combine.cu -- weighted combine back to token order.
//
// Token trace page, hop 4 ("dispatch to two experts"): the experts return
// their outputs along the reverse path and the source sums them with the
// routing weights, y = p5 E5(x) + p27 E27(x).  On one GPU:
//   y[t] = sum_{j<k} w[t,j] * y_perm[dest[t*k+j]]   (fp32, j ascending) -> bf16
// The k source rows are read with 16-byte loads.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kCombineVec = 2;  // 16-byte column vectors per thread

// One CTA per (token, kCombineVec * 1024-column segment): every thread keeps
// kCombineVec * k 16-byte loads in flight, so even a few hundred tokens fill
// the GPU.
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float4 *__restrict__ y_perm, int64_t y_rows,
                   const int32_t *__restrict__ dest, const float *__restrict__ w, int T, int k,
                   int d4, int segs, uint2 *__restrict__ y) {
  pdl_begin();
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  const int t = blockIdx.x / segs;
  const int seg = blockIdx.x - t * segs;
  if (threadIdx.x < k) {
    // a row outside [0, y_rows) (a dropped assignment, or a caller-supplied
    // dest that is not a permutation) contributes nothing
    const int r = dest[(size_t)t * k + threadIdx.x];
    const bool in = r >= 0 && static_cast<int64_t>(r) < y_rows;
    s_row[threadIdx.x] = in ? r : 0;
    s_w[threadIdx.x] = in ? w[(size_t)t * k + threadIdx.x] : 0.0f;
  }
  __syncthreads();
  const int v0 = seg * kCombineThreads * kCombineVec + threadIdx.x;
  float4 acc[kCombineVec];
#pragma unroll
  for (int u = 0; u < kCombineVec; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const float wj = s_w[j];
    const float4 *row = y_perm + (size_t)s_row[j] * d4;
    float4 yv[kCombineVec];
#pragma unroll
    for (int u = 0; u < kCombineVec; ++u) {
      const int v = v0 + u * kCombineThreads;
      yv[u] = (v < d4) ? __ldg(row + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kCombineVec; ++u) {
      acc[u].x = fmaf(wj, yv[u].x, acc[u].x);
      acc[u].y = fmaf(wj, yv[u].y, acc[u].y);
      acc[u].z = fmaf(wj, yv[u].z, acc[u].z);
      acc[u].w = fmaf(wj, yv[u].w, acc[u].w);
    }
  }
#pragma unroll
  for (int u = 0; u < kCombineVec; ++u) {
    const int v = v0 + u * kCombineThreads;
    if (v < d4)
      y[(size_t)t * d4 + v] =
          make_uint2(pack_bf16x2(acc[u].x, acc[u].y), pack_bf16x2(acc[u].z, acc[u].w));
  }
}

// The same from the compact rows: 8 fp16 values (16 bytes) per vector, the
// scale of their 32-column group from its code byte; each value is restored
// exactly (q * 2^(c - 141)) before the same fp32 weighted sum.
__global__ void __launch_bounds__(kCombineThreads)
    combine16_kernel(const uint4 *__restrict__ y16, const uint8_t *__restrict__ codes,
                     int64_t y_rows, const int32_t *__restrict__ dest,
                     const float *__restrict__ w, int T, int k, int d8, int segs,
                     uint4 *__restrict__ y) {
  pdl_begin();
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  const int t = blockIdx.x / segs;
  const int seg = blockIdx.x - t * segs;
  if (threadIdx.x < k) {
    const int r = dest[(size_t)t * k + threadIdx.x];
    const bool in = r >= 0 && static_cast<int64_t>(r) < y_rows;
    s_row[threadIdx.x] = in ? r : 0;
    s_w[threadIdx.x] = in ? w[(size_t)t * k + threadIdx.x] : 0.0f;
  }
  __syncthreads();
  const int v0 = seg * kCombineThreads * kCombineVec + threadIdx.x;
  const int cpr = d8 / 4;  // code bytes per row
  float acc[kCombineVec][8];
#pragma unroll
  for (int u = 0; u < kCombineVec; ++u)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[u][e] = 0.0f;
  for (int j = 0; j < k; ++j) {
    const float wj = s_w[j];
    const uint4 *row = y16 + (size_t)s_row[j] * d8;
    const uint8_t *crow = codes + (size_t)s_row[j] * cpr;
    uint4 yv[kCombineVec];
    uint32_t cv[kCombineVec];
#pragma unroll
    for (int u = 0; u < kCombineVec; ++u) {
      const int v = v0 + u * kCombineThreads;
      yv[u] = (v < d8) ? __ldg(row + v) : make_uint4(0, 0, 0, 0);
      cv[u] = (v < d8) ? __ldg(crow + v / 4) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kCombineVec; ++u) {
      const float mul = y16_dec_mul(cv[u]);
      const uint32_t h[4] = {yv[u].x, yv[u].y, yv[u].z, yv[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[q]));
        acc[u][2 * q] = fmaf(wj, f.x * mul, acc[u][2 * q]);
        acc[u][2 * q + 1] = fmaf(wj, f.y * mul, acc[u][2 * q + 1]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kCombineVec; ++u) {
    const int v = v0 + u * kCombineThreads;
    if (v < d8)
      y[(size_t)t * d8 + v] =
          make_uint4(pack_bf16x2(acc[u][0], acc[u][1]), pack_bf16x2(acc[u][2], acc[u][3]),
                     pack_bf16x2(acc[u][4], acc[u][5]), pack_bf16x2(acc[u][6], acc[u][7]));
  }
}

}  // namespace

cudaError_t launch_combine16(const void *y16, const uint8_t *codes, int64_t y_rows,
                             const int32_t *dest, const float *w, int T, int k, int d, void *y,
                             cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (d % 32 != 0) return cudaErrorInvalidValue;
  const int d8 = d / 8;
  const int segs = (d8 + kCombineThreads * kCombineVec - 1) / (kCombineThreads * kCombineVec);
  const int64_t blocks = static_cast<int64_t>(T) * segs;
  MOE_LAUNCH_PDL(combine16_kernel, static_cast<unsigned>(blocks), kCombineThreads, 0, s,
                 static_cast<const uint4 *>(y16), codes, y_rows, dest, w, T, k, d8, segs,
                 static_cast<uint4 *>(y));
  return cudaGetLastError();
}

cudaError_t launch_combine(const float *y_perm, int64_t y_rows, const int32_t *dest,
                           const float *w, int T, int k, int d, void *y, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int d4 = d / 4;
  const int segs = (d4 + kCombineThreads * kCombineVec - 1) / (kCombineThreads * kCombineVec);
  const int64_t blocks = static_cast<int64_t>(T) * segs;
  MOE_LAUNCH_PDL(combine_kernel, static_cast<unsigned>(blocks), kCombineThreads, 0, s, 
      reinterpret_cast<const float4 *>(y_perm), y_rows, dest, w, T, k, d4, segs,
      static_cast<uint2 *>(y));
  return cudaGetLastError();
}

}  // namespace moe

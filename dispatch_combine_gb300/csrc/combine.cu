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

}  // namespace

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

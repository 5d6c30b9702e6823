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

// One CTA per (token, 1024-column segment): every thread keeps k 16-byte
// loads in flight, so even a few hundred tokens fill the GPU.
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float4 *__restrict__ y_perm, const int32_t *__restrict__ dest,
                   const float *__restrict__ w, int T, int k, int d4, int segs,
                   uint2 *__restrict__ y) {
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  const int t = blockIdx.x / segs;
  const int seg = blockIdx.x - t * segs;
  if (threadIdx.x < k) {
    // a row outside [0, T*k) (a caller-supplied dest that is not a
    // permutation) contributes nothing instead of reading out of bounds
    const int r = dest[(size_t)t * k + threadIdx.x];
    const bool in = r >= 0 && static_cast<int64_t>(r) < static_cast<int64_t>(T) * k;
    s_row[threadIdx.x] = in ? r : 0;
    s_w[threadIdx.x] = in ? w[(size_t)t * k + threadIdx.x] : 0.0f;
  }
  __syncthreads();
  const int v = seg * kCombineThreads + threadIdx.x;
  if (v >= d4) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const float wj = s_w[j];
    const float4 yv = __ldg(y_perm + (size_t)s_row[j] * d4 + v);
    acc.x = fmaf(wj, yv.x, acc.x);
    acc.y = fmaf(wj, yv.y, acc.y);
    acc.z = fmaf(wj, yv.z, acc.z);
    acc.w = fmaf(wj, yv.w, acc.w);
  }
  y[(size_t)t * d4 + v] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
}

}  // namespace

cudaError_t launch_combine(const float *y_perm, const int32_t *dest, const float *w, int T,
                           int k, int d, void *y, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int d4 = d / 4;
  const int segs = (d4 + kCombineThreads - 1) / kCombineThreads;
  const int64_t blocks = static_cast<int64_t>(T) * segs;
  combine_kernel<<<static_cast<unsigned>(blocks), kCombineThreads, 0, s>>>(
      reinterpret_cast<const float4 *>(y_perm), dest, w, T, k, d4, segs,
      static_cast<uint2 *>(y));
  return cudaGetLastError();
}

}  // namespace moe

// combine.cu -- weighted combine back to token order.
//
// Token trace page, hop 4 ("dispatch to two experts"): the experts return
// their outputs along the reverse path and the source sums them with the
// routing weights, y = p5 E5(x) + p27 E27(x).  On one GPU:
//   y[t] = sum_{j<k} w[t,j] * y_perm[dest[t*k+j]]   (fp32, j ascending) -> bf16
// One warp per token; each lane walks 4-float vectors of the row, the k
// source rows are read with 16-byte loads.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const float4 *__restrict__ y_perm, const int32_t *__restrict__ dest,
                   const float *__restrict__ w, int T, int k, int d4,
                   uint2 *__restrict__ y) {
  __shared__ int s_row[kCombineWarps][32];
  __shared__ float s_w[kCombineWarps][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = blockIdx.x * kCombineWarps + warp; t < T; t += gridDim.x * kCombineWarps) {
    __syncwarp();
    if (lane < k) {
      // a row outside [0, T*k) (a caller-supplied dest that is not a
      // permutation) contributes nothing instead of reading out of bounds
      const int r = dest[(size_t)t * k + lane];
      const bool in = r >= 0 && static_cast<int64_t>(r) < static_cast<int64_t>(T) * k;
      s_row[warp][lane] = in ? r : 0;
      s_w[warp][lane] = in ? w[(size_t)t * k + lane] : 0.0f;
    }
    __syncwarp();
    for (int v = lane; v < d4; v += 32) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < k; ++j) {
        const float wj = s_w[warp][j];
        const float4 yv = __ldg(y_perm + (size_t)s_row[warp][j] * d4 + v);
        acc.x = fmaf(wj, yv.x, acc.x);
        acc.y = fmaf(wj, yv.y, acc.y);
        acc.z = fmaf(wj, yv.z, acc.z);
        acc.w = fmaf(wj, yv.w, acc.w);
      }
      y[(size_t)t * d4 + v] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  }
}

}  // namespace

cudaError_t launch_combine(const float *y_perm, const int32_t *dest, const float *w, int T,
                           int k, int d, void *y, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int64_t want = (T + kCombineWarps - 1) / kCombineWarps;
  const int64_t cap = (int64_t)num_sms() * 8;
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  combine_kernel<<<blocks, kCombineWarps * 32, 0, s>>>(
      reinterpret_cast<const float4 *>(y_perm), dest, w, T, k, d / 4,
      static_cast<uint2 *>(y));
  return cudaGetLastError();
}

}  // namespace moe

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
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// logits: a CUDA-core GEMM [T,d] x [d,E] whose K dimension is split in 32
// interleaved slices (one per lane), each slice summed in order.
// CTA tile: 16 tokens x 64 experts, 8 warps; warp w owns tokens
// (w & 1) * 8 .. +8 and experts (w >> 1) * 16 .. +16; lane = slice.
// ---------------------------------------------------------------------------
constexpr int kRtTok = 16;
constexpr int kRtExp = 64;
constexpr int kRtThreads = 256;
constexpr int kXsStride = 8 * kRtTok + 4;  // floats per slice in xs (padded)
constexpr int kWsStride = 8 * kRtExp + 4;  // floats per slice in ws (padded)
constexpr int kRtSmemBytes = 32 * (kXsStride + kWsStride) * 4;

__global__ void __launch_bounds__(kRtThreads, 1)
    router_logits_kernel(const __nv_bfloat16 *__restrict__ x,
                         const __nv_bfloat16 *__restrict__ w_r, int T, int d, int E,
                         float *__restrict__ logits) {
  extern __shared__ __align__(16) float rsm[];
  float *xs = rsm;                   // [slice][j][token]
  float *ws = rsm + 32 * kXsStride;  // [slice][j][expert]
  const int t0 = blockIdx.x * kRtTok;
  const int e0 = blockIdx.y * kRtExp;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int tb = (warp & 1) * 8;
  const int eb = (warp >> 1) * 16;
  const bool e_vec = (E % 8) == 0;

  float acc[8][16];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 16; ++b) acc[a][b] = 0.0f;

  const int rounds = (d + 255) / 256;
  for (int r = 0; r < rounds; ++r) {
    __syncthreads();
    // x tile: 16 tokens x 32 chunks of 8 bf16
    for (int q = threadIdx.x; q < kRtTok * 32; q += kRtThreads) {
      const int t = q >> 5, c = q & 31;
      const int i0 = r * 256 + c * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t0 + t < T && i0 < d)
        v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + t) * d + i0));
      float *dst = xs + c * kXsStride + t;
      dst[0 * kRtTok] = bf16lo(v.x);
      dst[1 * kRtTok] = bf16hi(v.x);
      dst[2 * kRtTok] = bf16lo(v.y);
      dst[3 * kRtTok] = bf16hi(v.y);
      dst[4 * kRtTok] = bf16lo(v.z);
      dst[5 * kRtTok] = bf16hi(v.z);
      dst[6 * kRtTok] = bf16lo(v.w);
      dst[7 * kRtTok] = bf16hi(v.w);
    }
    // w tile: 256 rows x 64 experts
    for (int q = threadIdx.x; q < 256 * 8; q += kRtThreads) {
      const int ii = q >> 3, ec = (q & 7) * 8;
      const int i = r * 256 + ii;
      float vals[8];
      if (e_vec && i < d && e0 + ec + 8 <= E) {
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(w_r + (size_t)i * E + e0 + ec));
        vals[0] = bf16lo(v.x); vals[1] = bf16hi(v.x);
        vals[2] = bf16lo(v.y); vals[3] = bf16hi(v.y);
        vals[4] = bf16lo(v.z); vals[5] = bf16hi(v.z);
        vals[6] = bf16lo(v.w); vals[7] = bf16hi(v.w);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          vals[u] = (i < d && e0 + ec + u < E)
                        ? __bfloat162float(w_r[(size_t)i * E + e0 + ec + u])
                        : 0.0f;
      }
      float *dst = ws + (ii >> 3) * kWsStride + (ii & 7) * kRtExp + ec;
      *reinterpret_cast<float4 *>(dst) = make_float4(vals[0], vals[1], vals[2], vals[3]);
      *reinterpret_cast<float4 *>(dst + 4) = make_float4(vals[4], vals[5], vals[6], vals[7]);
    }
    __syncthreads();
    const float *xsl = xs + lane * kXsStride + tb;
    const float *wsl = ws + lane * kWsStride + eb;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float xv[8], wv[16];
      *reinterpret_cast<float4 *>(&xv[0]) = *reinterpret_cast<const float4 *>(xsl + j * kRtTok);
      *reinterpret_cast<float4 *>(&xv[4]) =
          *reinterpret_cast<const float4 *>(xsl + j * kRtTok + 4);
#pragma unroll
      for (int b4 = 0; b4 < 4; ++b4)
        *reinterpret_cast<float4 *>(&wv[b4 * 4]) =
            *reinterpret_cast<const float4 *>(wsl + j * kRtExp + b4 * 4);
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 16; ++b) acc[a][b] = __fmaf_rn(xv[a], wv[b], acc[a][b]);
    }
  }

  // xor butterfly across the 32 slices; every lane ends with the same value
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      float v = acc[a][b];
      v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
      v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
      v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
      v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
      acc[a][b] = v;
    }
  // lane l stores the outputs whose flat index is congruent to l mod 32
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      if (((a * 16 + b) & 31) == lane) {
        const int t = t0 + tb + a, e = e0 + eb + b;
        if (t < T && e < E) logits[(size_t)t * E + e] = acc[a][b];
      }
    }
}

// ---------------------------------------------------------------------------
// exp / sigmoid with a fixed evaluation (Cody & Waite 1980 argument
// reduction; Taylor polynomial of degree 7).
// ---------------------------------------------------------------------------
// ln 2 split: head = fl(ln 2) with its 8 low stored bits cleared (16
// significant bits), tail = fl(ln 2 - head).
__device__ __forceinline__ float canon_exp(float y) {
  const float kLn2Head = 0x1.62e4p-1f;
  const float kLn2Tail = 0x1.7f7d1cp-20f;
  const float kLog2e = 0x1.715476p+0f;
  y = fminf(fmaxf(y, -80.0f), 80.0f);
  const float n = rintf(__fmul_rn(y, kLog2e));
  float r = __fmaf_rn(-n, kLn2Head, y);
  r = __fmaf_rn(-n, kLn2Tail, r);
  // 1/j! rounded to fp32
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0x1p-1f);
  p = __fmaf_rn(p, r, 0x1p+0f);
  p = __fmaf_rn(p, r, 0x1p+0f);
  const int ni = static_cast<int>(n);
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));  // exact: result is normal
}

__device__ __forceinline__ float canon_sigmoid(float l) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, canon_exp(-l)));
}

// (value desc, index asc) arg-max over the warp
__device__ __forceinline__ void warp_argmax(float &v, int &idx) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
    if (ov > v || (ov == v && oi < idx)) {
      v = ov;
      idx = oi;
    }
  }
}

constexpr int kSelWarps = 8;

// One warp per token.  Lane l holds experts l, l+32, ... (E <= 1024).
__global__ void __launch_bounds__(kSelWarps * 32)
    router_select_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T,
                         int E, int G, int topk_group, int k, int score, float bias_scale,
                         int mode, int32_t *__restrict__ ids, float *__restrict__ weights) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
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

}  // namespace

cudaError_t launch_router_logits(const void *x, const void *w_r, int T, int d, int E,
                                 float *logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(router_logits_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kRtSmemBytes);
  if (err != cudaSuccess) return err;
  dim3 grid((T + kRtTok - 1) / kRtTok, (E + kRtExp - 1) / kRtExp);
  router_logits_kernel<<<grid, kRtThreads, kRtSmemBytes, s>>>(
      static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(w_r), T, d, E,
      logits);
  return cudaGetLastError();
}

cudaError_t launch_router_select(const float *logits, const float *bias, int T, int E, int G,
                                 int topk_group, int k, int score, float bias_scale, int mode,
                                 int32_t *ids, float *weights, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = (T + kSelWarps - 1) / kSelWarps;
  router_select_kernel<<<grid, kSelWarps * 32, 0, s>>>(logits, bias, T, E, G, topk_group, k,
                                                       score, bias_scale, mode, ids, weights);
  return cudaGetLastError();
}

}  // namespace moe

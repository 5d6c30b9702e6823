// route_common.cuh -- device arithmetic of the routing decisions shared by
// the fixed-order router (router.cu) and the screened router
// (route_screen.cu): the fixed exp/sigmoid evaluation, the warp arg-max with
// its tie rule, and the fixed-order dot product of one token row with one
// expert's weight row.
//
// "第十五章：多节点大模型推理" section 4.1 (gating) and the "ep-deploy"
// handbook page, section "EPLB 与路由约束" (group-limited top-k) define what
// these serve.  The logit's summation order is fixed: "lane" l of 32 owns the
// 8-element chunks c with c mod 32 == l and sums their exact bf16 x bf16
// products in increasing index from +0; the 32 lane sums are combined by the
// xor butterfly (offsets 16, 8, 4, 2, 1).
#pragma once

#include "common.cuh"

namespace moe {

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

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float f[8]) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// xor butterfly over the warp (offsets 16 .. 1): every lane ends with the
// canonical combination of the 32 lane sums
__device__ __forceinline__ float butterfly_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Fixed-order dot product of a bf16 row pair of nch 8-element chunks (x in
// shared memory): lane l sums chunks l, l+32, ... in increasing order, then
// the xor butterfly.  The weight chunks are loaded eight (then four) ahead;
// the x chunks come from shared memory when they are used.
template <int U>
__device__ __forceinline__ void canon_block(const uint4 *xr, const uint4 *__restrict__ wr, int c,
                                            float &acc) {
  uint4 wv[U];
#pragma unroll
  for (int u = 0; u < U; ++u) wv[u] = __ldg(wr + c + 32 * u);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float xf[8], wf[8];
    bf16x8_to_f32(xr[c + 32 * u], xf);
    bf16x8_to_f32(wv[u], wf);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = __fmaf_rn(xf[i], wf[i], acc);
  }
}
__device__ __forceinline__ float canon_dot(const uint4 *xr, const uint4 *__restrict__ wr,
                                           int nch, int lane) {
  float acc = 0.0f;
  int c = lane;
  for (; c + 32 * 7 < nch; c += 32 * 8) canon_block<8>(xr, wr, c, acc);
  if (c + 32 * 3 < nch) {
    canon_block<4>(xr, wr, c, acc);
    c += 32 * 4;
  }
  for (; c < nch; c += 32) canon_block<1>(xr, wr, c, acc);
  return butterfly_sum(acc);
}

}  // namespace moe

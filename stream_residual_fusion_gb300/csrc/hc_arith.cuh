// hc_arith.cuh -- the float32 arithmetic of hc_post and hc_pre, shared by the fused step and the
// standalone kernels so that both round identically.
//
// Stream weights for the feed-forward, Code: hc_post and hc_pre build every product of a float32
// weight and a stream element as its own float32 tensor and then sum the products over the
// stream index, so each product is rounded to float32 before it is added. The sums run in stream
// order (j = 0, 1, 2, 3, each addition rounded), hc_post adds its sublayer product last, and the
// float32 result is cast to bf16. The paired multiplies and adds are CUDA's __fmul2_rn and
// __fadd2_rn, which behave per lane like __fmul_rn and __fadd_rn: never merged into a fused
// multiply-add.
#pragma once
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace mhc {

__device__ __forceinline__ f2 mul2_rn(f2 a, f2 b) {
  const float2 r = __fmul2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y));
  return f2{r.x, r.y};
}
__device__ __forceinline__ f2 add2_rn(f2 a, f2 b) {
  const float2 r = __fadd2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y));
  return f2{r.x, r.y};
}

// X'_k for a pair of features: bf16(fl(u_k F) + (((fl(C_0k X_0) + fl(C_1k X_1)) + fl(C_2k X_2))
// + fl(C_3k X_3))). cc[j] = C_jk, x[j] = X_j.
__device__ __forceinline__ f2 hc_post_pair(const f2 (&cc)[4], f2 cu, const f2 (&x)[4], f2 f) {
  f2 s = mul2_rn(cc[0], x[0]);
  s = add2_rn(s, mul2_rn(cc[1], x[1]));
  s = add2_rn(s, mul2_rn(cc[2], x[2]));
  s = add2_rn(s, mul2_rn(cc[3], x[3]));
  return add2_rn(mul2_rn(cu, f), s);
}

// y_hat for a pair of features before its bf16 rounding:
// ((fl(p_0 X'_0) + fl(p_1 X'_1)) + fl(p_2 X'_2)) + fl(p_3 X'_3).
__device__ __forceinline__ f2 hc_pre_pair(const f2 (&cp)[4], const f2 (&xp)[4]) {
  f2 s = mul2_rn(cp[0], xp[0]);
  s = add2_rn(s, mul2_rn(cp[1], xp[1]));
  s = add2_rn(s, mul2_rn(cp[2], xp[2]));
  return add2_rn(s, mul2_rn(cp[3], xp[3]));
}

}  // namespace mhc

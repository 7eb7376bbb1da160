// hc_arith.cuh -- the float32 arithmetic of hc_post and hc_pre, shared by the fused step and the
// standalone kernels so that both round identically.
//
// Stream weights for the feed-forward, Code: hc_post and hc_pre build every product of a float32
// weight and a stream element as its own float32 tensor and then sum the products over the
// stream index, so each product is rounded to float32 before it is added. The sums run in stream
// order (j = 0, 1, 2, 3, each addition rounded), hc_post adds its sublayer product last, and the
// float32 result is cast to bf16.
//
// Each product is a paired fused multiply-add with a zero addend that only arrives at run time
// (`nz`, -0.0 passed as a kernel parameter): fma(a, b, -0) is a * b rounded once, exactly the
// rounded product (the sign of a zero product included), and unlike a multiply it cannot be
// merged with the addition that follows. Measured on sm_103a with this toolchain: a paired
// multiply followed by a paired add -- inline PTX mul.rn/add.rn.f32x2, __fmul2_rn/__fadd2_rn, a
// volatile multiply, a product routed through a register move, fma(a, b, -0) with a constant
// -0 -- all came out as one rounding on constructed near ties, even with -fmad=false. Scalar
// __fmul_rn/__fadd_rn round correctly but made the fused step 14% slower; this form costs 3%.
#pragma once
#include "ptx.cuh"

namespace mhc {

// X'_k for a pair of features, before the bf16 rounding:
// fl(u F) + (((fl(C_0k X_0) + fl(C_1k X_1)) + fl(C_2k X_2)) + fl(C_3k X_3)), cc[j] = C_jk,
// x[j] = X_j, nz = {-0, -0} from a kernel parameter.
__device__ __forceinline__ f2 hc_post_pair(const f2 (&cc)[4], f2 cu, const f2 (&x)[4], f2 f, f2 nz) {
  f2 s = fma2(cc[0], x[0], nz);
  s = add2(s, fma2(cc[1], x[1], nz));
  s = add2(s, fma2(cc[2], x[2], nz));
  s = add2(s, fma2(cc[3], x[3], nz));
  return add2(fma2(cu, f, nz), s);
}

// y_hat for a pair of features before its bf16 rounding:
// ((fl(p_0 X'_0) + fl(p_1 X'_1)) + fl(p_2 X'_2)) + fl(p_3 X'_3).
__device__ __forceinline__ f2 hc_pre_pair(const f2 (&cp)[4], const f2 (&xp)[4], f2 nz) {
  f2 s = fma2(cp[0], xp[0], nz);
  s = add2(s, fma2(cp[1], xp[1], nz));
  s = add2(s, fma2(cp[2], xp[2], nz));
  return add2(s, fma2(cp[3], xp[3], nz));
}

}  // namespace mhc

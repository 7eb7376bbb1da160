// mix_math.cuh -- per-token split of the 24 mix numbers and the 4x4 Sinkhorn, in registers.
//
// Stream weights for the feed-forward, "All 5 steps" and Code: hc_split_sinkhorn kernel:
//   p_j  = sigmoid(s_0 m_j + b_j) + eps
//   u_j  = 2 sigmoid(s_1 m_{4+j} + b_{4+j})
//   L_jk = s_2 m_{8+4j+k} + b_{8+4j+k}
//   C    = softmax over k (max subtracted) + eps; columns / (sum + eps);
//          then (iters-1) x [rows / (sum + eps), columns / (sum + eps)].
// split_sinkhorn (standalone kernel): one thread owns one token. The fused kernel uses
// split_sinkhorn_row (four lanes own one token, lane j holding row j of comb; column sums go
// through warp shuffles) or split_sinkhorn_all (every lane of the token holds the whole matrix:
// more arithmetic, no shuffle latency; for launches with few tokens per CTA). Divisions by a row
// or column sum are a reciprocal followed by a multiply (4 reciprocals instead of 16 divisions
// per step).
#pragma once

namespace mhc {

// Hardware reciprocal (rcp.approx: within 1 ulp for normal positive inputs).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ void split_sinkhorn(const float (&m)[24], float s0, float s1, float s2,
                                               const float* __restrict__ base, int iters,
                                               float eps, float (&p)[4], float (&u)[4],
                                               float (&c)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    p[j] = sigmoid_f(fmaf(m[j], s0, __ldg(base + j))) + eps;
    u[j] = 2.0f * sigmoid_f(fmaf(m[4 + j], s1, __ldg(base + 4 + j)));
  }
#pragma unroll
  for (int jk = 0; jk < 16; ++jk) c[jk] = fmaf(m[8 + jk], s2, __ldg(base + 8 + jk));

  // row softmax, then + eps
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float mx = fmaxf(fmaxf(c[4 * j], c[4 * j + 1]), fmaxf(c[4 * j + 2], c[4 * j + 3]));
    float e0 = expf(c[4 * j] - mx), e1 = expf(c[4 * j + 1] - mx);
    float e2 = expf(c[4 * j + 2] - mx), e3 = expf(c[4 * j + 3] - mx);
    float r = __frcp_rn((e0 + e1) + (e2 + e3));
    c[4 * j] = fmaf(e0, r, eps);
    c[4 * j + 1] = fmaf(e1, r, eps);
    c[4 * j + 2] = fmaf(e2, r, eps);
    c[4 * j + 3] = fmaf(e3, r, eps);
  }
  auto col_step = [&]() {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float r = __frcp_rn(((c[k] + c[4 + k]) + (c[8 + k] + c[12 + k])) + eps);
      c[k] *= r;
      c[4 + k] *= r;
      c[8 + k] *= r;
      c[12 + k] *= r;
    }
  };
  auto row_step = [&]() {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float r = __frcp_rn(((c[4 * j] + c[4 * j + 1]) + (c[4 * j + 2] + c[4 * j + 3])) + eps);
      c[4 * j] *= r;
      c[4 * j + 1] *= r;
      c[4 * j + 2] *= r;
      c[4 * j + 3] *= r;
    }
  };
  col_step();
  for (int it = 1; it < iters; ++it) {
    row_step();
    col_step();
  }
}

// Four cooperating lanes (lane j of the aligned group of 4 holds row j). Inputs: this row's
// four logit mix numbers mrow[k] = m[8+4j+k], and m[j], m[4+j]. Outputs: p_j, u_j, comb row j.
// All four lanes must call it together (shuffles over the group).
__device__ __forceinline__ void split_sinkhorn_row(const float (&mrow)[4], float m_p, float m_u,
                                                   int j, float s0, float s1, float s2,
                                                   const float* __restrict__ base, int iters,
                                                   float eps, float& p, float& u, float (&c)[4]) {
  p = sigmoid_f(fmaf(m_p, s0, __ldg(base + j))) + eps;
  u = 2.0f * sigmoid_f(fmaf(m_u, s1, __ldg(base + 4 + j)));
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = fmaf(mrow[k], s2, __ldg(base + 8 + 4 * j + k));
  {
    const float mx = fmaxf(fmaxf(c[0], c[1]), fmaxf(c[2], c[3]));
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] = expf(c[k] - mx);
    const float r = rcp_approx((c[0] + c[1]) + (c[2] + c[3]));
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] = fmaf(c[k], r, eps);
  }
  auto col_step = [&]() {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float t = c[k] + __shfl_xor_sync(0xffffffffu, c[k], 1);
      t += __shfl_xor_sync(0xffffffffu, t, 2);
      c[k] *= rcp_approx(t + eps);
    }
  };
  col_step();
  for (int it = 1; it < iters; ++it) {
    const float r = rcp_approx(((c[0] + c[1]) + (c[2] + c[3])) + eps);
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] *= r;
    col_step();
  }
}

// The same arithmetic as split_sinkhorn_row with one lane holding the whole 4 x 4 matrix (no
// shuffles: each column sum is ((c0 + c1) + (c2 + c3)) over the rows, the value the row
// version's butterfly leaves in every lane), so the two give bitwise the same result. Lanes that
// run it on the same token hold the same result. Inputs: the 24 mix numbers m, the split's
// scales s0..s2 and biases b. Outputs: p, u, comb.
__device__ __forceinline__ void split_sinkhorn_all(const float (&m)[24], float s0, float s1,
                                                   float s2, const float (&b)[24], int iters,
                                                   float eps, float (&p)[4], float (&u)[4],
                                                   float (&c)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    p[j] = sigmoid_f(fmaf(m[j], s0, b[j])) + eps;
    u[j] = 2.0f * sigmoid_f(fmaf(m[4 + j], s1, b[4 + j]));
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float* row = c + 4 * j;
#pragma unroll
    for (int k = 0; k < 4; ++k) row[k] = fmaf(m[8 + 4 * j + k], s2, b[8 + 4 * j + k]);
    const float mx = fmaxf(fmaxf(row[0], row[1]), fmaxf(row[2], row[3]));
#pragma unroll
    for (int k = 0; k < 4; ++k) row[k] = expf(row[k] - mx);
    const float r = rcp_approx((row[0] + row[1]) + (row[2] + row[3]));
#pragma unroll
    for (int k = 0; k < 4; ++k) row[k] = fmaf(row[k], r, eps);
  }
  auto col_step = [&]() {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float r = rcp_approx(((c[k] + c[4 + k]) + (c[8 + k] + c[12 + k])) + eps);
#pragma unroll
      for (int j = 0; j < 4; ++j) c[4 * j + k] *= r;
    }
  };
  col_step();
  for (int it = 1; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float* row = c + 4 * j;
      const float r = rcp_approx(((row[0] + row[1]) + (row[2] + row[3])) + eps);
#pragma unroll
      for (int k = 0; k < 4; ++k) row[k] *= r;
    }
    col_step();
  }
}
// ... with the biases read from global memory.
__device__ __forceinline__ void split_sinkhorn_all(const float (&m)[24], float s0, float s1,
                                                   float s2, const float* __restrict__ base,
                                                   int iters, float eps, float (&p)[4],
                                                   float (&u)[4], float (&c)[16]) {
  float b[24];
#pragma unroll
  for (int e = 0; e < 24; ++e) b[e] = __ldg(base + e);
  split_sinkhorn_all(m, s0, s1, s2, b, iters, eps, p, u, c);
}

}  // namespace mhc

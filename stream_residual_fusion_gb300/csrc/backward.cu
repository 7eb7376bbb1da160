// backward.cu -- gradients of the single-pass mHC step on sm_103a.
//
// The pages define the forward step only (Stream weights for the feed-forward, Code: hc_post,
// hc_mixes, hc_pre, hc_split_sinkhorn; MoE RMSNorm, Code: RMSNorm, Block.forward). The gradients
// here are those of reverse-mode differentiation of that code, with its casts to bf16 passed
// straight through and every derivative taken at the values the forward computed (its bf16 X'
// and y_hat). Per token, with K = 4d, x = flat(X'), r = (|x|^2/K + eps)^(-1/2), m = (W x) r,
// r_y = (|y_hat|^2/d + eps)^(-1/2) and T = sum_i gain_i gy_i y_hat_i:
//   g_m      from (g_p, g_u, g_C) through the split and the Sinkhorn rounds;
//   g_y_hat  = r_y gain gy - (r_y^3 T / d) y_hat;
//   g_X'_k   = gXp_k + p_k g_y_hat + (W^T (r g_m))_k - (r^2/K)(g_m . m) X'_k;
//   gX_j     = sum_k C_jk g_X'_k,  gF = sum_k u_k g_X'_k;
//   gu_k     = g_X'_k . F,  gC_jk = g_X'_k . X_j,  gp_j = g_y_hat . X'_j;
//   gW      += (r g_m) x^T,  ggain += r_y gy y_hat,  and the split's g_base, g_scale.
//
// Five launches on the caller's stream:
//   bwd_mix_kernel     one thread per token: g_m by the split's and Sinkhorn's derivatives (the
//                      Sinkhorn rounds are recomputed from checkpoints), per-block partial sums of
//                      g_base and g_scale.
//   bwd_token_kernel   one warp per token: the token reductions over X' and gy (|x|^2, |y_hat|^2,
//                      T, and gain gy . X'_j, y_hat . X'_j for gp), the per-token scalars and the
//                      two bf16 planes of r g_m that the stream kernel's tensor cores read.
//   bwd_stream_kernel  one CTA per token tile (up to 112 tokens), all columns, in slots of 32: two
//                      TMA rings bring X, F (freed once gX, gF written over them are stored) and
//                      gXp, gy (freed once read); one thread issues tcgen05.mma for W^T (r g_m) into TMEM
//                      (A = the tile's planes of r g_m, B = the slot's planes of W^T, fp32
//                      accumulate); 8 consumer warps recompute X' and y_hat exactly as the forward
//                      does, form g_X', write gX and gF in place of X and F, and accumulate gu and
//                      gC; a second lane of the producer warp stores gX and gF with TMA.
//   bwd_weight_kernel  per (64-column block, token range): gW partial sums on the tensor cores
//                      (X'^T against the planes of r g_m, both token-major), ggain beside them.
//   bwd_reduce_kernel  sums the partials into gW, ggain, g_base, g_scale (fixed order).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "hc_arith.cuh"
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int MIXN = 24;
constexpr uint64_t BWD_WAIT_NS = 2000000000ull;   // 2 s

// ---------------------------------------------------------------------------------------------
// bwd_mix_kernel

constexpr int MIX_THREADS = 64;
constexpr int CK_EVERY = 8;         // least Sinkhorn checkpoint spacing (steps)
constexpr int CK_MAX = 6;           // checkpoints held per token (shared memory)

// Reciprocal of a positive normal float within 1 ulp (the hardware approximation).
__device__ __forceinline__ float rcp_fast(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// One Sinkhorn normalisation of c in place: step i even divides columns, odd divides rows.
__device__ __forceinline__ void sk_step(float (&c)[16], int i, float eps) {
  if ((i & 1) == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float r = rcp_fast(((c[k] + c[4 + k]) + (c[8 + k] + c[12 + k])) + eps);
#pragma unroll
      for (int j = 0; j < 4; ++j) c[4 * j + k] *= r;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float r = rcp_fast(((c[4 * j] + c[4 * j + 1]) + (c[4 * j + 2] + c[4 * j + 3])) + eps);
#pragma unroll
      for (int k = 0; k < 4; ++k) c[4 * j + k] *= r;
    }
  }
}

// Derivative of step i at its input c: g <- g / s - (sum_line g c) / s^2 along each line.
__device__ __forceinline__ void sk_step_back(float (&g)[16], const float (&c)[16], int i, float eps) {
  if ((i & 1) == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float s = ((c[k] + c[4 + k]) + (c[8 + k] + c[12 + k])) + eps;
      const float gc = (g[k] * c[k] + g[4 + k] * c[4 + k]) + (g[8 + k] * c[8 + k] + g[12 + k] * c[12 + k]);
      const float inv = rcp_fast(s);
      const float t = gc * inv * inv;
#pragma unroll
      for (int j = 0; j < 4; ++j) g[4 * j + k] = g[4 * j + k] * inv - t;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* cr = c + 4 * j;
      float* gr = g + 4 * j;
      const float s = ((cr[0] + cr[1]) + (cr[2] + cr[3])) + eps;
      const float gc = (gr[0] * cr[0] + gr[1] * cr[1]) + (gr[2] * cr[2] + gr[3] * cr[3]);
      const float inv = rcp_fast(s);
      const float t = gc * inv * inv;
#pragma unroll
      for (int k = 0; k < 4; ++k) gr[k] = gr[k] * inv - t;
    }
  }
}

__device__ __forceinline__ float sigmoid_b(float z) { return 1.0f / (1.0f + expf(-z)); }

__global__ void __launch_bounds__(MIX_THREADS) bwd_mix_kernel(
    const float* __restrict__ mixes, const float* __restrict__ gpre, const float* __restrict__ gpost,
    const float* __restrict__ gcomb, const float* __restrict__ scale, const float* __restrict__ base,
    float* __restrict__ gm_out, float* __restrict__ part, int64_t N, int iters, float eps, int ck_every) {
  // step inputs every ck_every steps (at most CK_MAX of them), one column per thread
  __shared__ float ck[CK_MAX][16][MIX_THREADS];
  const int64_t t = blockIdx.x * static_cast<int64_t>(MIX_THREADS) + threadIdx.x;
  float contrib[MIXN + 3];
#pragma unroll
  for (int i = 0; i < MIXN + 3; ++i) contrib[i] = 0.f;
  if (t < N) {
    float m[MIXN];
#pragma unroll
    for (int i = 0; i < MIXN / 4; ++i) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(mixes + t * MIXN) + i);
      m[4 * i] = v.x;
      m[4 * i + 1] = v.y;
      m[4 * i + 2] = v.z;
      m[4 * i + 3] = v.w;
    }
    const float s0 = __ldg(scale), s1 = __ldg(scale + 1), s2 = __ldg(scale + 2);
    float g[16], c0[16], sm[16];
    // split: p_j = sigmoid(s0 m_j + b_j) + eps, u_j = 2 sigmoid(s1 m_{4+j} + b_{4+j})
    const float4 gp = __ldg(reinterpret_cast<const float4*>(gpre + t * 4));
    const float4 gu = __ldg(reinterpret_cast<const float4*>(gpost + t * 4));
    const float gpa[4] = {gp.x, gp.y, gp.z, gp.w}, gua[4] = {gu.x, gu.y, gu.z, gu.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float sp = sigmoid_b(fmaf(s0, m[j], __ldg(base + j)));
      const float su = sigmoid_b(fmaf(s1, m[4 + j], __ldg(base + 4 + j)));
      const float gzp = gpa[j] * sp * (1.0f - sp);
      const float gzu = 2.0f * gua[j] * su * (1.0f - su);
      contrib[j] = gzp;
      contrib[4 + j] = gzu;
      contrib[MIXN] += gzp * m[j];
      contrib[MIXN + 1] += gzu * m[4 + j];
    }
    // row softmax of the logits L = s2 m_L + b_L, then + eps
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float l[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) l[k] = fmaf(s2, m[8 + 4 * j + k], __ldg(base + 8 + 4 * j + k));
      const float mx = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
#pragma unroll
      for (int k = 0; k < 4; ++k) l[k] = expf(l[k] - mx);
      const float inv = 1.0f / ((l[0] + l[1]) + (l[2] + l[3]));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sm[4 * j + k] = l[k] * inv;
        c0[4 * j + k] = sm[4 * j + k] + eps;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(gcomb + t * 16) + i);
      g[4 * i] = v.x;
      g[4 * i + 1] = v.y;
      g[4 * i + 2] = v.z;
      g[4 * i + 3] = v.w;
    }
    // checkpoints of the step inputs every ck_every steps; then each step's derivative at its
    // input, recomputed from the checkpoint below it
    const int nsteps = 2 * iters - 1;
    {
      float c[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) c[e] = c0[e];
      for (int i = 0; i < nsteps; ++i) {
        if (i % ck_every == 0) {
#pragma unroll
          for (int e = 0; e < 16; ++e) ck[i / ck_every][e][threadIdx.x] = c[e];
        }
        sk_step(c, i, eps);
      }
    }
    for (int i = nsteps - 1; i >= 0; --i) {
      float c[16];
      const int base_i = (i / ck_every) * ck_every;
#pragma unroll
      for (int e = 0; e < 16; ++e) c[e] = ck[i / ck_every][e][threadIdx.x];
      for (int q = base_i; q < i; ++q) sk_step(c, q, eps);
      sk_step_back(g, c, i, eps);
    }
    // softmax: g_L = sm (g - sum_row(g sm)); the + eps has no derivative
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* s = sm + 4 * j;
      const float* gg = g + 4 * j;
      const float dot = (gg[0] * s[0] + gg[1] * s[1]) + (gg[2] * s[2] + gg[3] * s[3]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float gl = s[k] * (gg[k] - dot);
        contrib[8 + 4 * j + k] = gl;
        contrib[MIXN + 2] += gl * m[8 + 4 * j + k];
      }
    }
    float gmv[MIXN];
#pragma unroll
    for (int i = 0; i < MIXN; ++i) gmv[i] = contrib[i] * (i < 4 ? s0 : i < 8 ? s1 : s2);
#pragma unroll
    for (int i = 0; i < MIXN / 4; ++i)
      reinterpret_cast<float4*>(gm_out + t * MIXN)[i] =
          make_float4(gmv[4 * i], gmv[4 * i + 1], gmv[4 * i + 2], gmv[4 * i + 3]);
  }
  // block sums of g_base (contrib[0..23]) and g_scale (contrib[24..26])
  __shared__ float red[MIX_THREADS / 32][MIXN + 3];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < MIXN + 3; ++i) {
    float v = contrib[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp][i] = v;
  }
  __syncthreads();
  if (threadIdx.x < MIXN + 3) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < MIX_THREADS / 32; ++w) v += red[w][threadIdx.x];
    part[static_cast<int64_t>(blockIdx.x) * 32 + threadIdx.x] = v;
  }
}

// ---------------------------------------------------------------------------------------------
// bwd_token_kernel

constexpr int TOK_THREADS = 256;

// Per token: rec = {r, r_y, tau = r_y^3 T / d, c1 = (r^2 / K)(g_m . m)}, gp_prev, r g_m in fp32
// and as two bf16 planes (hi = bf16(v), lo = bf16(v - hi); 8 zero columns after each).
__global__ void __launch_bounds__(TOK_THREADS) bwd_token_kernel(
    const __nv_bfloat16* __restrict__ Xp, const __nv_bfloat16* __restrict__ gy,
    const float* __restrict__ pre_prev, const float* __restrict__ gain,
    const float* __restrict__ mixes, const float* __restrict__ gm, float* __restrict__ rec,
    float* __restrict__ gsf, __nv_bfloat16* __restrict__ gplanes, float* __restrict__ gpre_prev,
    int64_t N, int d, float norm_eps, float neg_zero) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (TOK_THREADS / 32);
  const f2 nz{neg_zero, neg_zero};
  const int chunks = d / 8;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(TOK_THREADS / 32) + (threadIdx.x >> 5); t < N;
       t += warps) {
    const float4 pv = __ldg(reinterpret_cast<const float4*>(pre_prev + t * 4));
    const f2 cp[4] = {f2{pv.x, pv.x}, f2{pv.y, pv.y}, f2{pv.z, pv.z}, f2{pv.w, pv.w}};
    f2 sx{0.f, 0.f}, sy{0.f, 0.f}, tt{0.f, 0.f}, A[4], Bv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) A[j] = Bv[j] = f2{0.f, 0.f};
    const __nv_bfloat16* xrow = Xp + t * 4 * static_cast<int64_t>(d);
    const __nv_bfloat16* grow = gy + t * static_cast<int64_t>(d);
#pragma unroll 2
    for (int c = lane; c < chunks; c += 32) {
      uint4 xw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) xw[j] = __ldg(reinterpret_cast<const uint4*>(xrow + j * static_cast<int64_t>(d)) + c);
      const uint4 yw = __ldg(reinterpret_cast<const uint4*>(grow) + c);
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(gain) + 2 * c);
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(gain) + 2 * c + 1);
      const uint32_t xa[4][4] = {{xw[0].x, xw[0].y, xw[0].z, xw[0].w}, {xw[1].x, xw[1].y, xw[1].z, xw[1].w},
                                 {xw[2].x, xw[2].y, xw[2].z, xw[2].w}, {xw[3].x, xw[3].y, xw[3].z, xw[3].w}};
      const uint32_t ya[4] = {yw.x, yw.y, yw.z, yw.w};
      const f2 ga[4] = {f2{g0.x, g0.y}, f2{g0.z, g0.w}, f2{g1.x, g1.y}, f2{g1.z, g1.w}};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        f2 xp[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xp[j] = bf2_to_f2(xa[j][w]);
          sx = fma2(xp[j], xp[j], sx);
        }
        const f2 yh = bf2_to_f2(f2_to_bf2(hc_pre_pair(cp, xp, nz)));
        sy = fma2(yh, yh, sy);
        const f2 gg = mul2(ga[w], bf2_to_f2(ya[w]));
        tt = fma2(gg, yh, tt);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          A[j] = fma2(gg, xp[j], A[j]);
          Bv[j] = fma2(yh, xp[j], Bv[j]);
        }
      }
    }
    float v[11] = {sx.x + sx.y, sy.x + sy.y, tt.x + tt.y};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[3 + j] = A[j].x + A[j].y;
      v[7 + j] = Bv[j].x + Bv[j].y;
    }
#pragma unroll
    for (int i = 0; i < 11; ++i)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    const float K = 4.0f * d;
    const float r = __frsqrt_rn(__fdiv_rn(v[0], K) + norm_eps);
    const float ry = __frsqrt_rn(__fdiv_rn(v[1], static_cast<float>(d)) + norm_eps);
    const float tau = ry * ry * ry * v[2] / static_cast<float>(d);
    const float gmi = lane < MIXN ? __ldg(gm + t * MIXN + lane) : 0.f;
    float gmm = lane < MIXN ? gmi * __ldg(mixes + t * MIXN + lane) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gmm += __shfl_xor_sync(0xffffffffu, gmm, o);
    const float c1 = r * r / K * gmm;
    const float gs = r * gmi;
    if (lane < MIXN) gsf[t * MIXN + lane] = gs;
    const __nv_bfloat16 hi = __float2bfloat16_rn(gs);
    const __nv_bfloat16 lo = __float2bfloat16_rn(gs - __bfloat162float(hi));
    gplanes[t * 64 + lane] = lane < MIXN ? hi : __float2bfloat16_rn(0.f);
    gplanes[t * 64 + 32 + lane] = lane < MIXN ? lo : __float2bfloat16_rn(0.f);
    if (lane == 0) {
      reinterpret_cast<float4*>(rec)[t] = make_float4(r, ry, tau, c1);
      reinterpret_cast<float4*>(gpre_prev)[t] =
          make_float4(ry * v[3] - tau * v[7], ry * v[4] - tau * v[8], ry * v[5] - tau * v[9],
                      ry * v[6] - tau * v[10]);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// bwd_stream_kernel

constexpr int BT = 128;                      // the MMA's M: rows of its A operand and of D
constexpr int BTR = 112;                     // token rows of a tile (at most): the ring tiles' height
constexpr int BDC = 32;                      // columns per slot
constexpr int BROWB = BDC * 2;               // 64-byte tile rows (64-byte swizzle)
constexpr int BTILE = BTR * BROWB;           // one [112 x 32] bf16 tile
constexpr int BSETB = 5 * BTILE;             // five tiles: X_0..3 and F, or gXp_0..3 and gy
// Two rings, by how long a slot's tiles are held: X and F are written over by gX and gF and freed
// once the stores have read them; gXp and gy are freed as soon as the consumers have read them.
constexpr int BNA = 3;                       // X/F entries
constexpr int BNB = 2;                       // gXp/gy entries
constexpr int BWB = 128 * 128;               // W^T planes of a slot: 128 rows (stream, column) x 128 B
constexpr int BNW = 1;                       // weight entries (refilled once a slot's MMAs are done)
constexpr int BAB = BT * 128;                // the tile's planes of r g_m: 128 rows x 128 B
constexpr int BOFF_B = BNA * BSETB;
constexpr int BOFF_W = BOFF_B + BNB * BSETB;
constexpr int BOFF_A = BOFF_W + BNW * BWB;
constexpr int BOFF_RED = BOFF_A + BAB;       // [BT][20] partial sums of the tile's second threads
constexpr int BOFF_BARS = BOFF_RED + BT * 20 * 4;
// fullA, emptyA, xready per X/F entry; fullB, emptyB per gXp/gy entry; wfull, wempty per weight
// entry; dready, dfree per TMEM buffer; afull, aempty
constexpr int BNBARS = 3 * BNA + 2 * BNB + 2 * BNW + 4 + 2;
constexpr int BOFF_TMEM = BOFF_BARS + BNBARS * 8;
constexpr int BSMEM = BOFF_TMEM + 16 + 1024;
static_assert(BSMEM <= 232448, "shared memory budget");
static_assert(BTILE % 512 == 0 && BSETB % 1024 == 0 && BWB % 1024 == 0 && BOFF_A % 1024 == 0,
              "tile alignment");
constexpr int BNCONS = 8;
constexpr int BTHREADS = (2 + BNCONS) * 32;
constexpr uint32_t BTMEM_COLS = 256;         // two [128 x 128] fp32 accumulators

__host__ __device__ constexpr int bx_tile(int a, int k) { return a * BSETB + k * BTILE; }            // X_k
__host__ __device__ constexpr int bf_tile(int a) { return a * BSETB + 4 * BTILE; }                   // F
__host__ __device__ constexpr int bg_tile(int b, int k) { return BOFF_B + b * BSETB + k * BTILE; }   // gXp_k
__host__ __device__ constexpr int by_tile(int b) { return BOFF_B + b * BSETB + 4 * BTILE; }          // gy

struct BwdParams {
  const float* pre_prev;
  const float* post_prev;
  const float* comb_prev;
  const float* rec;
  const float* gain;
  const uint8_t* wT;           // packed W^T planes, d / 32 slots of BWB bytes
  float* gpost_prev;
  float* gcomb_prev;
  unsigned* status;
  int N;
  int tt;
  int d;
  int ntiles;
  float neg_zero;
  unsigned flags;
};

__global__ void __launch_bounds__(BTHREADS, 1)
    bwd_stream_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_f,
                      const __grid_constant__ CUtensorMap tm_gxp, const __grid_constant__ CUtensorMap tm_gy,
                      const __grid_constant__ CUtensorMap tm_gx, const __grid_constant__ CUtensorMap tm_gf,
                      const __grid_constant__ CUtensorMap tm_g, const BwdParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* fullA = reinterpret_cast<uint64_t*>(sm + BOFF_BARS);
  uint64_t* emptyA = fullA + BNA;
  uint64_t* xready = emptyA + BNA;
  uint64_t* fullB = xready + BNA;
  uint64_t* emptyB = fullB + BNB;
  uint64_t* wfull = emptyB + BNB;
  uint64_t* wempty = wfull + BNW;
  uint64_t* dready = wempty + BNW;
  uint64_t* dfree = dready + 2;
  uint64_t* afull = dfree + 2;
  uint64_t* aempty = afull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + BOFF_TMEM);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tt = P.tt;
  const int S = P.d / BDC;
  const int ntiles = P.ntiles;
  bool timed_out = false;
  auto limit = [&]() { return timed_out ? 0ull : BWD_WAIT_NS; };
  const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int total = my_tiles * S;   // this CTA's slots

  if (threadIdx.x == 0) {
    for (int a = 0; a < BNA; ++a) {
      mbar_init(&fullA[a], 1);
      mbar_init(&emptyA[a], 1);
      mbar_init(&xready[a], BNCONS);
    }
    for (int b = 0; b < BNB; ++b) {
      mbar_init(&fullB[b], 1);
      mbar_init(&emptyB[b], BNCONS);
    }
    for (int e = 0; e < BNW; ++e) {
      mbar_init(&wfull[e], 1);
      mbar_init(&wempty[e], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&dready[i], 1);
      mbar_init(&dfree[i], BNCONS);
    }
    mbar_init(afull, 1);
    mbar_init(aempty, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, BTMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  block_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_f);
      tma_prefetch_desc(&tm_gxp);
      tma_prefetch_desc(&tm_gy);
      // normal eviction priority: each CTA reads its slots one after another, so a tile's rows
      // stay in L2 between the slots that read them (measured 9% faster than evict-first)
      const uint64_t pol = policy_evict_normal();
      const uint32_t bytes = 5u * static_cast<uint32_t>(tt * BROWB);   // five tt-row boxes
      int gs = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int t0 = tile * tt;
        for (int s = 0; s < S; ++s, ++gs) {
          const int a = gs % BNA, b = gs % BNB;
          const int col = s * BDC;
          if (gs >= BNA && !mbar_wait(&emptyA[a], ((gs / BNA) - 1) & 1, limit())) timed_out = true;
          mbar_arrive_expect_tx(&fullA[a], bytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) tma_load_3d_hint(sm + bx_tile(a, k), &tm_x, &fullA[a], col, k, t0, pol);
          tma_load_2d_hint(sm + bf_tile(a), &tm_f, &fullA[a], col, t0, pol);
          if (gs >= BNB && !mbar_wait(&emptyB[b], ((gs / BNB) - 1) & 1, limit())) timed_out = true;
          mbar_arrive_expect_tx(&fullB[b], bytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) tma_load_3d_hint(sm + bg_tile(b, k), &tm_gxp, &fullB[b], col, k, t0, pol);
          tma_load_2d_hint(sm + by_tile(b), &tm_gy, &fullB[b], col, t0, pol);
        }
      }
    } else if (lane == 1) {
      // -------------------------------------------------------------- gX / gF stores
      tma_prefetch_desc(&tm_gx);
      tma_prefetch_desc(&tm_gf);
      const uint64_t pol = policy_evict_first();
      int gs = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int t0 = tile * tt;
        for (int s = 0; s < S; ++s, ++gs) {
          const int a = gs % BNA;
          if (!mbar_wait(&xready[a], (gs / BNA) & 1, limit())) timed_out = true;
          const int col = s * BDC;
#pragma unroll
          for (int k = 0; k < 4; ++k) tma_store_3d_hint(&tm_gx, sm + bx_tile(a, k), col, k, t0, pol);
          tma_store_2d_hint(&tm_gf, sm + bf_tile(a), col, t0, pol);
          bulk_commit();
          bulk_wait_read<0>();
          mbar_arrive(&emptyA[a]);
        }
      }
      bulk_wait<0>();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && total > 0) {
      tma_prefetch_desc(&tm_g);
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint64_t wpol = policy_evict_last();
      auto load_w = [&](int u) {   // slot u of this CTA (slot u % S of its tile) into entry u % BNW
        const int e = u % BNW;
        mbar_arrive_expect_tx(&wfull[e], BWB);
        bulk_load_hint(sm + BOFF_W + e * BWB, P.wT + static_cast<size_t>(u % S) * BWB, BWB, &wfull[e], wpol);
      };
      auto load_a = [&](int tile) {
        mbar_arrive_expect_tx(afull, static_cast<uint32_t>(tt * 128));
        tma_load_2d(sm + BOFF_A, &tm_g, afull, 0, tile * tt);
      };
      for (int u = 0; u < BNW && u < total; ++u) load_w(u);
      load_a(blockIdx.x);
      int gs = 0;
      for (int tile = blockIdx.x, it = 0; tile < ntiles; tile += gridDim.x, ++it) {
        if (!mbar_wait(afull, it & 1, limit())) timed_out = true;
        for (int s = 0; s < S; ++s, ++gs) {
          const int db = gs & 1, e = gs % BNW;
          if (!mbar_wait(&wfull[e], (gs / BNW) & 1, limit())) timed_out = true;
          if (gs >= 2 && !mbar_wait(&dfree[db], ((gs >> 1) - 1) & 1, limit())) timed_out = true;
          tc_fence_after();
          const uint32_t acc = tmem + static_cast<uint32_t>(db * 128);
          const uint32_t a0 = smem_u32(sm + BOFF_A);
          const uint32_t b0 = smem_u32(sm + BOFF_W + e * BWB);
          // (hi, hi), (hi, lo), (lo, hi): columns 0..31 of a plane row hold hi, 32..63 lo
          int n = 0;
#pragma unroll
          for (int pr = 0; pr < 3; ++pr) {
            const int pa = pr == 2 ? 1 : 0, pb = pr == 1 ? 1 : 0;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk, ++n)
              umma_bf16(acc, sdesc_kmajor_swizzled(a0 + 64 * pa + 32 * kk, 128),
                        sdesc_kmajor_swizzled(b0 + 64 * pb + 32 * kk, 128), idesc, n == 0 ? 0u : 1u);
          }
          umma_commit(&dready[db]);
          umma_commit(&wempty[e]);
          if (s == S - 1) umma_commit(aempty);
          if (gs + BNW < total) {
            if (!mbar_wait(&wempty[e], (gs / BNW) & 1, limit())) timed_out = true;
            load_w(gs + BNW);
          }
        }
        if (tile + static_cast<int>(gridDim.x) < ntiles) {
          if (!mbar_wait(aempty, it & 1, limit())) timed_out = true;
          load_a(tile + gridDim.x);
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ consumers
    const int c = warp - 2;
    const int sub = warp & 3;            // TMEM lane quarter
    const int h = c >> 2;                // which 16 columns of the slot
    const int tl = sub * 32 + lane;      // token row of the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    // Threads whose row is past the tiles' height (tl >= 112) read the first rows of the next
    // buffer in shared memory (no token of theirs is ever stored) and write nothing.
    const bool inrows = tl < BTR;
    uint32_t row_off[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) row_off[q] = tile_chunk_offset(tl, 2 * h + q);
    auto at = [&](int tile_off, int q) { return sm + tile_off + row_off[q]; };
    const f2 nz{P.neg_zero, P.neg_zero};
    const bool row_dest = (P.flags & 1u) != 0;
    float* red = reinterpret_cast<float*>(sm + BOFF_RED) + tl * 20;
    int gs = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const int token = tile * tt + tl;
      const bool valid = tl < tt && token < P.N;
      // the token's coefficients: cc[j][k] = weight of input stream j in output stream k
      f2 cc[4][4], cu[4], cpp[4];
      f2 r_y2, tau2, c12;
      {
        float cm[16], u[4], p[4], rc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = valid ? __ldg(reinterpret_cast<const float4*>(P.comb_prev) + static_cast<size_t>(token) * 4 + i)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
          cm[4 * i] = v.x;
          cm[4 * i + 1] = v.y;
          cm[4 * i + 2] = v.z;
          cm[4 * i + 3] = v.w;
        }
        const float4 uv = valid ? __ldg(reinterpret_cast<const float4*>(P.post_prev) + token) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 pv = valid ? __ldg(reinterpret_cast<const float4*>(P.pre_prev) + token) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 rv = valid ? __ldg(reinterpret_cast<const float4*>(P.rec) + token) : make_float4(0.f, 0.f, 0.f, 0.f);
        u[0] = uv.x; u[1] = uv.y; u[2] = uv.z; u[3] = uv.w;
        p[0] = pv.x; p[1] = pv.y; p[2] = pv.z; p[3] = pv.w;
        rc[0] = rv.x; rc[1] = rv.y; rc[2] = rv.z; rc[3] = rv.w;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          cu[k] = f2{u[k], u[k]};
          cpp[k] = f2{p[k], p[k]};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float w = row_dest ? cm[4 * k + j] : cm[4 * j + k];
            cc[j][k] = f2{w, w};
          }
        }
        r_y2 = f2{rc[1], rc[1]};
        tau2 = f2{-rc[2], -rc[2]};
        c12 = f2{-rc[3], -rc[3]};
      }
      float acc_u[4], acc_c[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc_u[k] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc_c[j][k] = 0.f;
      }
      for (int s = 0; s < S; ++s, ++gs) {
        const int a = gs % BNA, b = gs % BNB, db = gs & 1;
        if (!mbar_wait(&fullA[a], (gs / BNA) & 1, limit())) timed_out = true;
        if (!mbar_wait(&fullB[b], (gs / BNB) & 1, limit())) timed_out = true;
        if (!mbar_wait(&dready[db], (gs >> 1) & 1, limit())) timed_out = true;
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          // W^T (r g_m) of this thread's 8 columns of each stream
          uint32_t gw[4][8];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tmem_ld_x8_nowait(lane_base + static_cast<uint32_t>(db * 128 + k * 32 + 16 * h + 8 * q), gw[k]);
          uint32_t xa[4][4], fa[4], ga[4][4], ya[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(at(bx_tile(a, k), q));
            xa[k][0] = v.x; xa[k][1] = v.y; xa[k][2] = v.z; xa[k][3] = v.w;
            const uint4 g = *reinterpret_cast<const uint4*>(at(bg_tile(b, k), q));
            ga[k][0] = g.x; ga[k][1] = g.y; ga[k][2] = g.z; ga[k][3] = g.w;
          }
          {
            const uint4 v = *reinterpret_cast<const uint4*>(at(bf_tile(a), q));
            fa[0] = v.x; fa[1] = v.y; fa[2] = v.z; fa[3] = v.w;
            const uint4 y = *reinterpret_cast<const uint4*>(at(by_tile(b), q));
            ya[0] = y.x; ya[1] = y.y; ya[2] = y.z; ya[3] = y.w;
          }
          const int col = s * BDC + 16 * h + 8 * q;
          const float4 g0 = __ldg(reinterpret_cast<const float4*>(P.gain + col));
          const float4 g1 = __ldg(reinterpret_cast<const float4*>(P.gain + col + 4));
          const f2 gn[4] = {f2{g0.x, g0.y}, f2{g0.z, g0.w}, f2{g1.x, g1.y}, f2{g1.z, g1.w}};
          tmem_ld_wait();
          uint32_t ox[4][4], of[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const f2 f = bf2_to_f2(fa[w]);
            f2 x[4], xp[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = bf2_to_f2(xa[j][w]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const f2 ck[4] = {cc[0][k], cc[1][k], cc[2][k], cc[3][k]};
              xp[k] = bf2_to_f2(f2_to_bf2(hc_post_pair(ck, cu[k], x, f, nz)));
            }
            const f2 yh = bf2_to_f2(f2_to_bf2(hc_pre_pair(cpp, xp, nz)));
            // g_y_hat = r_y gain gy - tau y_hat
            const f2 gyh = fma2(mul2(r_y2, gn[w]), bf2_to_f2(ya[w]), mul2(tau2, yh));
            f2 gxp[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const f2 gmix{__uint_as_float(gw[k][2 * w]), __uint_as_float(gw[k][2 * w + 1])};
              f2 v = fma2(cpp[k], gyh, bf2_to_f2(ga[k][w]));
              v = add2(v, gmix);
              gxp[k] = fma2(c12, xp[k], v);
              acc_u[k] = fmaf(gxp[k].x, f.x, fmaf(gxp[k].y, f.y, acc_u[k]));
#pragma unroll
              for (int j = 0; j < 4; ++j)
                acc_c[j][k] = fmaf(gxp[k].x, x[j].x, fmaf(gxp[k].y, x[j].y, acc_c[j][k]));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              f2 v = mul2(cc[j][0], gxp[0]);
              v = fma2(cc[j][1], gxp[1], v);
              v = fma2(cc[j][2], gxp[2], v);
              v = fma2(cc[j][3], gxp[3], v);
              ox[j][w] = f2_to_bf2(v);
            }
            f2 vf = mul2(cu[0], gxp[0]);
            vf = fma2(cu[1], gxp[1], vf);
            vf = fma2(cu[2], gxp[2], vf);
            vf = fma2(cu[3], gxp[3], vf);
            of[w] = f2_to_bf2(vf);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (inrows) *reinterpret_cast<uint4*>(at(bx_tile(a, k), q)) = make_uint4(ox[k][0], ox[k][1], ox[k][2], ox[k][3]);
          if (inrows) *reinterpret_cast<uint4*>(at(bf_tile(a), q)) = make_uint4(of[0], of[1], of[2], of[3]);
        }
        tc_fence_before();   // the TMEM loads above, before the MMA that reuses the buffer
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&dfree[db]);
          mbar_arrive(&emptyB[b]);   // this warp has read the slot's gXp and gy
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&xready[a]);
      }
      // the token's gu and gC: the second thread's partial sums through shared memory
      if (h == 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          red[k] = acc_u[k];
#pragma unroll
          for (int j = 0; j < 4; ++j) red[4 + 4 * j + k] = acc_c[j][k];
        }
      }
      named_bar_sync(1 + sub, 64);
      if (h == 0 && valid) {
        float4 u4 = make_float4(acc_u[0] + red[0], acc_u[1] + red[1], acc_u[2] + red[2], acc_u[3] + red[3]);
        reinterpret_cast<float4*>(P.gpost_prev)[token] = u4;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) o[k] = acc_c[j][k] + red[4 + 4 * j + k];
          if (!row_dest) {
            reinterpret_cast<float4*>(P.gcomb_prev)[static_cast<size_t>(token) * 4 + j] = make_float4(o[0], o[1], o[2], o[3]);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) P.gcomb_prev[static_cast<size_t>(token) * 16 + 4 * k + j] = o[k];
          }
        }
      }
      named_bar_sync(1 + sub, 64);
    }
  }

  if (timed_out) atomicOr(P.status, STATUS_TIMEOUT);
  tc_fence_before();
  block_sync();
  if (warp == 1) tmem_dealloc(tmem, BTMEM_COLS);
}

// W^T planes for the stream kernel's B operand: slot s (columns 32s .. 32s + 31 of every stream)
// is 128 rows, row 32k + c for column c of stream k, each 64 bf16: W_hi[0..23], 8 zeros,
// W_lo[0..23], 8 zeros (hi = bf16(w), lo = bf16(w - hi)), with the 128-byte swizzle of the
// tensor cores' operand tiles. One thread per 16-byte chunk.
__global__ void pack_wt_kernel(const float* __restrict__ W, uint8_t* __restrict__ out, int d) {
  const int64_t K = 4 * static_cast<int64_t>(d);
  const int64_t total = static_cast<int64_t>(d / BDC) * 128 * 8;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int chunk = static_cast<int>(idx % 8);
    const int row = static_cast<int>((idx / 8) % 128);
    const int64_t s = idx / (8 * 128);
    const int64_t col = (row / 32) * static_cast<int64_t>(d) + s * BDC + row % 32;
    uint32_t words[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint16_t hv[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = chunk * 8 + 2 * e + q;      // 0..63
        const int o = j & 31;
        __nv_bfloat16 v = __float2bfloat16_rn(0.f);
        if (o < MIXN) {
          const float w = W[o * K + col];
          const __nv_bfloat16 hi = __float2bfloat16_rn(w);
          v = j < 32 ? hi : __float2bfloat16_rn(w - __bfloat162float(hi));
        }
        hv[q] = __bfloat16_as_ushort(v);
      }
      words[e] = static_cast<uint32_t>(hv[0]) | (static_cast<uint32_t>(hv[1]) << 16);
    }
    uint8_t* dst = out + s * BWB + swizzled_chunk_offset(row, chunk, 128);
    *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
  }
}

// ---------------------------------------------------------------------------------------------
// bwd_weight_kernel: per work item (64-column block cb of all four streams, token range tr), the
// partial sums over the range's tokens of gW[o][k d + c] = sum_t (r g_m)_t,o X'_t,k,c on the
// tensor cores, and of ggain[c] = sum_t r_y gy_t,c y_hat_t,c on the consumer warps.
//
// The contraction runs over tokens, so both operands are read token-major as TMA lays them
// down: A = X'^T (M = 128 of the block's 256 (stream, column) values, MN-major, 128-byte
// swizzle: 64 columns of one stream per 128-byte row, two streams LBO apart, 8-token groups
// 1 KB apart) and B = both bf16 planes of r g_m side by side (N = 64: hi in columns 0-31, lo in
// 32-63, 24 mix rows of each used; MN-major, 128-byte swizzle), so one MMA takes a K-step of
// both planes: 8 MMAs per stage. Two accumulators of [128 x 64] (streams 0-1 and 2-3, hi then lo
// columns) stay in TMEM for the whole range; the epilogue adds each row's hi and lo sums (X' is
// exact in bf16).

constexpr int WT_COLS = 64;                  // columns per work item (of each stream)
constexpr int WT_TB = 64;                    // tokens per stage (four MMA K-steps)
constexpr int WT_NST = 4;                    // stages
constexpr int WT_XB = WT_TB * 128;           // one X'_k box: [64 tokens x 64 columns] bf16
constexpr int WT_OFF_GY = 4 * WT_XB;
constexpr int WT_OFF_G = WT_OFF_GY + WT_XB;          // planes [64 tokens x (32 hi | 32 lo)] bf16
constexpr int WT_OFF_P = WT_OFF_G + WT_TB * 128;     // p_prev [64][4] fp32
constexpr int WT_OFF_R = WT_OFF_P + WT_TB * 16;      // {r, r_y, tau, c1} [64][4] fp32
constexpr int WT_STAGE = WT_OFF_R + WT_TB * 16;
constexpr int WT_OFF_RED = WT_NST * WT_STAGE;        // ggain partials [4 phases][64 columns]
constexpr int WT_OFF_BARS = WT_OFF_RED + 4 * WT_COLS * 4;
// full, empty per stage; dfull, dfree
constexpr int WT_NBARS = 2 * WT_NST + 2;
constexpr int WT_OFF_TMEM = WT_OFF_BARS + WT_NBARS * 8;
constexpr int WT_SMEM = WT_OFF_TMEM + 16 + 1024;
static_assert(WT_STAGE % 1024 == 0, "stage alignment (128-byte swizzle)");
static_assert(WT_SMEM <= 232448, "shared memory budget");
constexpr int WT_CONS = 4;                   // consumer / epilogue warps (2..5)
constexpr int WT_THREADS = (2 + WT_CONS) * 32;
constexpr uint32_t WT_TMEM_COLS = 128;

// Shared-memory descriptor of an MN-major operand: `row_bytes` (64 or 128) of the MN dimension
// per row with the swizzle of that width, consecutive K rows row_bytes apart, 8-row K groups
// `sbo` bytes apart, the next MN atom `lbo` bytes on.
__device__ __forceinline__ uint64_t sdesc_mnmajor(uint32_t saddr, int row_bytes, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(row_bytes == 128 ? 2 : 4) << 61);
}

struct WtParams {
  float* partW;
  float* partG;
  const float* pre_prev;
  const float* rec;
  unsigned* status;
  int64_t N;
  int d;
  int ranges;
  int64_t per;          // tokens per range (a multiple of WT_TB)
  float neg_zero;
};

__global__ void __launch_bounds__(WT_THREADS, 1)
    bwd_weight_kernel(const __grid_constant__ CUtensorMap tm_xp, const __grid_constant__ CUtensorMap tm_gy,
                      const __grid_constant__ CUtensorMap tm_gp, const WtParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + WT_OFF_BARS);
  uint64_t* empty = full + WT_NST;
  uint64_t* dfull = empty + WT_NST;
  uint64_t* dfree = dfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + WT_OFF_TMEM);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblocks = P.d / WT_COLS;
  const int64_t items = static_cast<int64_t>(nblocks) * P.ranges;
  bool timed_out = false;
  auto limit = [&]() { return timed_out ? 0ull : BWD_WAIT_NS; };
  // batches of an item: its token range cut into stages of WT_TB tokens
  auto range_of = [&](int64_t item, int64_t& t0, int64_t& t1) {
    const int tr = static_cast<int>(item / nblocks);
    t0 = tr * P.per;
    t1 = std::min<int64_t>(P.N, t0 + P.per);
  };

  if (threadIdx.x == 0) {
    for (int b = 0; b < WT_NST; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], 1 + WT_CONS);
    }
    mbar_init(dfull, 1);
    mbar_init(dfree, WT_CONS);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, WT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  block_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_xp);
      tma_prefetch_desc(&tm_gy);
      tma_prefetch_desc(&tm_gp);
      const uint64_t pol = policy_evict_first();
      int g = 0;
      for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int cb = static_cast<int>(item % nblocks);
        int64_t t0, t1;
        range_of(item, t0, t1);
        for (int64_t tb = t0; tb < t1; tb += WT_TB, ++g) {
          const int b = g % WT_NST;
          if (g >= WT_NST && !mbar_wait(&empty[b], ((g / WT_NST) - 1) & 1, limit())) timed_out = true;
          const uint32_t nt = static_cast<uint32_t>(std::min<int64_t>(WT_TB, P.N - tb));
          uint8_t* st = sm + b * WT_STAGE;
          // the boxes always move WT_TB rows (rows past N read as zero); p and rec move nt rows
          mbar_arrive_expect_tx(&full[b], 5u * WT_XB + WT_TB * 128u + 2u * nt * 16);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tma_load_3d_hint(st + k * WT_XB, &tm_xp, &full[b], cb * WT_COLS, k, static_cast<int>(tb), pol);
          tma_load_2d_hint(st + WT_OFF_GY, &tm_gy, &full[b], cb * WT_COLS, static_cast<int>(tb), pol);
          tma_load_2d(st + WT_OFF_G, &tm_gp, &full[b], 0, static_cast<int>(tb));
          bulk_load_hint(st + WT_OFF_P, P.pre_prev + tb * 4, nt * 16, &full[b], pol);
          bulk_load_hint(st + WT_OFF_R, P.rec + tb * 4, nt * 16, &full[b], pol);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // bf16 A and B, fp32 D, M = 128, N = 64 (both planes), both operands MN-major
      constexpr uint32_t idesc = idesc_bf16_f32(128, 64) | (1u << 15) | (1u << 16);
      int g = 0, it = 0;
      for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
        int64_t t0, t1;
        range_of(item, t0, t1);
        // the epilogue has read the previous item's accumulators
        if (it > 0 && !mbar_wait(dfree, (it - 1) & 1, limit())) timed_out = true;
        tc_fence_after();
        bool first = true;
        for (int64_t tb = t0; tb < t1; tb += WT_TB, ++g) {
          const int b = g % WT_NST;
          if (!mbar_wait(&full[b], (g / WT_NST) & 1, limit())) timed_out = true;
          tc_fence_after();
          const uint32_t st = smem_u32(sm + b * WT_STAGE);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
            for (int ks = 0; ks < WT_TB / 16; ++ks) {
              const uint64_t a = sdesc_mnmajor(st + 2 * mt * WT_XB + ks * 2048, 128, WT_XB, 1024);
              const uint64_t bd = sdesc_mnmajor(st + WT_OFF_G + ks * 2048, 128, 0, 1024);
              umma_bf16(tmem + static_cast<uint32_t>(mt * 64), a, bd, idesc, (first && ks == 0) ? 0u : 1u);
            }
          }
          first = false;
          umma_commit(&empty[b]);
        }
        umma_commit(dfull);
      }
    }
  } else {
    // ------------------------------------------------------------------ ggain and epilogue
    const int ct = threadIdx.x - 64;            // 0..127
    const int cp = ct & 31;                     // column pair: columns 2cp, 2cp+1 of the block
    const int ph = ct >> 5;                     // tokens ph, ph + 4, ...
    const int q = warp & 3;                     // TMEM lane quarter
    const f2 nz{P.neg_zero, P.neg_zero};
    float* red = reinterpret_cast<float*>(sm + WT_OFF_RED);
    int g = 0, it = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
      const int cb = static_cast<int>(item % nblocks);
      const int tr = static_cast<int>(item / nblocks);
      int64_t t0, t1;
      range_of(item, t0, t1);
      f2 gacc{0.f, 0.f};
      for (int64_t tb = t0; tb < t1; tb += WT_TB, ++g) {
        const int b = g % WT_NST;
        if (!mbar_wait(&full[b], (g / WT_NST) & 1, limit())) timed_out = true;
        const int nt = static_cast<int>(std::min<int64_t>(WT_TB, t1 - tb));
        const uint8_t* st = sm + b * WT_STAGE;
        const float* sp = reinterpret_cast<const float*>(st + WT_OFF_P);
        const float* sr = reinterpret_cast<const float*>(st + WT_OFF_R);
        for (int t = ph; t < nt; t += 4) {
          // column pair cp of token row t in a 128-byte-swizzled box
          const uint32_t off = static_cast<uint32_t>(t * 128) +
                               ((static_cast<uint32_t>((cp >> 2) ^ (t & 7))) << 4) + (cp & 3) * 4;
          f2 xp[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) xp[k] = bf2_to_f2(*reinterpret_cast<const uint32_t*>(st + k * WT_XB + off));
          const float4 p = *reinterpret_cast<const float4*>(sp + 4 * t);
          const f2 cpv[4] = {f2{p.x, p.x}, f2{p.y, p.y}, f2{p.z, p.z}, f2{p.w, p.w}};
          const f2 yh = bf2_to_f2(f2_to_bf2(hc_pre_pair(cpv, xp, nz)));
          const f2 gyv = bf2_to_f2(*reinterpret_cast<const uint32_t*>(st + WT_OFF_GY + off));
          const float ry = sr[4 * t + 1];
          gacc = fma2(mul2(gyv, f2{ry, ry}), yh, gacc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
      }
      // gW partials of the range: accumulator mt holds (stream 2mt + m / 64, column m % 64) in
      // TMEM lane m, mix row o's hi-plane sum in column 64 mt + o and lo-plane sum in 64 mt + 32 + o
      if (!mbar_wait(dfull, it & 1, limit())) timed_out = true;
      tc_fence_after();
      float* pw = P.partW + static_cast<int64_t>(tr) * MIXN * 4 * P.d;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        uint32_t v[32], w[32];
        tmem_ld_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(mt * 64), v);
        tmem_ld_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(mt * 64 + 32), w);
        if (t1 <= t0) {   // a range past the last token: no MMA ran, its sums are zero
#pragma unroll
          for (int o = 0; o < 32; ++o) v[o] = w[o] = 0u;
        }
        const int m = q * 32 + lane;
        const int64_t col = static_cast<int64_t>(2 * mt + (m >> 6)) * P.d + cb * WT_COLS + (m & 63);
#pragma unroll
        for (int o = 0; o < MIXN; ++o)
          pw[static_cast<int64_t>(o) * 4 * P.d + col] = __uint_as_float(v[o]) + __uint_as_float(w[o]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dfree);
      // ggain partials of the range: the four token phases of each column added in order
      red[ph * WT_COLS + 2 * cp] = gacc.x;
      red[ph * WT_COLS + 2 * cp + 1] = gacc.y;
      named_bar_sync(1, WT_CONS * 32);
      if (ct < WT_COLS)
        P.partG[static_cast<int64_t>(tr) * P.d + cb * WT_COLS + ct] =
            (red[ct] + red[WT_COLS + ct]) + (red[2 * WT_COLS + ct] + red[3 * WT_COLS + ct]);
      named_bar_sync(1, WT_CONS * 32);
    }
  }

  if (timed_out) atomicOr(P.status, STATUS_TIMEOUT);
  tc_fence_before();
  block_sync();
  if (warp == 1) tmem_dealloc(tmem, WT_TMEM_COLS);
}

// Sums of the partials in a fixed order: gW [24][4d] and ggain [d] over `ranges` (four
// consecutive outputs per thread, one float4 load per range), and in the last block g_base [24]
// and g_scale [3] over the mix kernel's blocks (eight strided partial sums per output, then
// added in order).
__global__ void __launch_bounds__(256) bwd_reduce_kernel(
    const float* __restrict__ partW, const float* __restrict__ partG, const float* __restrict__ part0,
    float* __restrict__ gW, float* __restrict__ ggain, float* __restrict__ gbase,
    float* __restrict__ gscale, int d, int ranges, int blocks0) {
  if (blockIdx.x == gridDim.x - 1) {
    __shared__ float red[8][32];
    const int j = threadIdx.x & 31, q = threadIdx.x >> 5;
    float v = 0.f;
    if (j < MIXN + 3)
      for (int b = q; b < blocks0; b += 8) v += part0[static_cast<int64_t>(b) * 32 + j];
    red[q][j] = v;
    __syncthreads();
    if (threadIdx.x < MIXN + 3) {
      float t = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) t += red[k][threadIdx.x];
      if (threadIdx.x < MIXN) gbase[threadIdx.x] = t;
      else gscale[threadIdx.x - MIXN] = t;
    }
    return;
  }
  const int64_t nW4 = static_cast<int64_t>(MIXN) * d;     // float4s of gW (24 x 4d floats)
  const int64_t nG4 = d / 4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nW4 + nG4;
       i += static_cast<int64_t>(gridDim.x - 1) * blockDim.x) {
    const bool w = i < nW4;
    const float4* src = w ? reinterpret_cast<const float4*>(partW) + i
                          : reinterpret_cast<const float4*>(partG) + (i - nW4);
    const int64_t stride = w ? nW4 : nG4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int r = 0; r < ranges; ++r) {
      const float4 p = __ldg(src + r * stride);
      v.x += p.x;
      v.y += p.y;
      v.z += p.z;
      v.w += p.w;
    }
    if (w) reinterpret_cast<float4*>(gW)[i] = v;
    else reinterpret_cast<float4*>(ggain)[i - nW4] = v;
  }
}

// ---------------------------------------------------------------------------------------------
// host side

// No L2 promotion: a CTA of these kernels reads the neighbouring columns of a row only slots
// later, so fetching them early only adds traffic.
bool bmap(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
          const cuuint32_t* box, CUtensorMapSwizzle swz) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool bmap_streams(CUtensorMap* m, const void* p, int64_t N, int d, uint32_t rows) {   // [N, 4, d]
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), 4, static_cast<cuuint64_t>(N)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 8};
  const cuuint32_t box[3] = {BDC, 1, rows};
  return bmap(m, p, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B);
}
bool bmap_streams_box(CUtensorMap* m, const void* p, int64_t N, int d, uint32_t cols, uint32_t rows,
                      CUtensorMapSwizzle swz) {   // [N, 4, d], boxes of [rows x cols] of one stream
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), 4, static_cast<cuuint64_t>(N)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 8};
  const cuuint32_t box[3] = {cols, 1, rows};
  return bmap(m, p, 3, dims, str, box, swz);
}
bool bmap_rows(CUtensorMap* m, const void* p, int64_t N, int cols, uint32_t box_cols, uint32_t rows,
               CUtensorMapSwizzle swz) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(N)};
  const cuuint64_t str[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {box_cols, rows};
  return bmap(m, p, 2, dims, str, box, swz);
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

int gcd_i(int a, int b) { return b == 0 ? a : gcd_i(b, a % b); }

size_t a256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

BwdLayout bwd_layout(int64_t N, int d) {
  BwdLayout L{};
  const int sms = sm_count();
  if (sms <= 0 || d <= 0 || d % WT_COLS != 0) return L;
  const int grid = sms;
  const int nblocks = d / WT_COLS;
  int ranges = grid / gcd_i(grid, nblocks);
  ranges = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({static_cast<int64_t>(ranges), 64,
                                                                     (N + WT_TB - 1) / WT_TB})));
  // tokens per range: a multiple of the stage height, so only the last range ends in a partial
  // stage (whose rows past N read as zero)
  L.per = std::max<int64_t>(WT_TB, ((N + ranges - 1) / ranges + WT_TB - 1) / WT_TB * WT_TB);
  L.ranges = ranges;
  L.blocks0 = static_cast<int>(std::max<int64_t>(1, (N + MIX_THREADS - 1) / MIX_THREADS));
  size_t off = 0;
  L.off_wt = off;    off += a256(static_cast<size_t>(d / BDC) * BWB);
  L.off_gm = off;    off += a256(static_cast<size_t>(N) * MIXN * 4);
  L.off_rec = off;   off += a256(static_cast<size_t>(N) * 16);
  L.off_gsf = off;   off += a256(static_cast<size_t>(N) * MIXN * 4);
  L.off_gpl = off;   off += a256(static_cast<size_t>(N) * 128);
  L.off_part0 = off; off += a256(static_cast<size_t>(L.blocks0) * 128);
  L.off_partW = off; off += a256(static_cast<size_t>(ranges) * MIXN * 4 * d * 4);
  L.off_partG = off; off += a256(static_cast<size_t>(ranges) * d * 4);
  L.bytes = off;
  return L;
}

cudaError_t launch_backward(const BwdArgs& a, cudaStream_t stream) {
  const BwdLayout L = bwd_layout(a.N, a.d);
  if (L.bytes == 0) return cudaErrorInvalidValue;
  if (a.workspace_bytes < L.bytes) return cudaErrorInvalidValue;
  const int sms = sm_count();
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  auto wsf = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  const int d = a.d;
  const int64_t N = a.N;
  unsigned* status = status_word();
  if (status == nullptr) return cudaErrorInvalidDevice;

  // W^T planes
  {
    const int64_t chunks = static_cast<int64_t>(d / BDC) * 128 * 8;
    const int blocks = static_cast<int>(std::min<int64_t>((chunks + 255) / 256, 4096));
    pack_wt_kernel<<<blocks, 256, 0, stream>>>(a.W, ws + L.off_wt, d);
  }
  bwd_mix_kernel<<<L.blocks0, MIX_THREADS, 0, stream>>>(a.mixes, a.gpre, a.gpost, a.gcomb, a.scale, a.base,
                                                        wsf(L.off_gm), wsf(L.off_part0), N, a.iters,
                                                        a.hc_eps, std::max(CK_EVERY, (2 * a.iters - 1 + CK_MAX - 1) / CK_MAX));
  // (ck_every >= ceil(steps / CK_MAX): every checkpoint index stays below CK_MAX)
  {
    const int64_t warps_needed = N;
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((warps_needed + 7) / 8, 8 * sms)));
    bwd_token_kernel<<<blocks, TOK_THREADS, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.Xp), static_cast<const __nv_bfloat16*>(a.gy), a.pre_prev, a.gain,
        a.mixes, wsf(L.off_gm), wsf(L.off_rec), wsf(L.off_gsf),
        reinterpret_cast<__nv_bfloat16*>(ws + L.off_gpl), a.gpre_prev, N, d, a.norm_eps, -0.0f);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // stream kernel: tile height that balances the tiles over the SMs
  {
    int best_tt = BTR;
    int64_t best = INT64_MAX;
    for (int tt = BTR; tt >= 8; tt -= 8) {
      const int64_t tiles = (N + tt - 1) / tt;
      const int64_t rounds = (tiles + sms - 1) / sms;
      const int64_t cost = rounds * (tt + 32);
      if (cost < best) {
        best = cost;
        best_tt = tt;
      }
    }
    const int tt = best_tt;
    const int ntiles = static_cast<int>((N + tt - 1) / tt);
    CUtensorMap tx, tf, tgxp, tgy, tgx, tgf, tg;
    if (!bmap_streams(&tx, a.X, N, d, tt) || !bmap_rows(&tf, a.F, N, d, BDC, tt, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !bmap_streams(&tgxp, a.gXp, N, d, tt) || !bmap_rows(&tgy, a.gy, N, d, BDC, tt, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !bmap_streams(&tgx, a.gX, N, d, tt) || !bmap_rows(&tgf, a.gF, N, d, BDC, tt, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !bmap_rows(&tg, ws + L.off_gpl, N, 64, 64, tt, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    BwdParams P{};
    P.pre_prev = a.pre_prev;
    P.post_prev = a.post_prev;
    P.comb_prev = a.comb_prev;
    P.rec = wsf(L.off_rec);
    P.gain = a.gain;
    P.wT = ws + L.off_wt;
    P.gpost_prev = a.gpost_prev;
    P.gcomb_prev = a.gcomb_prev;
    P.status = status;
    P.N = static_cast<int>(N);
    P.tt = tt;
    P.d = d;
    P.ntiles = ntiles;
    P.neg_zero = -0.0f;
    P.flags = a.flags;
    e = cudaFuncSetAttribute(bwd_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BSMEM);
    if (e != cudaSuccess) return e;
    bwd_stream_kernel<<<std::min(ntiles, sms), BTHREADS, BSMEM, stream>>>(tx, tf, tgxp, tgy, tgx, tgf, tg, P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    CUtensorMap txp, tgy, tgp;
    if (!bmap_streams_box(&txp, a.Xp, N, d, WT_COLS, WT_TB, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !bmap_rows(&tgy, a.gy, N, d, WT_COLS, WT_TB, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !bmap_rows(&tgp, ws + L.off_gpl, N, 64, 64, WT_TB, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    WtParams W{};
    W.partW = wsf(L.off_partW);
    W.partG = wsf(L.off_partG);
    W.pre_prev = a.pre_prev;
    W.rec = wsf(L.off_rec);
    W.status = status;
    W.N = N;
    W.d = d;
    W.ranges = L.ranges;
    W.per = L.per;
    W.neg_zero = -0.0f;
    const int64_t items = static_cast<int64_t>(d / WT_COLS) * L.ranges;
    e = cudaFuncSetAttribute(bwd_weight_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, WT_SMEM);
    if (e != cudaSuccess) return e;
    bwd_weight_kernel<<<static_cast<int>(std::min<int64_t>(items, sms)), WT_THREADS, WT_SMEM, stream>>>(txp, tgy, tgp, W);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    const int64_t total4 = static_cast<int64_t>(MIXN) * d + d / 4;
    const int blocks = static_cast<int>(std::min<int64_t>((total4 + 255) / 256, 4 * sms)) + 1;
    bwd_reduce_kernel<<<blocks, 256, 0, stream>>>(wsf(L.off_partW), wsf(L.off_partG), wsf(L.off_part0), a.gW,
                                                  a.ggain, a.gbase, a.gscale, d, L.ranges, L.blocks0);
  }
  return cudaGetLastError();
}

}  // namespace mhc

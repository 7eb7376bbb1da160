// small.cu -- the standalone kernels: weight packing, split + Sinkhorn, RMSNorm, and the
// one-op-per-kernel hc_post / hc_pre of the unfused form.
#include <cuda_runtime.h>

#include "hc_arith.cuh"
#include "internal.h"
#include "layout.cuh"
#include "mix_math.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

// Split W fp32 [24, 4d] into three bf16 planes, hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid) (the differences are exact in fp32), and store them as the fused
// kernel's shared-memory image: column block jb (STEP_WDC columns of every stream) is
// [4 streams][80 rows][STEP_WDC columns] with plane pl of mix row r in row packed_row(r, pl),
// rows 72..79 zero, and the 16-byte chunks of each row swizzled as the tensor cores read them.
// One thread per 8 weights (a 16-byte chunk of each plane): it reads them once and writes all
// three planes; the threads past those write the zero rows.
__global__ void pack_kernel(const float* __restrict__ W, uint8_t* __restrict__ P, int d) {
  const int64_t K = 4 * static_cast<int64_t>(d);
  const int64_t nblocks = d / STEP_WDC;
  constexpr int MIXR = STEP_WROWS / 3;                          // 24 mix rows
  constexpr int PADR = STEP_MMA_N - STEP_WROWS;                 // 8 zero rows
  const int64_t main_items = nblocks * 4 * MIXR * STEP_WCHUNKS;
  const int64_t total = main_items + nblocks * 4 * PADR * STEP_WCHUNKS;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (idx < main_items) {
      // consecutive threads: the chunks of one row, then the rows (mix numbers), so a warp reads
      // 8 rows x 128 contiguous bytes of W
      const int chunk = static_cast<int>(idx % STEP_WCHUNKS);
      const int r = static_cast<int>((idx / STEP_WCHUNKS) % MIXR);
      const int k = static_cast<int>((idx / (STEP_WCHUNKS * MIXR)) % 4);
      const int64_t jb = idx / (STEP_WCHUNKS * MIXR * 4);
      const int64_t col = k * static_cast<int64_t>(d) + jb * STEP_WDC + chunk * 8;
      const float4* src = reinterpret_cast<const float4*>(W + r * K + col);
      const float4 a = src[0], b = src[1];
      const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t planes[3][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t hv[2], mv[2], lv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float x = w[2 * e + h];
          const __nv_bfloat16 hi = __float2bfloat16_rn(x);
          const float rem1 = x - __bfloat162float(hi);
          const __nv_bfloat16 mid = __float2bfloat16_rn(rem1);
          const __nv_bfloat16 lo = __float2bfloat16_rn(rem1 - __bfloat162float(mid));
          hv[h] = __bfloat16_as_ushort(hi);
          mv[h] = __bfloat16_as_ushort(mid);
          lv[h] = __bfloat16_as_ushort(lo);
        }
        planes[0][e] = hv[0] | (hv[1] << 16);
        planes[1][e] = mv[0] | (mv[1] << 16);
        planes[2][e] = lv[0] | (lv[1] << 16);
      }
      uint8_t* blk = P + jb * STEP_WBLOCK_BYTES + k * STEP_WSTREAM_BYTES;
#pragma unroll
      for (int pl = 0; pl < 3; ++pl)
        *reinterpret_cast<uint4*>(blk + wtile_chunk_offset(packed_row(r, pl), chunk)) =
            make_uint4(planes[pl][0], planes[pl][1], planes[pl][2], planes[pl][3]);
    } else {
      const int64_t q = idx - main_items;
      const int chunk = static_cast<int>(q % STEP_WCHUNKS);
      const int row = STEP_WROWS + static_cast<int>((q / STEP_WCHUNKS) % PADR);
      const int k = static_cast<int>((q / (STEP_WCHUNKS * PADR)) % 4);
      const int64_t jb = q / (STEP_WCHUNKS * PADR * 4);
      *reinterpret_cast<uint4*>(P + jb * STEP_WBLOCK_BYTES + k * STEP_WSTREAM_BYTES +
                                wtile_chunk_offset(row, chunk)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// One thread per token (Stream weights for the feed-forward, Code: hc_split_sinkhorn kernel).
__global__ void sinkhorn_kernel(const float* __restrict__ mixes, const float* __restrict__ scale,
                                const float* __restrict__ base, float* __restrict__ pre,
                                float* __restrict__ post, float* __restrict__ comb, int64_t N,
                                int iters, float eps) {
  const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (t >= N) return;
  float m[24];
  const float4* src = reinterpret_cast<const float4*>(mixes + t * 24);
#pragma unroll
  for (int r = 0; r < 6; ++r) {
    const float4 v = __ldg(src + r);
    m[4 * r] = v.x;
    m[4 * r + 1] = v.y;
    m[4 * r + 2] = v.z;
    m[4 * r + 3] = v.w;
  }
  float p[4], u[4], c[16];
  split_sinkhorn(m, __ldg(scale), __ldg(scale + 1), __ldg(scale + 2), base, iters, eps, p, u, c);
  reinterpret_cast<float4*>(pre)[t] = make_float4(p[0], p[1], p[2], p[3]);
  reinterpret_cast<float4*>(post)[t] = make_float4(u[0], u[1], u[2], u[3]);
  float4* co = reinterpret_cast<float4*>(comb + t * 16);
#pragma unroll
  for (int r = 0; r < 4; ++r) co[r] = make_float4(c[4 * r], c[4 * r + 1], c[4 * r + 2], c[4 * r + 3]);
}

__device__ __forceinline__ float block_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) scratch[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += scratch[i];
  __syncthreads();
  return t;
}

// One block per row (MoE RMSNorm, Code: RMSNorm): sum of squares in fp32, then
// y = bf16(gain * (x * rsqrt(mean + eps))).
__global__ void rmsnorm_kernel(const uint4* __restrict__ x, const float* __restrict__ gain,
                               uint4* __restrict__ y, int64_t N, int d, float eps) {
  __shared__ float scratch[32];
  const int chunks = d / 8;
  for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
    const uint4* xr = x + row * chunks;
    f2 acc{0.f, 0.f};
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      const uint4 v = xr[c];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const f2 a = bf2_to_f2(w[e]);
        acc = fma2(a, a, acc);
      }
    }
    const float ss = block_sum(acc.x + acc.y, scratch);
    const float r = rsqrtf(__fdiv_rn(ss, static_cast<float>(d)) + eps);
    const f2 r2{r, r};
    uint4* yr = y + row * chunks;
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      const uint4 v = xr[c];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(gain) + 2 * c);
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(gain) + 2 * c + 1);
      const f2 gp[4] = {f2{g0.x, g0.y}, f2{g0.z, g0.w}, f2{g1.x, g1.y}, f2{g1.z, g1.w}};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = f2_to_bf2(mul2(gp[e], mul2(bf2_to_f2(w[e]), r2)));
      yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// The same RMSNorm with the row held in registers between the sum of squares and the scaling
// (one read of the row, not two) and 128-thread CTAs, so that more rows are in flight per SM:
// for rows of at most RMS_MAXC * 8 * RMS_THREADS columns.
constexpr int RMS_THREADS = 128;
constexpr int RMS_MAXC = 8;   // 16-byte chunks per thread: d <= 8192
__global__ void __launch_bounds__(RMS_THREADS) rmsnorm_row_kernel(const uint4* __restrict__ x,
                                                                 const float* __restrict__ gain,
                                                                 uint4* __restrict__ y, int d,
                                                                 float eps) {
  __shared__ float scratch[RMS_THREADS / 32];
  const int chunks = d / 8;
  const uint4* xr = x + static_cast<int64_t>(blockIdx.x) * chunks;
  uint4 v[RMS_MAXC];
  f2 acc{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < RMS_MAXC; ++i) {
    const int c = static_cast<int>(threadIdx.x) + i * RMS_THREADS;
    v[i] = c < chunks ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const f2 a = bf2_to_f2(w[e]);
      acc = fma2(a, a, acc);
    }
  }
  const float ss = block_sum(acc.x + acc.y, scratch);
  const float r = rsqrtf(__fdiv_rn(ss, static_cast<float>(d)) + eps);
  const f2 r2{r, r};
  uint4* yr = y + static_cast<int64_t>(blockIdx.x) * chunks;
#pragma unroll
  for (int i = 0; i < RMS_MAXC; ++i) {
    const int c = static_cast<int>(threadIdx.x) + i * RMS_THREADS;
    if (c >= chunks) break;
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(gain) + 2 * c);
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(gain) + 2 * c + 1);
    const f2 gp[4] = {f2{g0.x, g0.y}, f2{g0.z, g0.w}, f2{g1.x, g1.y}, f2{g1.z, g1.w}};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = f2_to_bf2(mul2(gp[e], mul2(bf2_to_f2(w[e]), r2)));
    yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// hc_post alone: one thread per 8 columns of one token, all 4 streams (the float32 evaluation of
// hc_arith.cuh, as in the fused kernel).
__global__ void hc_post_kernel(const uint4* __restrict__ X, const uint4* __restrict__ F,
                               const float* __restrict__ post, const float* __restrict__ comb,
                               uint4* __restrict__ Xo, int64_t N, int d, int row_dest,
                               float neg_zero) {
  const int chunks = d / 8;
  const int64_t total = N * chunks;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / chunks;
    const int c = static_cast<int>(idx - t * chunks);
    f2 cu[4], cc[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float uk = __ldg(post + t * 4 + k);
      cu[k] = f2{uk, uk};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float v = __ldg(comb + t * 16 + (row_dest ? k * 4 + j : j * 4 + k));
        cc[j][k] = f2{v, v};
      }
    }
    const uint4 fv = F[t * chunks + c];
    uint4 xv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) xv[j] = X[(t * 4 + j) * chunks + c];
    const uint32_t fw[4] = {fv.x, fv.y, fv.z, fv.w};
    uint32_t ow[4][4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const f2 f = bf2_to_f2(fw[w]);
      f2 x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t xw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        x[j] = bf2_to_f2(xw[w]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const f2 ck[4] = {cc[0][k], cc[1][k], cc[2][k], cc[3][k]};
        ow[k][w] = f2_to_bf2(hc_post_pair(ck, cu[k], x, f, f2{neg_zero, neg_zero}));
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) Xo[(t * 4 + k) * chunks + c] = make_uint4(ow[k][0], ow[k][1], ow[k][2], ow[k][3]);
  }
}

// hc_pre alone: y_hat = bf16 of the float32 evaluation of hc_arith.cuh.
__global__ void hc_pre_kernel(const uint4* __restrict__ Xp, const float* __restrict__ pre,
                              uint4* __restrict__ y, int64_t N, int d, float neg_zero) {
  const int chunks = d / 8;
  const int64_t total = N * chunks;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / chunks;
    const int c = static_cast<int>(idx - t * chunks);
    f2 cp[4];
    uint4 xv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float pj = __ldg(pre + t * 4 + j);
      cp[j] = f2{pj, pj};
      xv[j] = Xp[(t * 4 + j) * chunks + c];
    }
    uint32_t o[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      f2 x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t xw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        x[j] = bf2_to_f2(xw[w]);
      }
      o[w] = f2_to_bf2(hc_pre_pair(cp, x, f2{neg_zero, neg_zero}));
    }
    y[t * chunks + c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

int grid_for(int64_t work, int threads) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_pack(const float* W, void* packed, int d, cudaStream_t stream) {
  // one thread per 8 weights of a mix row, plus one per 16-byte chunk of the zero rows
  const int64_t chunks = static_cast<int64_t>(d / STEP_WDC) * 4 *
                         (STEP_WROWS / 3 + STEP_MMA_N - STEP_WROWS) * STEP_WCHUNKS;
  pack_kernel<<<grid_for(chunks, 256), 256, 0, stream>>>(W, static_cast<uint8_t*>(packed), d);
  return cudaGetLastError();
}

cudaError_t launch_sinkhorn(const float* mixes, const float* scale, const float* base, float* pre,
                            float* post, float* comb, int64_t N, int iters, float eps,
                            cudaStream_t stream) {
  const int threads = 128;
  const int64_t blocks = (N + threads - 1) / threads;
  sinkhorn_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(mixes, scale, base, pre,
                                                                         post, comb, N, iters, eps);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* x, const float* gain, void* y, int64_t N, int d, float eps,
                           cudaStream_t stream) {
  if (d / 8 <= RMS_MAXC * RMS_THREADS && N <= 0x7fffffff) {
    rmsnorm_row_kernel<<<static_cast<unsigned>(N), RMS_THREADS, 0, stream>>>(
        static_cast<const uint4*>(x), gain, static_cast<uint4*>(y), d, eps);
    return cudaGetLastError();
  }
  const int threads = 256;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = N < static_cast<int64_t>(sms) * 8 ? N : static_cast<int64_t>(sms) * 8;
  rmsnorm_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(x), gain, static_cast<uint4*>(y), N, d, eps);
  return cudaGetLastError();
}

cudaError_t launch_hc_post(const void* X, const void* F, const float* post, const float* comb,
                           void* X_out, int64_t N, int d, bool row_dest, cudaStream_t stream) {
  const int threads = 256;
  hc_post_kernel<<<grid_for(N * (d / 8), threads), threads, 0, stream>>>(
      static_cast<const uint4*>(X), static_cast<const uint4*>(F), post, comb,
      static_cast<uint4*>(X_out), N, d, row_dest ? 1 : 0, -0.0f);
  return cudaGetLastError();
}

cudaError_t launch_hc_pre(const void* Xp, const float* pre, void* y_hat, int64_t N, int d,
                          cudaStream_t stream) {
  const int threads = 256;
  hc_pre_kernel<<<grid_for(N * (d / 8), threads), threads, 0, stream>>>(
      static_cast<const uint4*>(Xp), pre, static_cast<uint4*>(y_hat), N, d, -0.0f);
  return cudaGetLastError();
}

}  // namespace mhc

// fused.cu -- the single-pass mHC step on sm_103a: one kernel reads X and F once and writes X',
// the normalised sublayer input y and the new mix coefficients (p, u, C).
//
// What it computes: MoE RMSNorm, Code: Block.forward (FFN half) with hc_post, hc_mixes, hc_pre
// from Stream weights for the feed-forward, Code; the single pass is the one that page's "Why"
// section describes (one pass over the streams serves the read and the next weights).
//
// Work decomposition (one thread-block cluster per tile of 128 tokens):
//   * The cluster's `split` CTAs each own a slice of the width d (d/split columns of every
//     stream) for all 128 tokens of the tile. d = 5120 uses 8 CTAs of 640 columns.
//   * Per CTA, a 3-stage TMA ring brings [128 tokens x 32 columns] tiles of X_0..X_3 and F,
//     plus the matching [72 x 32] tiles of the packed projection weights (3 bf16 planes of W).
//   * 8 consumer warps (2 threads per token, 16 columns each) compute hc_post in place in
//     shared memory, its sum of squares, hc_pre and its sum of squares; y_hat goes to TMEM.
//   * One thread issues tcgen05.mma: D[128 tokens x 80] += X'[128 x 32] * Wp[80 x 32]^T per
//     stream, accumulating the three weight planes side by side in TMEM columns 0..71.
//     Another TMA path stores X' straight from the same shared-memory tiles.
//   * Epilogue: the cluster sums the per-slice partial projections and sums of squares through
//     distributed shared memory; each CTA finishes 128/split tokens (scale, split, Sinkhorn) and
//     every CTA normalises its own slice of y_hat from TMEM and stores y with TMA.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "mix_math.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int TT = 128;                 // tokens per tile (MMA M)
constexpr int DC = 32;                  // width columns per pipeline stage (64-byte rows)
constexpr int NSTAGE = 3;               // TMA ring depth
constexpr int WROWS = 72;               // 3 planes x 24 mix rows
constexpr int MMA_N = 80;               // N of the MMA (rows 72..79 of a weight tile unused)
constexpr int NCONS = 8;                // consumer warps (2 per TMEM lane quarter)
constexpr int NROLE = 2;                // warp 0: TMA producer; warp 1: TMEM owner, MMA, X' stores
constexpr int NTHREADS = (NROLE + NCONS) * 32;
constexpr int TILE_BYTES = TT * DC * 2;           // 8192
constexpr int WTILE_BYTES = MMA_N * DC * 2;       // 5120
constexpr int STAGE_BYTES = 5 * TILE_BYTES + 4 * WTILE_BYTES;
constexpr int PART_STRIDE = 32;                   // floats per token in the cluster partials
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t STASH_COL = 128;
constexpr int MAX_SLICE = 2 * (TMEM_COLS - STASH_COL);   // 768 bf16 per token row
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;        // 2 s
constexpr uint64_t DEBUG_WAIT_NS = 2000000ull;           // 2 ms

constexpr int OFF_PART = NSTAGE * STAGE_BYTES;
constexpr int OFF_RED = OFF_PART + TT * PART_STRIDE * 4;
constexpr int OFF_RY = OFF_RED + 2 * TT * 2 * 4;
constexpr int OFF_BARS = OFF_RY + TT * 4;
constexpr int NBARS = 3 * NSTAGE + 2;
constexpr int OFF_TMEM = OFF_BARS + NBARS * 8;
constexpr int SMEM_BYTES = OFF_TMEM + 16 + 1024;   // + slack for 1 KB alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");

__host__ __device__ constexpr int xtile(int b, int k) { return b * STAGE_BYTES + k * TILE_BYTES; }
__host__ __device__ constexpr int ftile(int b) { return b * STAGE_BYTES + 4 * TILE_BYTES; }
__host__ __device__ constexpr int wtile(int b, int k) {
  return b * STAGE_BYTES + 5 * TILE_BYTES + k * WTILE_BYTES;
}
// y staging reuses the X/F tiles of the idle ring: slot j -> stage j/5, tile j%5.
__host__ __device__ constexpr int yslot(int j) { return (j / 5) * STAGE_BYTES + (j % 5) * TILE_BYTES; }
constexpr int NYSLOTS = 5 * NSTAGE;

struct StepParams {
  const float* pre_prev;
  const float* post_prev;
  const float* comb_prev;
  const float* scale;
  const float* base;
  const float* gain;
  float* pre_out;
  float* post_out;
  float* comb_out;
  float* mixes_out;
  unsigned* status;
  int N;
  int d;
  int split;
  int slice;
  int nsteps;
  int iters;
  float hc_eps;
  float norm_eps;
  unsigned flags;
};

template <bool FUSED>
__global__ void __launch_bounds__(NTHREADS, 1)
    step_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_f,
                const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_xo,
                const __grid_constant__ CUtensorMap tm_y, const StepParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + OFF_BARS);
  uint64_t* empty = full + NSTAGE;
  uint64_t* xready = empty + NSTAGE;
  uint64_t* accfull = xready + NSTAGE;
  uint64_t* never = accfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM);
  float* part = reinterpret_cast<float*>(sm + OFF_PART);
  float* red = reinterpret_cast<float*>(sm + OFF_RED);
  float* ry = reinterpret_cast<float*>(sm + OFF_RY);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t g = cluster_ctarank();
  const int t0 = blockIdx.y * TT;
  const int i_base = static_cast<int>(g) * P.slice;
  const int S = P.nsteps;
  const int d = P.d;
  bool timed_out = false;

  if (threadIdx.x == 0) {
    for (int b = 0; b < NSTAGE; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], FUSED ? 2 : 1 + NCONS);
      mbar_init(&xready[b], NCONS);
    }
    mbar_init(accfull, 1);
    mbar_init(never, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
      if (FUSED) {
        tma_prefetch_desc(&tm_f);
        tma_prefetch_desc(&tm_xo);
        tma_prefetch_desc(&tm_y);
      }
      const uint32_t bytes = 4 * TILE_BYTES + (FUSED ? TILE_BYTES : 0) + 4 * WROWS * DC * 2;
      for (int s = 0; s < S; ++s) {
        const int b = s % NSTAGE;
        if (s >= NSTAGE) {
          const uint32_t par = ((s / NSTAGE) - 1) & 1;
          if (!mbar_wait(&empty[b], par, timed_out ? 0 : WAIT_LIMIT_NS)) timed_out = true;
        }
        const int i0 = i_base + s * DC;
        mbar_arrive_expect_tx(&full[b], bytes);
#pragma unroll
        for (int k = 0; k < 4; ++k) tma_load_3d(sm + xtile(b, k), &tm_x, &full[b], i0, k, t0);
        if (FUSED) tma_load_2d(sm + ftile(b), &tm_f, &full[b], i0, t0);
#pragma unroll
        for (int k = 0; k < 4; ++k) tma_load_2d(sm + wtile(b, k), &tm_w, &full[b], k * d + i0, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA + X' store issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(TT, MMA_N);
      for (int s = 0; s < S; ++s) {
        const int b = s % NSTAGE;
        const uint32_t par = (s / NSTAGE) & 1;
        if (!mbar_wait(FUSED ? &xready[b] : &full[b], par, timed_out ? 0 : WAIT_LIMIT_NS))
          timed_out = true;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a0 = smem_u32(sm + xtile(b, k));
          const uint32_t b0 = smem_u32(sm + wtile(b, k));
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            umma_bf16(tmem + ACC_COL, sdesc_kmajor_sw64(a0 + kk * 32), sdesc_kmajor_sw64(b0 + kk * 32),
                      idesc, (s | k | kk) != 0);
          }
        }
        umma_commit(&empty[b]);
        if (FUSED) {
          const int i0 = i_base + s * DC;
#pragma unroll
          for (int k = 0; k < 4; ++k) tma_store_3d(&tm_xo, sm + xtile(b, k), i0, k, t0);
          bulk_commit();
          bulk_wait_read<0>();  // this stage's X' has left shared memory
          mbar_arrive(&empty[b]);
        }
      }
      umma_commit(accfull);
    }
  } else {
    // ------------------------------------------------------------------ consumers
    const int c = warp - NROLE;
    const int sub = warp & 3;           // TMEM lane quarter this warp may access
    const int h = c >> 2;               // which half (16 columns) of the stage's 32 columns
    const int tl = sub * 32 + lane;     // token row within the tile
    const int token = t0 + tl;
    const bool valid = token < P.N;
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    // 64-byte swizzle: 16-byte chunk q of row r sits at chunk q ^ ((r >> 1) & 3)
    const uint32_t row_off0 = tl * 64 + (((2 * h) ^ ((tl >> 1) & 3)) << 4);
    const uint32_t row_off1 = tl * 64 + (((2 * h + 1) ^ ((tl >> 1) & 3)) << 4);

    f2 cu[4], cc[4][4], cp[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cu[k] = f2{0.f, 0.f};
      cp[k] = f2{0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) cc[j][k] = f2{0.f, 0.f};
    }
    if (FUSED && valid) {
      const bool row_dest = (P.flags & 1u) != 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float uk = __ldg(P.post_prev + static_cast<size_t>(token) * 4 + k);
        const float pk = __ldg(P.pre_prev + static_cast<size_t>(token) * 4 + k);
        cu[k] = f2{uk, uk};
        cp[k] = f2{pk, pk};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // cc[j][k]: coefficient of input stream j in output stream k
          const int idx = row_dest ? (k * 4 + j) : (j * 4 + k);
          const float v = __ldg(P.comb_prev + static_cast<size_t>(token) * 16 + idx);
          cc[j][k] = f2{v, v};
        }
      }
    }

    f2 sx2{0.f, 0.f}, sy2{0.f, 0.f};
    for (int s = 0; s < S; ++s) {
      const int b = s % NSTAGE;
      const uint32_t par = (s / NSTAGE) & 1;
      if (!mbar_wait(&full[b], par, timed_out ? 0 : WAIT_LIMIT_NS)) timed_out = true;
      if (FUSED) {
        uint32_t yw[8];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t ro = half ? row_off1 : row_off0;
          uint32_t xw[4][4], fw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(sm + xtile(b, k) + ro);
            xw[k][0] = v.x;
            xw[k][1] = v.y;
            xw[k][2] = v.z;
            xw[k][3] = v.w;
          }
          {
            const uint4 v = *reinterpret_cast<const uint4*>(sm + ftile(b) + ro);
            fw[0] = v.x;
            fw[1] = v.y;
            fw[2] = v.z;
            fw[3] = v.w;
          }
          uint32_t ow[4][4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const f2 f = bf2_to_f2(fw[w]);
            f2 x[4], xp[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = bf2_to_f2(xw[j][w]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // X'_k = fma(u_k, F, fma(C_3k, X_3, fma(C_2k, X_2, fma(C_1k, X_1, C_0k X_0))))
              f2 mixed = mul2(cc[0][k], x[0]);
              mixed = fma2(cc[1][k], x[1], mixed);
              mixed = fma2(cc[2][k], x[2], mixed);
              mixed = fma2(cc[3][k], x[3], mixed);
              ow[k][w] = f2_to_bf2(fma2(cu[k], f, mixed));
              xp[k] = bf2_to_f2(ow[k][w]);
              sx2 = fma2(xp[k], xp[k], sx2);
            }
            // y_hat = fma(p_3, X'_3, fma(p_2, X'_2, fma(p_1, X'_1, p_0 X'_0)))
            f2 yh = mul2(cp[0], xp[0]);
            yh = fma2(cp[1], xp[1], yh);
            yh = fma2(cp[2], xp[2], yh);
            yh = fma2(cp[3], xp[3], yh);
            yw[half * 4 + w] = f2_to_bf2(yh);
            const f2 yr = bf2_to_f2(yw[half * 4 + w]);
            sy2 = fma2(yr, yr, sy2);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(sm + xtile(b, k) + ro) =
                make_uint4(ow[k][0], ow[k][1], ow[k][2], ow[k][3]);
        }
        tmem_st_x8(tmem + lane_base + STASH_COL + static_cast<uint32_t>(h * S * 8 + s * 8), yw);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&xready[b]);
      } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t ro = half ? row_off1 : row_off0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(sm + xtile(b, k) + ro);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const f2 x = bf2_to_f2(wv[w]);
              sx2 = fma2(x, x, sx2);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
      }
    }
    if (FUSED) tmem_wait_st();

    // ---------------------------------------------------------------- partials of this slice
    red[(h * TT + tl) * 2 + 0] = sx2.x + sx2.y;
    red[(h * TT + tl) * 2 + 1] = sy2.x + sy2.y;
    named_bar_sync(1, NCONS * 32);
    if (h == 0) {
      if (!mbar_wait(accfull, 0, timed_out ? 0 : WAIT_LIMIT_NS)) timed_out = true;
      tc_fence_after();
      float acc[24];
#pragma unroll
      for (int r = 0; r < 24; ++r) acc[r] = 0.f;
#pragma unroll
      for (int pl = 2; pl >= 0; --pl) {   // smallest plane first
#pragma unroll
        for (int c8 = 0; c8 < 3; ++c8) {
          uint32_t v[8];
          tmem_ld_x8(tmem + lane_base + ACC_COL + pl * 24 + c8 * 8, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[c8 * 8 + e] += __uint_as_float(v[e]);
        }
      }
      float* pt = part + tl * PART_STRIDE;
#pragma unroll
      for (int r = 0; r < 24; ++r) pt[r] = acc[r];
      pt[24] = red[tl * 2 + 0] + red[(TT + tl) * 2 + 0];
      pt[25] = red[tl * 2 + 1] + red[(TT + tl) * 2 + 1];
    }
  }

  // ------------------------------------------------------------------ cluster reduction
  __syncwarp();
  cluster_sync();

  const int per = TT / P.split;
  if (static_cast<int>(threadIdx.x) < per) {
    // finish tokens [g*per, (g+1)*per) of the tile: scale, split, Sinkhorn
    const int tl2 = static_cast<int>(g) * per + threadIdx.x;
    const int token2 = t0 + tl2;
    float acc[24];
    float sx = 0.f;
#pragma unroll
    for (int r = 0; r < 24; ++r) acc[r] = 0.f;
    const uint32_t local = smem_u32(part + tl2 * PART_STRIDE);
    for (int rk = 0; rk < P.split; ++rk) {
      const uint32_t ra = map_cluster(local, rk);
#pragma unroll
      for (int r = 0; r < 24; ++r) acc[r] += ld_cluster_f32(ra + 4 * r);
      sx += ld_cluster_f32(ra + 4 * 24);
    }
    if (token2 < P.N) {
      const float rs = rsqrtf(__fdiv_rn(sx, static_cast<float>(4 * d)) + P.norm_eps);
      float m[24];
#pragma unroll
      for (int r = 0; r < 24; ++r) m[r] = acc[r] * rs;
      if (P.mixes_out != nullptr) {
        float4* mo = reinterpret_cast<float4*>(P.mixes_out + static_cast<size_t>(token2) * 24);
#pragma unroll
        for (int r = 0; r < 6; ++r) mo[r] = make_float4(m[4 * r], m[4 * r + 1], m[4 * r + 2], m[4 * r + 3]);
      }
      float pp[4], uu[4], cm[16];
      split_sinkhorn(m, __ldg(P.scale), __ldg(P.scale + 1), __ldg(P.scale + 2), P.base, P.iters,
                     P.hc_eps, pp, uu, cm);
      reinterpret_cast<float4*>(P.pre_out)[token2] = make_float4(pp[0], pp[1], pp[2], pp[3]);
      reinterpret_cast<float4*>(P.post_out)[token2] = make_float4(uu[0], uu[1], uu[2], uu[3]);
      float4* co = reinterpret_cast<float4*>(P.comb_out + static_cast<size_t>(token2) * 16);
#pragma unroll
      for (int r = 0; r < 4; ++r) co[r] = make_float4(cm[4 * r], cm[4 * r + 1], cm[4 * r + 2], cm[4 * r + 3]);
    }
  }

  if (FUSED && warp >= NROLE) {
    // ---------------------------------------------------------------- RMSNorm of this slice
    const int c = warp - NROLE;
    const int sub = warp & 3;
    const int h = c >> 2;
    const int tl = sub * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t row_off0 = tl * 64 + (((2 * h) ^ ((tl >> 1) & 3)) << 4);
    const uint32_t row_off1 = tl * 64 + (((2 * h + 1) ^ ((tl >> 1) & 3)) << 4);
    if (h == 0) {
      float sy = 0.f;
      const uint32_t local = smem_u32(part + tl * PART_STRIDE + 25);
      for (int rk = 0; rk < P.split; ++rk) sy += ld_cluster_f32(map_cluster(local, rk));
      ry[tl] = rsqrtf(__fdiv_rn(sy, static_cast<float>(d)) + P.norm_eps);
    }
    named_bar_sync(1, NCONS * 32);
    const float r = ry[tl];
    const f2 r2{r, r};
    for (int s0 = 0; s0 < S; s0 += NYSLOTS) {
      const int s1 = min(S, s0 + NYSLOTS);
      for (int s = s0; s < s1; ++s) {
        uint32_t w[8];
        tmem_ld_x8(tmem + lane_base + STASH_COL + static_cast<uint32_t>(h * S * 8 + s * 8), w);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int i = i_base + s * DC + (2 * h + half) * 8;
          const float4 g0 = __ldg(reinterpret_cast<const float4*>(P.gain + i));
          const float4 g1 = __ldg(reinterpret_cast<const float4*>(P.gain + i + 4));
          const f2 gp[4] = {f2{g0.x, g0.y}, f2{g0.z, g0.w}, f2{g1.x, g1.y}, f2{g1.z, g1.w}};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] = f2_to_bf2(mul2(gp[e], mul2(bf2_to_f2(w[half * 4 + e]), r2)));
          *reinterpret_cast<uint4*>(sm + yslot(s - s0) + (half ? row_off1 : row_off0)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, NCONS * 32);
      if (warp == NROLE && lane == 0) {
        for (int s = s0; s < s1; ++s) tma_store_2d(&tm_y, sm + yslot(s - s0), i_base + s * DC, t0);
        bulk_commit();
        bulk_wait<0>();
      }
      named_bar_sync(1, NCONS * 32);
    }
  }

  if ((P.flags & 2u) != 0 && threadIdx.x == 0) {
    if (!mbar_wait(never, 0, DEBUG_WAIT_NS)) timed_out = true;
  }
  if (timed_out) atomicOr(P.status, STATUS_TIMEOUT);

  // ------------------------------------------------------------------ leave together
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool map_streams(CUtensorMap* m, const void* p, int64_t N, int d) {   // [N, 4, d]
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), 4, static_cast<cuuint64_t>(N)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 8};
  const cuuint32_t box[3] = {DC, 1, TT};
  return make_map(m, p, 3, dims, str, box);
}
bool map_rows(CUtensorMap* m, const void* p, int64_t rows, int64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t str[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {DC, box_rows};
  return make_map(m, p, 2, dims, str, box);
}

}  // namespace

int choose_split(int d, int forced) {
  auto ok = [d](int s) { return d > 0 && d % (DC * s) == 0 && d / s <= MAX_SLICE; };
  if (forced != 0) return (forced == 1 || forced == 2 || forced == 4 || forced == 8) && ok(forced) ? forced : 0;
  for (int s : {1, 2, 4, 8})
    if (ok(s)) return s;
  return 0;
}

cudaError_t launch_step(bool fused, const StepArgs& a, cudaStream_t stream) {
  const int K = 4 * a.d;
  CUtensorMap tx, tf, tw, txo, ty;
  if (!map_streams(&tx, a.X, a.N, a.d)) return cudaErrorInvalidValue;
  if (!map_rows(&tw, a.W_packed, WROWS, K, WROWS)) return cudaErrorInvalidValue;
  if (fused) {
    if (!map_rows(&tf, a.F, a.N, a.d, TT)) return cudaErrorInvalidValue;
    if (!map_streams(&txo, a.X_out, a.N, a.d)) return cudaErrorInvalidValue;
    if (!map_rows(&ty, a.y_out, a.N, a.d, TT)) return cudaErrorInvalidValue;
  } else {
    tf = tx;
    txo = tx;
    ty = tx;
  }
  StepParams P{};
  P.pre_prev = a.pre_prev;
  P.post_prev = a.post_prev;
  P.comb_prev = a.comb_prev;
  P.scale = a.scale;
  P.base = a.base;
  P.gain = a.gain;
  P.pre_out = a.pre_out;
  P.post_out = a.post_out;
  P.comb_out = a.comb_out;
  P.mixes_out = a.mixes_out;
  P.status = status_word();
  if (P.status == nullptr) return cudaErrorInvalidDevice;
  P.N = static_cast<int>(a.N);
  P.d = a.d;
  P.split = a.split;
  P.slice = a.d / a.split;
  P.nsteps = P.slice / DC;
  P.iters = a.iters;
  P.hc_eps = a.hc_eps;
  P.norm_eps = a.norm_eps;
  P.flags = a.flags;

  auto kern = fused ? step_kernel<true> : step_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int tiles = static_cast<int>((a.N + TT - 1) / TT);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.split, tiles, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tx, tf, tw, txo, ty, P);
}

cudaError_t step_occupancy(int split, int* clusters) {
  auto kern = step_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, 1024, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, kern, &cfg);
}

}  // namespace mhc

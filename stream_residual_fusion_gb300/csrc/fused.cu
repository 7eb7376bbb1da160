// fused.cu -- the single-pass mHC step on sm_103a: one kernel reads X and F once and writes X',
// the normalised sublayer input y and the new mix coefficients (p, u, C).
//
// What it computes: MoE RMSNorm, Code: Block.forward (FFN half) with hc_post, hc_mixes, hc_pre
// from Stream weights for the feed-forward, Code; the single pass is the one that page's "Why"
// section describes (one pass over the streams serves the read and the next weights).
//
// Work decomposition (one thread-block cluster per tile of 128 tokens):
//   * The cluster's `split` CTAs each own a slice of the width d (d/split columns of every
//     stream) for all 128 tokens of the tile; d = 5120 uses 8 CTAs of 640 columns. The slices
//     interleave in steps of 16 columns, so at any stage the cluster reads one contiguous run of
//     16*split columns of each token row (one DRAM burst instead of split scattered pieces).
//   * Per CTA, a 6-stage TMA ring brings [128 tokens x 16 columns] tiles of X_0..X_3 and F,
//     plus the matching [72 x 16] tiles of the packed projection weights (3 bf16 planes of W).
//   * 8 consumer warps (2 threads per token, 8 columns each) compute hc_post in place in
//     shared memory, its sum of squares, hc_pre and its sum of squares; y_hat goes to TMEM.
//   * One thread issues tcgen05.mma: D[128 tokens x 80] += X'[128 x 16] * Wp[80 x 16]^T per
//     stream. Groups of PG stages accumulate into one of two TMEM accumulators; the consumers
//     fold each finished group into float32 running sums in shared memory, so no tensor-core
//     accumulation chain is longer than 4*PG MMAs.
//   * X' leaves through TMA stores straight from the shared-memory tiles it was computed in.
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
constexpr int DC = 16;                  // width columns per pipeline stage (32-byte rows)
constexpr int NSTAGE = 6;               // TMA ring depth
constexpr int WROWS = 72;               // 3 planes x 24 mix rows
constexpr int MMA_N = 80;               // N of the MMA (rows 72..79 of a weight tile unused)
constexpr int NCONS = 8;                // consumer warps (2 per TMEM lane quarter)
constexpr int NROLE = 2;                // warp 0: TMA producer; warp 1: TMEM owner, MMA, X' stores
constexpr int NTHREADS = (NROLE + NCONS) * 32;
constexpr int PG = 4;                   // stages per tensor-core accumulation group (16 MMAs)
constexpr int STORE_LAG = 2;            // X' store groups left in flight before a stage is freed
constexpr int TILE_BYTES = TT * DC * 2;           // 4096
constexpr int WTILE_BYTES = MMA_N * DC * 2;       // 2560
constexpr int STAGE_BYTES = 5 * TILE_BYTES + 4 * WTILE_BYTES;   // 30720
constexpr int PART_STRIDE = 28;                   // floats per token row of the running sums
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = MMA_N;              // two accumulators, at columns 0 and 80
constexpr uint32_t STASH_COL = 2 * ACC_COLS;
constexpr int MAX_SLICE = 2 * (TMEM_COLS - STASH_COL);   // 704 bf16 of y_hat per token row
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;        // 2 s
constexpr uint64_t DEBUG_WAIT_NS = 2000000ull;           // 2 ms

constexpr int OFF_PART = NSTAGE * STAGE_BYTES;
constexpr int OFF_RED = OFF_PART + TT * PART_STRIDE * 4;
constexpr int OFF_RY = OFF_RED + 2 * TT * 2 * 4;
constexpr int OFF_BARS = OFF_RY + TT * 4;
constexpr int NBARS = 3 * NSTAGE + 4;   // full, empty, xready per stage; accready[2], accfull, never
constexpr int OFF_TMEM = OFF_BARS + NBARS * 8;
constexpr int SMEM_BYTES = OFF_TMEM + 16 + 1024;   // + slack for 1 KB alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
static_assert(PG >= 2, "a group is folded one stage into the next group");

__host__ __device__ constexpr int xtile(int b, int k) { return b * STAGE_BYTES + k * TILE_BYTES; }
__host__ __device__ constexpr int ftile(int b) { return b * STAGE_BYTES + 4 * TILE_BYTES; }
__host__ __device__ constexpr int wtile(int b, int k) {
  return b * STAGE_BYTES + 5 * TILE_BYTES + k * WTILE_BYTES;
}
// y staging reuses the X/F tiles of the idle ring: slot j -> stage j/5, tile j%5.
__host__ __device__ constexpr int yslot(int j) { return (j / 5) * STAGE_BYTES + (j % 5) * TILE_BYTES; }
constexpr int NYSLOTS = 5 * NSTAGE;

// 32-byte swizzle: 16-byte chunk q of row r sits at chunk q ^ ((r >> 2) & 1).
__device__ __forceinline__ uint32_t sw32_offset(int row, int chunk) {
  return static_cast<uint32_t>(row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4));
}

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
  unsigned long long* trace;   // optional: 8 phase timestamps per CTA (mhc_set_trace)
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

// Fold accumulation group `grp` (TMEM accumulator grp & 1) into this thread's 12 running sums.
// The packed weight rows are ordered so that half h of the 24 mix numbers, all three planes,
// lands in accumulator columns [36h, 36h + 36): 12 hi, then 12 mid, then 12 lo.
__device__ __forceinline__ void fold_group(uint32_t tmem_lane, int grp, int h, float* run) {
  const uint32_t col = static_cast<uint32_t>((grp & 1) * ACC_COLS + 36 * h);
  uint32_t a[32], b[4];
  tmem_ld_x32(tmem_lane + col, a);
  tmem_ld_x4(tmem_lane + col + 32, b);
  float lo[12];
#pragma unroll
  for (int r = 0; r < 8; ++r) lo[r] = __uint_as_float(a[24 + r]);
#pragma unroll
  for (int r = 0; r < 4; ++r) lo[8 + r] = __uint_as_float(b[r]);
  float4* rp = reinterpret_cast<float4*>(run);
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    float4 v = rp[q];
    float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = 4 * q + e;
      vv[e] += (lo[r] + __uint_as_float(a[12 + r])) + __uint_as_float(a[r]);
    }
    rp[q] = make_float4(vv[0], vv[1], vv[2], vv[3]);
  }
}

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
  uint64_t* accready = xready + NSTAGE;     // [2]: an accumulation group finished in buffer i
  uint64_t* accfull = accready + 2;
  uint64_t* never = accfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM);
  float* part = reinterpret_cast<float*>(sm + OFF_PART);
  float* red = reinterpret_cast<float*>(sm + OFF_RED);
  float* ry = reinterpret_cast<float*>(sm + OFF_RY);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t g = cluster_ctarank();
  const int t0 = blockIdx.y * TT;
  const int col0 = static_cast<int>(g) * DC;          // first column of this CTA's slice
  const int cstride = DC * P.split;                   // stride between its stages' columns
  const int S = P.nsteps;
  const int ngroups = (S + PG - 1) / PG;
  // groups folded inside the main loop: group q is folded after stage (q+1)*PG + 1
  const int nfold_loop = S >= 2 ? (S - 2) / PG : 0;
  const int d = P.d;
  bool timed_out = false;
  // optional phase trace: [cta][0..7] = start, loads issued, main loop done, partials ready,
  // cluster reduced, mix numbers written, y written, end; slot 7 also carries the SM id.
  unsigned long long* tr = P.trace == nullptr
                               ? nullptr
                               : P.trace + 8ull * (static_cast<unsigned long long>(blockIdx.y) * gridDim.x + blockIdx.x);
  const unsigned long long t_start = global_timer_ns();
  auto stamp = [&](int k) {   // slot 0: absolute start; slots 1..7: ns since this CTA started
    if (tr != nullptr) tr[k] = k == 0 ? t_start : global_timer_ns() - t_start;
  };
  if (threadIdx.x == 0) stamp(0);

  if (threadIdx.x == 0) {
    for (int b = 0; b < NSTAGE; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], FUSED ? 2 : 1 + NCONS);
      mbar_init(&xready[b], NCONS);
    }
    mbar_init(&accready[0], 1);
    mbar_init(&accready[1], 1);
    mbar_init(accfull, 1);
    mbar_init(never, 1);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < TT * PART_STRIDE; i += NTHREADS) part[i] = 0.f;
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
      const uint64_t stream_pol = policy_evict_first();
      const uint64_t weight_pol = policy_evict_last();
      const uint32_t bytes = 4 * TILE_BYTES + (FUSED ? TILE_BYTES : 0) + 4 * WROWS * DC * 2;
      for (int s = 0; s < S; ++s) {
        const int b = s % NSTAGE;
        if (s >= NSTAGE) {
          const uint32_t par = ((s / NSTAGE) - 1) & 1;
          if (!mbar_wait(&empty[b], par, timed_out ? 0 : WAIT_LIMIT_NS)) timed_out = true;
        }
        const int i0 = col0 + s * cstride;
        mbar_arrive_expect_tx(&full[b], bytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tma_load_3d_hint(sm + xtile(b, k), &tm_x, &full[b], i0, k, t0, stream_pol);
        if (FUSED) tma_load_2d_hint(sm + ftile(b), &tm_f, &full[b], i0, t0, stream_pol);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tma_load_2d_hint(sm + wtile(b, k), &tm_w, &full[b], k * d + i0, 0, weight_pol);
      }
      stamp(1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA + X' store issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(TT, MMA_N);
      const uint64_t stream_pol = policy_evict_first();
      for (int s = 0; s < S; ++s) {
        const int b = s % NSTAGE;
        const uint32_t par = (s / NSTAGE) & 1;
        if (!mbar_wait(FUSED ? &xready[b] : &full[b], par, timed_out ? 0 : WAIT_LIMIT_NS))
          timed_out = true;
        tc_fence_after();
        const int grp = s / PG;
        const uint32_t acc = tmem + static_cast<uint32_t>((grp & 1) * ACC_COLS);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          umma_bf16(acc, sdesc_kmajor_sw32(smem_u32(sm + xtile(b, k))),
                    sdesc_kmajor_sw32(smem_u32(sm + wtile(b, k))), idesc,
                    (s % PG != 0 || k != 0) ? 1u : 0u);
        }
        umma_commit(&empty[b]);
        if (s % PG == PG - 1 || s == S - 1) umma_commit(&accready[grp & 1]);
        if (FUSED) {
          const int i0 = col0 + s * cstride;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tma_store_3d_hint(&tm_xo, sm + xtile(b, k), i0, k, t0, stream_pol);
          bulk_commit();
          // release the stage whose X' store is STORE_LAG groups old, without waiting for this one
          bulk_wait_read<STORE_LAG>();
          if (s >= STORE_LAG) mbar_arrive(&empty[(s - STORE_LAG) % NSTAGE]);
        }
      }
      umma_commit(accfull);
      if (FUSED) bulk_wait_read<0>();
    }
  } else {
    // ------------------------------------------------------------------ consumers
    const int c = warp - NROLE;
    const int sub = warp & 3;           // TMEM lane quarter this warp may access
    const int h = c >> 2;               // which 8 of the stage's 16 columns, which 12 mix numbers
    const int tl = sub * 32 + lane;     // token row within the tile
    const int token = t0 + tl;
    const bool valid = token < P.N;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const uint32_t row_off = sw32_offset(tl, h);
    float* run = part + tl * PART_STRIDE + 12 * h;

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
      uint32_t xw[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 v = *reinterpret_cast<const uint4*>(sm + xtile(b, k) + row_off);
        xw[k][0] = v.x;
        xw[k][1] = v.y;
        xw[k][2] = v.z;
        xw[k][3] = v.w;
      }
      f2 lx{0.f, 0.f};   // this stage's sum of squares, added to the running sum once
      if (FUSED) {
        uint32_t fw[4];
        {
          const uint4 v = *reinterpret_cast<const uint4*>(sm + ftile(b) + row_off);
          fw[0] = v.x;
          fw[1] = v.y;
          fw[2] = v.z;
          fw[3] = v.w;
        }
        uint32_t ow[4][4], yw[4];
        f2 ly{0.f, 0.f};
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
            lx = fma2(xp[k], xp[k], lx);
          }
          // y_hat = fma(p_3, X'_3, fma(p_2, X'_2, fma(p_1, X'_1, p_0 X'_0)))
          f2 yh = mul2(cp[0], xp[0]);
          yh = fma2(cp[1], xp[1], yh);
          yh = fma2(cp[2], xp[2], yh);
          yh = fma2(cp[3], xp[3], yh);
          yw[w] = f2_to_bf2(yh);
          const f2 yr = bf2_to_f2(yw[w]);
          ly = fma2(yr, yr, ly);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(sm + xtile(b, k) + row_off) =
              make_uint4(ow[k][0], ow[k][1], ow[k][2], ow[k][3]);
        tmem_st_x4(lane_base + STASH_COL + static_cast<uint32_t>(h * S * 4 + s * 4), yw[0], yw[1],
                   yw[2], yw[3]);
        sy2 = add2(sy2, ly);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&xready[b]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const f2 x = bf2_to_f2(xw[k][w]);
            lx = fma2(x, x, lx);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
      }
      sx2 = add2(sx2, lx);
      // Fold group q one stage into group q+1; the MMA that reuses q's accumulator (group q+2)
      // starts only after this warp's xready of a later stage.
      if (s % PG == 1 && s >= PG) {
        const int grp = s / PG - 1;
        if (!mbar_wait(&accready[grp & 1], (grp >> 1) & 1, timed_out ? 0 : WAIT_LIMIT_NS))
          timed_out = true;
        tc_fence_after();
        fold_group(lane_base, grp, h, run);
      }
    }
    if (FUSED) tmem_wait_st();
    if (warp == NROLE && lane == 0) stamp(2);
    for (int grp = nfold_loop; grp < ngroups; ++grp) {   // groups that ended too late to fold
      if (!mbar_wait(&accready[grp & 1], (grp >> 1) & 1, timed_out ? 0 : WAIT_LIMIT_NS))
        timed_out = true;
      tc_fence_after();
      fold_group(lane_base, grp, h, run);
    }

    // ---------------------------------------------------------------- partials of this slice
    red[(h * TT + tl) * 2 + 0] = sx2.x + sx2.y;
    red[(h * TT + tl) * 2 + 1] = sy2.x + sy2.y;
    named_bar_sync(1, NCONS * 32);
    if (h == 0) {
      float* pt = part + tl * PART_STRIDE;
      pt[24] = red[tl * 2 + 0] + red[(TT + tl) * 2 + 0];
      pt[25] = red[tl * 2 + 1] + red[(TT + tl) * 2 + 1];
    }
    if (!mbar_wait(accfull, 0, timed_out ? 0 : WAIT_LIMIT_NS)) timed_out = true;
    if (warp == NROLE && lane == 0) stamp(3);
  }

  // ------------------------------------------------------------------ cluster reduction
  __syncwarp();
  cluster_sync();
  if (threadIdx.x == 0) stamp(4);

  // Finish tokens [g*per, (g+1)*per) of the tile -- scale, split, Sinkhorn -- four lanes per
  // token (lane j of a group owns comb row j), NTHREADS/4 tokens at a time.
  const int per = TT / P.split;
  // whole warps only (the shuffles span the warp): 64 threads for split 8, all for split 1
  const int nthr = min(NTHREADS, ((4 * per + 31) / 32) * 32);
  for (int base_t = 0; static_cast<int>(threadIdx.x) < nthr && base_t < per; base_t += nthr / 4) {
    const int q = static_cast<int>(threadIdx.x) >> 2;    // token of this lane group
    const int j = static_cast<int>(threadIdx.x) & 3;     // comb row owned by this lane
    const bool in_range = base_t + q < per;
    const int tl2 = static_cast<int>(g) * per + base_t + (in_range ? q : 0);
    const int token2 = t0 + tl2;
    // float4 0 = m[0..3], 1 = m[4..7], 2 + j = logits row j, 6 = (S_x, S_y, -, -)
    float4 a0{0.f, 0.f, 0.f, 0.f}, a1 = a0, a2 = a0, a6 = a0;
    const uint32_t local = smem_u32(part + tl2 * PART_STRIDE);
    for (int rk = 0; rk < P.split; ++rk) {
      const uint32_t ra = map_cluster(local, rk);
      const float4 v0 = ld_cluster_f32x4(ra);
      const float4 v1 = ld_cluster_f32x4(ra + 16);
      const float4 v2 = ld_cluster_f32x4(ra + 16 * (2 + j));
      const float4 v6 = ld_cluster_f32x4(ra + 16 * 6);
      a0.x += v0.x; a0.y += v0.y; a0.z += v0.z; a0.w += v0.w;
      a1.x += v1.x; a1.y += v1.y; a1.z += v1.z; a1.w += v1.w;
      a2.x += v2.x; a2.y += v2.y; a2.z += v2.z; a2.w += v2.w;
      a6.x += v6.x;
    }
    const float rs = __frsqrt_rn(__fdiv_rn(a6.x, static_cast<float>(4 * d)) + P.norm_eps);
    const float m0[4] = {a0.x * rs, a0.y * rs, a0.z * rs, a0.w * rs};
    const float m1[4] = {a1.x * rs, a1.y * rs, a1.z * rs, a1.w * rs};
    const float mrow[4] = {a2.x * rs, a2.y * rs, a2.z * rs, a2.w * rs};
    float pj, uj, crow[4];
    split_sinkhorn_row(mrow, m0[j], m1[j], j, __ldg(P.scale), __ldg(P.scale + 1),
                       __ldg(P.scale + 2), P.base, P.iters, P.hc_eps, pj, uj, crow);
    if (in_range && token2 < P.N) {
      P.pre_out[static_cast<size_t>(token2) * 4 + j] = pj;
      P.post_out[static_cast<size_t>(token2) * 4 + j] = uj;
      reinterpret_cast<float4*>(P.comb_out + static_cast<size_t>(token2) * 16)[j] =
          make_float4(crow[0], crow[1], crow[2], crow[3]);
      if (P.mixes_out != nullptr) {
        float4* mo = reinterpret_cast<float4*>(P.mixes_out + static_cast<size_t>(token2) * 24);
        mo[2 + j] = make_float4(mrow[0], mrow[1], mrow[2], mrow[3]);
        if (j == 0) mo[0] = make_float4(m0[0], m0[1], m0[2], m0[3]);
        if (j == 1) mo[1] = make_float4(m1[0], m1[1], m1[2], m1[3]);
      }
    }
  }
  if (threadIdx.x == 0) stamp(5);

  if (FUSED && warp >= NROLE) {
    // ---------------------------------------------------------------- RMSNorm of this slice
    const int c = warp - NROLE;
    const int sub = warp & 3;
    const int h = c >> 2;
    const int tl = sub * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const uint32_t row_off = sw32_offset(tl, h);
    const uint64_t stream_pol = policy_evict_first();
    if (h == 0) {
      float sy = 0.f;
      const uint32_t local = smem_u32(part + tl * PART_STRIDE + 24);
      for (int rk = 0; rk < P.split; ++rk) sy += ld_cluster_f32x4(map_cluster(local, rk)).y;
      ry[tl] = __frsqrt_rn(__fdiv_rn(sy, static_cast<float>(d)) + P.norm_eps);
    }
    named_bar_sync(1, NCONS * 32);
    const float r = ry[tl];
    const f2 r2{r, r};
    auto norm_stage = [&](int s, int slot, const uint32_t* w) {
      const int i = col0 + s * cstride + h * 8;
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(P.gain + i));
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(P.gain + i + 4));
      const f2 gp[4] = {f2{g0.x, g0.y}, f2{g0.z, g0.w}, f2{g1.x, g1.y}, f2{g1.z, g1.w}};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = f2_to_bf2(mul2(gp[e], mul2(bf2_to_f2(w[e]), r2)));
      *reinterpret_cast<uint4*>(sm + yslot(slot) + row_off) = make_uint4(o[0], o[1], o[2], o[3]);
    };
    for (int s0 = 0; s0 < S; s0 += NYSLOTS) {
      const int s1 = min(S, s0 + NYSLOTS);
      int s = s0;
      for (; s + 8 <= s1; s += 8) {   // 8 stages of y_hat = 32 TMEM columns in one load
        uint32_t w[32];
        tmem_ld_x32(lane_base + STASH_COL + static_cast<uint32_t>(h * S * 4 + s * 4), w);
#pragma unroll
        for (int j = 0; j < 8; ++j) norm_stage(s + j, s + j - s0, w + 4 * j);
      }
      for (; s < s1; ++s) {
        uint32_t w[4];
        tmem_ld_x4(lane_base + STASH_COL + static_cast<uint32_t>(h * S * 4 + s * 4), w);
        norm_stage(s, s - s0, w);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, NCONS * 32);
      if (warp == NROLE && lane == 0) {
        for (int s = s0; s < s1; ++s)
          tma_store_2d_hint(&tm_y, sm + yslot(s - s0), col0 + s * cstride, t0, stream_pol);
        bulk_commit();
        bulk_wait_read<0>();   // staging slots may be rewritten once read
      }
      named_bar_sync(1, NCONS * 32);
    }
    if (warp == NROLE && lane == 0) stamp(6);
  }

  if ((P.flags & 2u) != 0 && threadIdx.x == 0) {
    if (!mbar_wait(never, 0, DEBUG_WAIT_NS)) timed_out = true;
  }
  if (timed_out) atomicOr(P.status, STATUS_TIMEOUT);

  // ------------------------------------------------------------------ leave together
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (threadIdx.x == 0 && tr != nullptr) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    tr[7] = (static_cast<unsigned long long>(smid) << 40) | (global_timer_ns() - t_start);
  }
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
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
  P.trace = trace_buffer(static_cast<int64_t>(a.split) * ((a.N + TT - 1) / TT));
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

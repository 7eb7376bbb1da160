// cluster.cu -- the fused single-pass mHC step for small batches (decode): one thread-block
// cluster per tile of 40 tokens, whose CTAs sum their partial results through distributed shared
// memory.
//
// What it computes is the step of fused.cu (MoE RMSNorm, Code: Block.forward, FFN half, with
// hc_post, hc_mixes, hc_pre from Stream weights for the feed-forward, Code; the single pass of that
// page's "Why" section), with the same float32 arithmetic per element (hc_arith.cuh) and per token
// (mix_math.cuh). Only the decomposition differs.
//
// Why a second kernel. With a few hundred tokens the persistent kernel's groups walk one tile
// each, and its time goes to latency chains, not bandwidth: a 128-row pipeline slot keeps half its
// consumer threads idle at 64-token tiles, and the group's partial sums travel through L2 behind
// GPU-scope release/acquire counters that a memset zeroes before every cooperative launch. Here:
//   * A cluster of CL CTAs (16, or 8) owns one tile; CTA r owns the columns {32 (s CL + r) + 0..31 :
//     s < S} of every stream, S = d / (32 CL) chunks (at most 10). At chunk s the cluster reads one
//     contiguous run of 32 CL columns of each token row. 40-token tiles: a GB300 runs 7 clusters
//     of 16 CTAs at once (a cluster's CTAs share a GPC), so 256 tokens take one wave.
//   * Every chunk of X and F stays in shared memory for the whole kernel (S x 15 KB): no ring to
//     recycle. The bulk copies one thread issues are served one after another (about 0.35 us each
//     in a probe, 8 KB or 16 KB), so every tile has a lane of its own: lane L of warp 0 copies
//     tiles L and L + 32 of the 5 S (X_0..X_3 and F of each chunk) and later stores X' or y from
//     them. Warp 0 also refills the weight ring, so that the MMA lane never waits for its own MMAs
//     to complete (a lane spinning on that wait, diverged from the MMA lane in the same warp,
//     delayed the MMA issue by up to 3 us).
//   * 10 consumer warps, 8 threads per token, 4 columns per thread and chunk, compute X' in place
//     over X and y_hat (bf16) in place over F, with the sums of squares of both.
//   * Lane 0 of warp 1 issues tcgen05.mma per chunk, D[128 x 80] += X'[128 x 16] Wp[80 x 16]^T
//     (rows at and past 40 read the next tiles of shared memory and are never used), the packed
//     weights streaming through a 3-entry ring (one 20 KB block per entry); each accumulation group
//     of 16 MMAs (two chunks) has its own TMEM accumulator, summed in float32 at the end.
//   * Exchange, push only, each row stored once with st.async into the destination CTA's shared
//     memory, counted by that CTA's mbarrier (expected bytes set before the cluster barrier):
//       - every CTA's S_y of the tile's tokens to every CTA of the cluster (the RMS factor of y);
//       - each token's 24 partial mix sums and S_x to the CTA that finishes the token
//         (token t -> CTA t mod CL).
//     No counters in global memory, no memset, no cooperative launch; the clusters are
//     independent, so a launch may hold more of them than the GPU runs at once.
//   * Warp 1 then finishes its tokens (four lanes per token sum the CL rows, scale, split,
//     Sinkhorn, outputs) while the consumers normalise y in place and warp 0 stores it.
// Every wait is bounded (2 s) and reports through the status word; the kernel never traps.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "hc_arith.cuh"
#include "layout.cuh"
#include "mix_math.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int CT = kClusterTile;             // tokens per tile (one cluster): 40
constexpr int CDC = STEP_WDC;                // columns per chunk: one packed weight block
constexpr int CROWB = CDC * 2;               // 64-byte tile rows (64-byte swizzle)
constexpr int CTILE = 3072;                  // one [CT tokens x 32 columns] bf16 tile, 1 KB aligned
constexpr int CCHUNK = 5 * CTILE;            // X_0..X_3, then F
constexpr int CMAX_S = 10;                   // chunks per CTA at most
constexpr int CMAX_CL = 16;                  // CTAs per cluster at most (non-portable size)
constexpr int CTPT = 8;                      // consumer threads per token, 4 columns each
constexpr int CNCW = CT * CTPT / 32;         // consumer warps: 10
constexpr int CTHREADS = (2 + CNCW) * 32;
constexpr int CNWB = 3;                      // weight ring entries
constexpr int CROWF = 28;                    // exchange row: 24 mix sums, S_x, 3 unused
constexpr int CMAX_TPO = (CT + 7) / 8;       // tokens a CTA finishes, at most (8-CTA clusters)
constexpr int CXROWS = 48;                   // exchange rows: slot j, rank r at j * CL + r
constexpr int MMA_M = 128;
constexpr uint32_t CTMEM_COLS = 512;         // (CMAX_S + 1) / 2 accumulators of 80 columns
static_assert(CROWB == STEP_WROW_BYTES && CDC == 32, "a chunk is one packed weight block");
static_assert(CT % 8 == 0 && CT * CROWB <= CTILE && CTILE % 1024 == 0, "tiles of whole 8-row groups, 1 KB aligned");
static_assert(CNCW * 32 == CT * CTPT, "whole consumer warps");
static_assert((CMAX_S + 1) / 2 * STEP_MMA_N <= static_cast<int>(CTMEM_COLS), "accumulators fit TMEM");
static_assert(CT <= 64, "tile rows in TMEM lane quarters 0 and 1");
static_assert(CXROWS >= ((CT + 15) / 16) * 16 && CXROWS >= CT, "exchange rows for 8- and 16-CTA clusters");
static_assert(4 * CMAX_TPO <= 32, "four finisher lanes per token");

constexpr int OFF_XF = 0;
constexpr int OFF_W = OFF_XF + CMAX_S * CCHUNK;
constexpr int OFF_MIX = OFF_W + CNWB * STEP_WBLOCK_BYTES;    // [CXROWS][CROWF]
constexpr int OFF_SY = OFF_MIX + CXROWS * CROWF * 4;         // [CL ranks][CT] S_y
constexpr int OFF_LOC = OFF_SY + CMAX_CL * CT * 4;           // this CTA's S_x[CT], S_y[CT]
constexpr int OFF_PAR = OFF_LOC + 2 * CT * 4;                // scale[3] at 0, base[24] at 8
constexpr int OFF_BARS = OFF_PAR + 32 * 4;
// full[CMAX_S], xready[CMAX_S], wfull[CNWB], wempty[CNWB], accdone, mixin, syin, ydone, never
constexpr int CNBARS = 2 * CMAX_S + 2 * CNWB + 5;
constexpr int OFF_TMEM = OFF_BARS + CNBARS * 8;
constexpr int CSMEM = OFF_TMEM + 16 + 1024;                  // + slack for 1 KB alignment
static_assert(CSMEM <= 232448, "shared memory budget");
// The MMA's A operand spans 128 rows (8 KB) from a tile's base: the last X tile's span stays
// inside shared memory (it ends in the weight ring).
static_assert(OFF_XF + (CMAX_S - 1) * CCHUNK + 3 * CTILE + MMA_M * CROWB <= OFF_MIX,
              "A-operand span inside shared memory");
static_assert(OFF_W % 1024 == 0 && STEP_WBLOCK_BYTES % 1024 == 0, "weight tiles 1 KB aligned");
static_assert(OFF_MIX % 16 == 0 && OFF_SY % 16 == 0 && (CROWF * 4) % 16 == 0 && (CT * 4) % 16 == 0,
              "16-byte st.async targets");

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s
constexpr uint64_t DEBUG_WAIT_NS = 2000000ull;      // 2 ms

struct ClusterParams {
  const float* pre_prev;
  const float* post_prev;
  const float* comb_prev;
  const float* scale;
  const float* base;
  const float* gain;
  const uint8_t* w_packed;
  float* pre_out;
  float* post_out;
  float* comb_out;
  float* mixes_out;            // nullable
  unsigned* status;
  int N;
  int d;
  int cl;                      // CTAs per cluster: 8 or 16
  int S;                       // chunks per CTA: d / (32 cl)
  int iters;
  float hc_eps;
  float norm_eps;
  float neg_zero;              // -0.0: the run-time zero addend of the rounded products
  unsigned flags;
};

// Bounds checks of the checked build (MHC_CHECKED=1), as in the persistent kernel: a failed test
// records STATUS_BOUNDS and the access is skipped.
__device__ __forceinline__ bool checked(bool ok, unsigned* status) {
#if MHC_CHECKED
  if (!ok) atomicOr(status, STATUS_BOUNDS);
  return ok;
#else
  (void)status;
  (void)ok;
  return true;
#endif
}

__global__ void __launch_bounds__(CTHREADS, 1)
    cluster_step_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_f,
                        const __grid_constant__ CUtensorMap tm_xo, const __grid_constant__ CUtensorMap tm_y,
                        const ClusterParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + OFF_BARS);   // [CMAX_S]: chunk s landed
  uint64_t* xready = full + CMAX_S;         // [CMAX_S]: chunk s's X' written (consumer warps)
  uint64_t* wfull = xready + CMAX_S;        // [CNWB]: weight entry landed
  uint64_t* wempty = wfull + CNWB;          // [CNWB]: the MMAs reading the entry completed
  uint64_t* accdone = wempty + CNWB;        // every MMA completed
  uint64_t* mixin = accdone + 1;            // the cluster's rows of this CTA's tokens arrived
  uint64_t* syin = mixin + 1;               // the cluster's S_y arrived
  uint64_t* ydone = syin + 1;               // y normalised in place (consumer warps)
  uint64_t* never = ydone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM);
  float* mixbuf = reinterpret_cast<float*>(sm + OFF_MIX);
  float* sybuf = reinterpret_cast<float*>(sm + OFF_SY);
  float* sxl = reinterpret_cast<float*>(sm + OFF_LOC);
  float* syl = sxl + CT;
  float* par = reinterpret_cast<float*>(sm + OFF_PAR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int CL = P.cl;
  const int S = P.S;
  const int d = P.d;
  const uint32_t rank = cluster_ctarank();
  const int t0 = static_cast<int>(blockIdx.x / CL) * CT;
  // tokens this CTA finishes: tile rows rank, rank + CL, ...
  const int tpo = (CT - static_cast<int>(rank) + CL - 1) / CL;
  bool timed_out = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < CMAX_S; ++s) {
      mbar_init(&full[s], 5);
      mbar_init(&xready[s], CNCW);
    }
    for (int e = 0; e < CNWB; ++e) {
      mbar_init(&wfull[e], 1);
      mbar_init(&wempty[e], 1);
    }
    mbar_init(accdone, 1);
    mbar_init(mixin, 1);
    mbar_init(syin, 1);
    mbar_init(ydone, CNCW);
    mbar_init(never, 1);
    // the bytes the cluster pushes here, expected before any CTA may push (cluster barrier below)
    if (tpo > 0) mbar_arrive_expect_tx(mixin, static_cast<uint32_t>(tpo * CL * CROWF * 4));
    mbar_arrive_expect_tx(syin, static_cast<uint32_t>(CL * CT * 4));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, CTMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  block_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // every thread arrives now and waits before its first access to another CTA's shared memory:
  // by then every CTA of the cluster runs and has initialised its barriers
  cluster_arrive_release();

  if (warp == 0) {
    // ------------------------------------------------------------------ loads, then stores
    // tile u = 5 s + k (k < 4: X_k of chunk s, k = 4: F) belongs to lane u % 32, which copies it
    // in and later stores X' or y from it
    const uint64_t pol = policy_evict_first();
    const uint64_t wpol = policy_evict_last();
    const int ntile = 5 * S;
    // chunk s's weight block (global column block s CL + rank) into ring entry s % CNWB
    auto load_w = [&](int s) {
      const int e = s % CNWB;
      const int blk = s * CL + static_cast<int>(rank);
      if (!checked(blk >= 0 && (blk + 1) * CDC <= d, P.status)) {
        mbar_arrive(&wfull[e]);
        return;
      }
      mbar_arrive_expect_tx(&wfull[e], STEP_WBLOCK_BYTES);
      bulk_load_hint(sm + OFF_W + e * STEP_WBLOCK_BYTES, P.w_packed + static_cast<size_t>(blk) * STEP_WBLOCK_BYTES,
                     STEP_WBLOCK_BYTES, &wfull[e], wpol);
    };
    if (lane >= 29 && lane - 29 < S) load_w(lane - 29);   // the first CNWB blocks, one lane each
    if (lane == 0) tma_prefetch_desc(&tm_x);
    if (lane == 1) tma_prefetch_desc(&tm_f);
    if (lane == 2) tma_prefetch_desc(&tm_xo);
    if (lane == 3) tma_prefetch_desc(&tm_y);
    for (int u = lane; u < ntile; u += 32) {
      const int s = u / 5, k = u % 5;
      const int col = (s * CL + static_cast<int>(rank)) * CDC;
      uint8_t* tile = sm + OFF_XF + s * CCHUNK + k * CTILE;
      if (checked(col >= 0 && col + CDC <= d && t0 >= 0 && t0 < P.N, P.status)) {
        mbar_arrive_expect_tx(&full[s], CT * CROWB);
        if (k < 4) tma_load_3d_hint(tile, &tm_x, &full[s], col, k, t0, pol);
        else tma_load_2d_hint(tile, &tm_f, &full[s], col, t0, pol);
      } else {
        mbar_arrive(&full[s]);          // the chunk completes without data
      }
    }
    // X' of chunk s once its consumers are done with it, from the lanes of its tiles; then the
    // weight entry of chunk s - 1, once its MMAs have read it, takes chunk s - 1 + CNWB's block
    for (int s = 0; s < S; ++s) {
      if (!mbar_wait(&xready[s], 0, WAIT_LIMIT_NS)) timed_out = true;
      const int k = (lane - 5 * s) & 31;       // this lane's tile of chunk s, if k < 4
      const int col = (s * CL + static_cast<int>(rank)) * CDC;
      if (k < 4 && checked(col >= 0 && col + CDC <= d && t0 >= 0 && t0 < P.N, P.status)) {
        tma_store_3d_hint(&tm_xo, sm + OFF_XF + s * CCHUNK + k * CTILE, col, k, t0, pol);
        bulk_commit();
      }
      if (s >= 1 && s - 1 + CNWB < S) {
        if (!mbar_wait(&wempty[(s - 1) % CNWB], ((s - 1) / CNWB) & 1, WAIT_LIMIT_NS)) timed_out = true;
        if (lane == (s - 1) % 32) load_w(s - 1 + CNWB);
      }
    }
    if (!mbar_wait(ydone, 0, WAIT_LIMIT_NS)) timed_out = true;
    // y (normalised in place of F) of the chunks whose F tile is this lane's
    for (int u = lane; u < ntile; u += 32) {
      const int s = u / 5;
      const int col = (s * CL + static_cast<int>(rank)) * CDC;
      if (u % 5 == 4 && checked(col >= 0 && col + CDC <= d && t0 >= 0 && t0 < P.N, P.status)) {
        tma_store_2d_hint(&tm_y, sm + OFF_XF + s * CCHUNK + 4 * CTILE, col, t0, pol);
        bulk_commit();
      }
    }
    bulk_wait_read<0>();                // shared memory stays valid until the stores read it
    if (lane == 0 && (P.flags & 2u) != 0 && !mbar_wait(never, 0, DEBUG_WAIT_NS)) timed_out = true;
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Lane 0 issues the MMAs; the other lanes bring in the split's parameters meanwhile.
    if (lane >= 4 && lane < 7) par[lane - 4] = __ldg(P.scale + (lane - 4));
    if (lane >= 8) par[lane] = __ldg(P.base + (lane - 8));
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(MMA_M, STEP_MMA_N);
      for (int s = 0; s < S; ++s) {
        const int e = s % CNWB;
        if (!mbar_wait(&xready[s], 0, WAIT_LIMIT_NS)) timed_out = true;
        if (!mbar_wait(&wfull[e], (s / CNWB) & 1, WAIT_LIMIT_NS)) timed_out = true;
        tc_fence_after();
        // accumulation group s / 2 (16 MMAs) into its own accumulator
        const uint32_t acc = tmem + static_cast<uint32_t>((s >> 1) * STEP_MMA_N);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a0 = smem_u32(sm + OFF_XF + s * CCHUNK + k * CTILE);
          const uint32_t b0 = smem_u32(sm + OFF_W + e * STEP_WBLOCK_BYTES + k * STEP_WSTREAM_BYTES);
#pragma unroll
          for (int kk = 0; kk < CDC / 16; ++kk)
            umma_bf16(acc, sdesc_kmajor_swizzled(a0 + 32 * kk, CROWB),
                      sdesc_kmajor_swizzled(b0 + 32 * kk, STEP_WROW_BYTES), idesc,
                      ((s & 1) != 0 || k != 0 || kk != 0) ? 1u : 0u);
        }
        umma_commit(&wempty[e]);
      }
      umma_commit(accdone);
    }
    __syncwarp();
    // ------------------------------------------------------------------ finisher
    // Tile rows j CL + rank (j < tpo): lane 4j + jr adds the rows of ranks jr, jr + 4, ... of slot
    // j, two shuffles give the four lanes the token's sums, each runs the whole split + Sinkhorn
    // (split_sinkhorn_all), and lane 4j + jr writes row jr.
    if (tpo > 0) {
      if (!mbar_wait_cluster(mixin, 0, WAIT_LIMIT_NS)) timed_out = true;
      const int j = lane >> 2;
      const int jr = lane & 3;
      const int js = j < tpo ? j : 0;
      float acc[25];
#pragma unroll
      for (int e = 0; e < 25; ++e) acc[e] = 0.f;
      for (int r = jr; r < CL; r += 4) {
        const float4* row = reinterpret_cast<const float4*>(mixbuf + (js * CL + r) * CROWF);
#pragma unroll
        for (int q = 0; q < 7; ++q) {
          const float4 v = row[q];
          const float a4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (4 * q + c < 25) acc[4 * q + c] += a4[c];
        }
      }
#pragma unroll
      for (int e = 0; e < 25; ++e) {
        acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 1);
        acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 2);
      }
      const int tl = js * CL + static_cast<int>(rank);
      const int token = t0 + tl;
      const float rs = __frsqrt_rn(__fdiv_rn(acc[24], static_cast<float>(4 * d)) + P.norm_eps);
      float m[24], b[24];
#pragma unroll
      for (int e = 0; e < 24; ++e) {
        m[e] = acc[e] * rs;
        b[e] = par[8 + e];
      }
      float pv[4], uv[4], cv[16];
      split_sinkhorn_all(m, par[0], par[1], par[2], b, P.iters, P.hc_eps, pv, uv, cv);
      const float pj = jr == 0 ? pv[0] : jr == 1 ? pv[1] : jr == 2 ? pv[2] : pv[3];
      const float uj = jr == 0 ? uv[0] : jr == 1 ? uv[1] : jr == 2 ? uv[2] : uv[3];
      float crow[4], mrow[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        crow[k] = jr == 0 ? cv[k] : jr == 1 ? cv[4 + k] : jr == 2 ? cv[8 + k] : cv[12 + k];
        mrow[k] = jr == 0 ? m[8 + k] : jr == 1 ? m[12 + k] : jr == 2 ? m[16 + k] : m[20 + k];
      }
#if MHC_CHECKED
      // test hook: the first token's row goes N rows past the end (the checks skip it)
      const int row = token + ((P.flags & FLAG_PLANT_OOB) != 0 && blockIdx.x == 0 && j == 0 ? P.N : 0);
#else
      const int row = token;
#endif
      if (j < tpo && token < P.N && checked(row >= 0 && row < P.N, P.status)) {
        P.pre_out[static_cast<size_t>(row) * 4 + jr] = pj;
        P.post_out[static_cast<size_t>(row) * 4 + jr] = uj;
        reinterpret_cast<float4*>(P.comb_out + static_cast<size_t>(row) * 16)[jr] =
            make_float4(crow[0], crow[1], crow[2], crow[3]);
        if (P.mixes_out != nullptr) {
          float4* mo = reinterpret_cast<float4*>(P.mixes_out + static_cast<size_t>(row) * 24);
          mo[2 + jr] = make_float4(mrow[0], mrow[1], mrow[2], mrow[3]);
          if (jr == 0) mo[0] = make_float4(m[0], m[1], m[2], m[3]);
          if (jr == 1) mo[1] = make_float4(m[4], m[5], m[6], m[7]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ consumers
    const int c = warp - 2;
    const int i = c * 32 + lane;
    const int t = i / CTPT;                  // token row of the tile
    const int q = i % CTPT;                  // columns 4q .. 4q + 3 of every chunk
    const uint32_t off = tile_chunk_offset(t, q >> 1) + 8u * static_cast<uint32_t>(q & 1);
    const int token = t0 + t;
    const bool valid = token < P.N;
    const bool row_dest = (P.flags & 1u) != 0;
    f2 cu[4], cpv[4], cc[4][4];
    {
      float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f), p4 = u4, cm[4] = {u4, u4, u4, u4};
      if (valid) {
        u4 = __ldg(reinterpret_cast<const float4*>(P.post_prev) + token);
        p4 = __ldg(reinterpret_cast<const float4*>(P.pre_prev) + token);
#pragma unroll
        for (int r = 0; r < 4; ++r) cm[r] = __ldg(reinterpret_cast<const float4*>(P.comb_prev) + 4 * static_cast<size_t>(token) + r);
      }
      const float uu[4] = {u4.x, u4.y, u4.z, u4.w}, pp[4] = {p4.x, p4.y, p4.z, p4.w};
      float cmf[16];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        cmf[4 * r] = cm[r].x;
        cmf[4 * r + 1] = cm[r].y;
        cmf[4 * r + 2] = cm[r].z;
        cmf[4 * r + 3] = cm[r].w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cu[k] = f2{uu[k], uu[k]};
        cpv[k] = f2{pp[k], pp[k]};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // cc[j][k]: coefficient of input stream j in output stream k
          const float v = cmf[row_dest ? (k * 4 + j) : (j * 4 + k)];
          cc[j][k] = f2{v, v};
        }
      }
    }
    const f2 nz2{P.neg_zero, P.neg_zero};
    f2 lx{0.f, 0.f}, ly{0.f, 0.f};
    for (int s = 0; s < S; ++s) {
      if (!mbar_wait(&full[s], 0, WAIT_LIMIT_NS)) timed_out = true;
      uint8_t* ch = sm + OFF_XF + s * CCHUNK;
      uint2 xw[4], ow[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) xw[k] = *reinterpret_cast<const uint2*>(ch + k * CTILE + off);
      const uint2 fw = *reinterpret_cast<const uint2*>(ch + 4 * CTILE + off);
      uint32_t yw[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        f2 x[4], xp[4];
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = bf2_to_f2(h == 0 ? xw[k].x : xw[k].y);
        const f2 f = bf2_to_f2(h == 0 ? fw.x : fw.y);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // X'_k: rounded products summed in stream order (hc_arith.cuh)
          const f2 ck[4] = {cc[0][k], cc[1][k], cc[2][k], cc[3][k]};
          o[k] = f2_to_bf2(hc_post_pair(ck, cu[k], x, f, nz2));
          xp[k] = bf2_to_f2(o[k]);
          lx = fma2(xp[k], xp[k], lx);
        }
        yw[h] = f2_to_bf2(hc_pre_pair(cpv, xp, nz2));
        const f2 yr = bf2_to_f2(yw[h]);
        ly = fma2(yr, yr, ly);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (h == 0) ow[k].x = o[k];
          else ow[k].y = o[k];
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) *reinterpret_cast<uint2*>(ch + k * CTILE + off) = ow[k];
      *reinterpret_cast<uint2*>(ch + 4 * CTILE + off) = make_uint2(yw[0], yw[1]);   // y_hat over F
      fence_proxy_async_smem();          // X' is read by the tensor cores and the store copies
      __syncwarp();
      if (lane == 0) mbar_arrive(&xready[s]);
    }
    // the token's sums of squares over this CTA's columns: CTPT lanes per token
    float sx = lx.x + lx.y, sy = ly.x + ly.y;
#pragma unroll
    for (int o = 1; o < CTPT; o <<= 1) {
      sx += __shfl_xor_sync(0xffffffffu, sx, o);
      sy += __shfl_xor_sync(0xffffffffu, sy, o);
    }
    if (q == 0) {
      sxl[t] = sx;
      syl[t] = sy;
    }
    // this thread's gains, in flight during the exchange
    float4 gl[CMAX_S];
#pragma unroll
    for (int s = 0; s < CMAX_S; ++s)
      gl[s] = s < S ? __ldg(reinterpret_cast<const float4*>(P.gain + (s * CL + static_cast<int>(rank)) * CDC + 4 * q))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    named_bar_sync(1, CNCW * 32);            // S_x, S_y of every token in shared memory
    cluster_wait_acquire();
    if (c == 0) {
      // this CTA's S_y of the tile's tokens to every CTA of the cluster: [rank][CT] there
      for (int k = lane; k < CL * (CT / 4); k += 32) {
        const uint32_t dst = static_cast<uint32_t>(k / (CT / 4));
        const int v = k % (CT / 4);
        const float4 val = reinterpret_cast<const float4*>(syl)[v];
        st_async_v4(mapa_shared(smem_u32(sybuf + rank * CT + 4 * v), dst), val,
                    mapa_shared(smem_u32(syin), dst));
      }
    }
    if (warp == 4 || warp == 5 || warp == 8 || warp == 9) {
      // The accumulator rows (tile rows) of TMEM lane quarter 0 belong to warps 4 and 8, those of
      // quarter 1 to warps 5 and 9; warps 4, 5 sum mix numbers 0..11, warps 8, 9 12..23. The
      // packed weight rows put half h of the 24 mix numbers, all three planes, in accumulator
      // columns [36h, 36h + 36): 12 hi, 12 mid, 12 lo.
      const int h = warp >= 8 ? 1 : 0;
      const int tr = (warp & 3) * 32 + lane;   // tile row of this lane
      if (!mbar_wait(accdone, 0, WAIT_LIMIT_NS)) timed_out = true;
      tc_fence_after();
      float run[12];
#pragma unroll
      for (int e = 0; e < 12; ++e) run[e] = 0.f;
      const int nacc = (S + 1) / 2;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      for (int a = 0; a < nacc; ++a) {
        uint32_t v[32], w4[4];
        const uint32_t col = lane_base + static_cast<uint32_t>(a * STEP_MMA_N + 36 * h);
        tmem_ld_x32(col, v);
        tmem_ld_x4(col + 32, w4);
#pragma unroll
        for (int e = 0; e < 12; ++e) {
          const float lo = __uint_as_float(e < 8 ? v[24 + e] : w4[e - 8]);
          run[e] += (lo + __uint_as_float(v[12 + e])) + __uint_as_float(v[e]);
        }
      }
      if (tr < CT) {
        // token row tr is finished by CTA tr % CL, slot tr / CL: row (slot, rank) there
        const uint32_t dst = static_cast<uint32_t>(tr % CL);
        const int j = tr / CL;
        const uint32_t ra = mapa_shared(smem_u32(mixbuf + (j * CL + static_cast<int>(rank)) * CROWF), dst);
        const uint32_t rb = mapa_shared(smem_u32(mixin), dst);
#pragma unroll
        for (int e = 0; e < 3; ++e)
          st_async_v4(ra + 48u * h + 16u * e, make_float4(run[4 * e], run[4 * e + 1], run[4 * e + 2], run[4 * e + 3]), rb);
        if (h == 0) st_async_v4(ra + 96u, make_float4(sxl[tr], 0.f, 0.f, 0.f), rb);
      }
    }
    // y = bf16(gain * (y_hat * r_y)) in place of y_hat, r_y from the cluster's S_y (rank order)
    if (!mbar_wait_cluster(syin, 0, WAIT_LIMIT_NS)) timed_out = true;
    float tot = 0.f;
    for (int r = 0; r < CL; ++r) tot += sybuf[r * CT + t];
    const float rr = __frsqrt_rn(__fdiv_rn(tot, static_cast<float>(d)) + P.norm_eps);
    const f2 r2{rr, rr};
#pragma unroll
    for (int s = 0; s < CMAX_S; ++s) {
      if (s < S) {
        uint2* p = reinterpret_cast<uint2*>(sm + OFF_XF + s * CCHUNK + 4 * CTILE + off);
        const uint2 w = *p;
        *p = make_uint2(f2_to_bf2(mul2(f2{gl[s].x, gl[s].y}, mul2(bf2_to_f2(w.x), r2))),
                        f2_to_bf2(mul2(f2{gl[s].z, gl[s].w}, mul2(bf2_to_f2(w.y), r2))));
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(ydone);
  }

  if (timed_out) atomicOr(P.status, STATUS_TIMEOUT);
  if (warp < 2) cluster_wait_acquire();      // the consumers waited before their pushes
  tc_fence_before();
  block_sync();
  if (warp == 1) tmem_dealloc(tmem, CTMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// host side

bool cmap(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
          const cuuint32_t* box) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [N, 4, d] as (column, stream, token), one stream's [CT x 32] tile per box.
bool cmap_streams(CUtensorMap* m, const void* p, int64_t N, int d) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), 4, static_cast<cuuint64_t>(N)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 8};
  const cuuint32_t box[3] = {CDC, 1, CT};
  return cmap(m, p, 3, dims, str, box);
}
bool cmap_rows(CUtensorMap* m, const void* p, int64_t N, int d) {   // [N, d]
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N)};
  const cuuint64_t str[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {CDC, CT};
  return cmap(m, p, 2, dims, str, box);
}

// The kernel's attributes on the current device (they are per device: set once for each).
cudaError_t prepare() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  err = cudaFuncSetAttribute(cluster_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CSMEM);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(cluster_step_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (err == cudaSuccess) done[dev] = true;
  return err;
}

}  // namespace

int cluster_size_for(int d, int forced) {
  for (int cl : {16, 8}) {
    if (forced != 0 && cl != forced) continue;
    if (d > 0 && d % (CDC * cl) == 0 && d / (CDC * cl) <= CMAX_S) return cl;
  }
  return 0;
}

int cluster_capacity(int cl) {
  static std::mutex mu;
  static int cache[2][64] = {};          // [cl == 16][device]
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& v = cache[cl == 16 ? 1 : 0][dev];
  if (v != 0) return v < 0 ? 0 : v;
  int n = 0;
  if (prepare() == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cl), 1, 1);
    cfg.blockDim = dim3(CTHREADS, 1, 1);
    cfg.dynamicSmemBytes = CSMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, cluster_step_kernel, &cfg) != cudaSuccess) {
      n = 0;
      cudaGetLastError();                // the refused query's error is not the caller's
    }
  }
  v = n > 0 ? n : -1;
  return n;
}

int cluster_path(int64_t N, int d, unsigned flags, bool fused_bf16) {
  if (!fused_bf16 || (flags & FLAG_PATH_PERSISTENT) != 0) return 0;
  const bool forced = (flags & FLAG_PATH_CLUSTER) != 0;
  const int fs = split_flag_value(flags);
  if (!forced && (fs != 0 || tile_flag(flags) != 0)) return 0;   // shape flags of the persistent kernel
  int cl = cluster_size_for(d, forced ? fs : 0);
  if (cl == 0) return 0;
  // 16-CTA clusters are a non-portable size: where the device runs none, 8 if d fits them
  if (cl == 16 && fs == 0 && cluster_capacity(16) == 0 && cluster_size_for(d, 8) == 8) cl = 8;
  if (forced) return cl;
  // automatic: while every tile's cluster runs at once
  const int64_t tiles = (N + CT - 1) / CT;
  const int cap = cluster_capacity(cl);
  return (cap > 0 && tiles <= static_cast<int64_t>(cap) * kClusterWaves) ? cl : 0;
}

cudaError_t launch_cluster_step(const StepArgs& a, int cl, cudaStream_t stream) {
  cudaError_t e = prepare();
  if (e != cudaSuccess) return e;
  if (cluster_size_for(a.d, cl) != cl) return cudaErrorInvalidConfiguration;
  CUtensorMap tx, tf, txo, ty;
  if (!cmap_streams(&tx, a.X, a.N, a.d) || !cmap_streams(&txo, a.X_out, a.N, a.d) ||
      !cmap_rows(&tf, a.F, a.N, a.d) || !cmap_rows(&ty, a.y_out, a.N, a.d))
    return cudaErrorInvalidValue;
  ClusterParams P{};
  P.pre_prev = a.pre_prev;
  P.post_prev = a.post_prev;
  P.comb_prev = a.comb_prev;
  P.scale = a.scale;
  P.base = a.base;
  P.gain = a.gain;
  P.w_packed = static_cast<const uint8_t*>(a.W_packed);
  P.pre_out = a.pre_out;
  P.post_out = a.post_out;
  P.comb_out = a.comb_out;
  P.mixes_out = a.mixes_out;
  P.status = status_word();
  if (P.status == nullptr) return cudaErrorInvalidDevice;
  P.N = static_cast<int>(a.N);
  P.d = a.d;
  P.cl = cl;
  P.S = a.d / (CDC * cl);
  P.iters = a.iters;
  P.hc_eps = a.hc_eps;
  P.norm_eps = a.norm_eps;
  P.neg_zero = -0.0f;
  P.flags = a.flags;
  const int64_t tiles = (a.N + CT - 1) / CT;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * cl), 1, 1);
  cfg.blockDim = dim3(CTHREADS, 1, 1);
  cfg.dynamicSmemBytes = CSMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cluster_step_kernel, tx, tf, txo, ty, P);
}

}  // namespace mhc

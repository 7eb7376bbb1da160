// fused.cu -- the single-pass mHC step on sm_103a: one kernel reads X and F once and writes X',
// the normalised sublayer input y and the new mix coefficients (p, u, C).
//
// What it computes: MoE RMSNorm, Code: Block.forward (FFN half) with hc_post, hc_mixes, hc_pre
// from Stream weights for the feed-forward, Code; the single pass is the one that page's "Why"
// section describes (one pass over the streams serves the read and the next weights).
//
// Work decomposition. A group of `split` CTAs owns a tile of 128 tokens at a time and walks its
// tiles persistently (tile c, c + #groups, ...). The launch is cooperative with one CTA per SM,
// so every CTA of a group is resident and the groups use all SMs:
//   * Each CTA owns d/split columns of every stream (d = 5120: 8 CTAs x 640 columns). The CTAs'
//     columns interleave in slots of STEP_DC columns, so at every slot the group reads one
//     contiguous run of STEP_DC*split columns of each token row.
//   * Warp 0, lane 0 drives the X/F ring: per slot, [128 tokens x STEP_DC] tiles of X_0..X_3 and
//     F (tensor copies). The packed projection weights (32-column blocks, packed as the exact
//     shared-memory image the tensor cores read) flow through a ring of their own that the MMA
//     thread refills, so weight traffic never holds up the stream loads. Lane 1 (the poster)
//     does the CTA's group-counter releases and polls and bulk-copies each tile's previous
//     coefficients (p, u, C) into shared memory ahead of time.
//   * 8 consumer warps (2 threads per token) compute hc_post in place in shared memory, its sum
//     of squares, hc_pre and its sum of squares; y_hat goes to a TMEM stash. While doing so they
//     normalise the previous tile's y_hat from the same stash slot into the F tile they just
//     read, so the previous tile's y leaves with this slot's stores.
//   * Warp 1 issues tcgen05.mma: D[128 tokens x 80] += X'[128 x 16] * Wp[80 x 16]^T per stream
//     and K-step. Accumulation groups of 16 MMAs alternate between two TMEM accumulators and the
//     consumers fold each finished group into float32 running sums in shared memory.
//   * Warp 10 stores X' and y with TMA straight from the slot's tiles and frees the slot as soon
//     as the stores have read it.
//   * After a tile's last slot the consumers post their slice's partial sums to the group
//     through a scratch area in global memory (L2); the poster publishes them with
//     release-ordered counters. Warp 11 finishes the tile's mix numbers (scale, split,
//     Sinkhorn) while the consumers move on.
//   * After a CTA's last tile the consumers normalise the y still in the stash into the idle
//     rings' tiles and store it in one batch.
// step_kernel<true, true> is the same step writing y as MXFP8 (E4M3 codes and E8M0 block
// scales) instead of bf16.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "hc_arith.cuh"
#include "layout.cuh"
#include "mix_math.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int TT = STEP_TT;             // token rows of a tile (at most)
constexpr int MMA_M = 128;              // the MMA's M: A and D rows at and past the tile are ignored
constexpr int DC = STEP_DC;             // columns per X/F slot
constexpr int ROWB = STEP_ROW_BYTES;
constexpr int WDC = STEP_WDC;           // columns per packed weight block
constexpr int HALVES = DC / WDC;        // weight blocks per slot
constexpr int KSTEPS = WDC / 16;        // MMA K-steps per stream per weight block
constexpr int PG = 16 / (4 * HALVES * KSTEPS);      // slots per accumulation group (16 MMAs)
constexpr int NSTAGE = 4;               // X/F ring depth (40 KB slots)
constexpr int NW = 2;                   // weight ring entries (one block each)
// slots by which the y_hat stash ring outlasts a tile: the previous tile's RMS factor is taken
// after slot RLAG - 1 and used from slot RLAG on
constexpr int RLAG = 2;
constexpr int NCONS = 8;                // consumer warps (2 per TMEM lane quarter)
constexpr int NROLE = 2;                // warp 0: TMA producer; warp 1: TMEM owner and MMA issuer
constexpr int STORE_WARP = NROLE + NCONS;           // warp 10: X'/y TMA stores
constexpr int FIN_WARP = STORE_WARP + 1;            // warp 11: scale, split, Sinkhorn
constexpr int NTHREADS = (FIN_WARP + 1) * 32;
// Consumer layout: TT tokens over the TT/32 lane quarters whose TMEM lanes hold their
// accumulator rows; TPT threads per token (2 per quarter holding the token, times the quarters
// that share it), each owning CPH 16-byte chunks of every row of a slot. Only the warps in the
// quarters that hold accumulator rows fold (NFOLD warps).
constexpr int QPT = TT / 32;
constexpr int TPT = NCONS * 32 / TT;
constexpr int CPH = STEP_CHUNKS / TPT;
constexpr int NFOLD = NCONS * QPT / 4;
static_assert(CPH == 2, "a consumer thread owns 32 bytes of each slot row");
static_assert(TPT == 2 && DC == 32, "MXFP8 y: a slot row is one 32-feature block, two threads");
static_assert(4 * HALVES * KSTEPS * PG == 16, "accumulation groups of 16 MMAs");
constexpr int TILE_BYTES = TT * ROWB;               // one [TT tokens x DC] tile
constexpr int STAGE_BYTES = 5 * TILE_BYTES;         // X_0..X_3 and F
constexpr int RUN_STRIDE = 24;                      // floats per token of the local running sums
// exchange row per token: 24 mix sums, then S_x of each of the TPT parts (the rest of the row,
// up to a whole float4, is unused). S_y goes through tagged words (below).
constexpr int PART_STRIDE = 24 + 2 * TPT;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = STEP_MMA_N;         // two accumulators, at columns 0 and 80
constexpr uint32_t STASH_COL = 2 * ACC_COLS;
// y_hat stash: a ring of S + RLAG slots; each TMEM lane holds two threads' PASS_COLS columns per
// slot, so the widest slice is STASH_SLOTS - RLAG slots.
constexpr int PASS_COLS = 4 * CPH;                   // packed bf16 pairs per thread and slot
constexpr int SLOT_COLS = 2 * PASS_COLS;
constexpr int STASH_SLOTS = static_cast<int>(TMEM_COLS - STASH_COL) / SLOT_COLS;
constexpr int MAX_SLICE = (STASH_SLOTS - RLAG) * DC;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;        // 2 s
constexpr uint64_t DEBUG_WAIT_NS = 2000000ull;           // 2 ms

constexpr int PART_BYTES = TT * PART_STRIDE * 4;   // one tile's exchange rows (global scratch)
static_assert(PART_STRIDE % 4 == 0, "exchange rows of whole float4s");
constexpr int RUN_BYTES = TT * RUN_STRIDE * 4;     // one tile's running sums; two of them
// The same buffers first hold the tile's coefficients, copied in by the poster lane: post_prev
// [TT][4], pre_prev [TT][4], comb_prev [TT][16] (96 bytes per token, as many as the sums).
constexpr int COEF_PRE = TT * 16;
constexpr int COEF_COMB = TT * 32;
static_assert(COEF_COMB + TT * 64 <= RUN_BYTES, "coefficients fit a running-sum buffer");
constexpr int OFF_W = NSTAGE * STAGE_BYTES;
constexpr int OFF_PART = OFF_W + NW * STEP_WBLOCK_BYTES;
constexpr int OFF_BARS = OFF_PART + 2 * RUN_BYTES;
// full/empty/xready per X/F slot; wfull/wempty per weight entry; accready[2]; mposted[2];
// pfreed[2]; cfull[2]; drained; never
constexpr int NBARS = 3 * NSTAGE + 2 * NW + 10;
constexpr int OFF_TMEM = OFF_BARS + NBARS * 8;
// MXFP8 y: each thread's block-maximum exponent for its partner, [2 slot parities][2 parts][TT]
constexpr int OFF_XCH = OFF_TMEM + 16;
// a tile's S_y of each of a token's TPT parts, summed per token before it is posted, [TPT][TT]
constexpr int OFF_SYX = OFF_XCH + 4 * TT;
constexpr int SMEM_BYTES = OFF_SYX + 4 * TPT * TT + 1024;   // + slack for 1 KB alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(STAGE_BYTES % 1024 == 0 && STEP_WBLOCK_BYTES % 1024 == 0, "tile alignment");

__host__ __device__ constexpr int xtile(int b, int k) { return b * STAGE_BYTES + k * TILE_BYTES; }
__host__ __device__ constexpr int ftile(int b) { return b * STAGE_BYTES + 4 * TILE_BYTES; }
__host__ __device__ constexpr int wtile(int e, int k) {
  return OFF_W + e * STEP_WBLOCK_BYTES + k * STEP_WSTREAM_BYTES;
}
// y staging at the very end reuses the X/F tiles of the idle ring (slot j -> stage j/5, tile
// j%5) and, from j = 5 NSTAGE on, the idle weight ring, so the last R <= NYSLOTS slots of y are
// staged at once.
__host__ __device__ constexpr int yslot(int j) {
  return j < 5 * NSTAGE ? (j / 5) * STAGE_BYTES + (j % 5) * TILE_BYTES : OFF_W + (j - 5 * NSTAGE) * TILE_BYTES;
}
constexpr int NYSLOTS = 5 * NSTAGE + NW * STEP_WBLOCK_BYTES / TILE_BYTES;
static_assert(NW * STEP_WBLOCK_BYTES % TILE_BYTES == 0, "weight ring holds whole staging tiles");
static_assert(STASH_SLOTS <= NYSLOTS, "the stash's slots of y are staged in one batch");
constexpr int EB = 4;                   // stash slots the MXFP8 epilogue loads per TMEM wait
constexpr int GAIN_PER_THREAD = (MAX_SLICE + NCONS * 32 - 1) / (NCONS * 32);   // epilogue gains
static_assert(STASH_SLOTS < NYSLOTS, "the gains' staging tile is not a y staging tile");

struct StepParams {
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
  float* mixes_out;
  uint8_t* y_scale;            // MXFP8 y only: E8M0 block scales [N, d / 32]
  unsigned* status;
  unsigned long long* trace;   // optional: 8 phase timestamps per (tile, CTA) (mhc_set_trace)
  unsigned* counters;          // per group: pready[2] at 2, pfree[2] at 4 (zeroed per launch)
  // per group: [2 buffers][TT tokens][split ranks] tagged words {S_y of the token over the
  // rank's columns, tile iteration + 1} (zeroed per launch)
  unsigned long long* sytag;
  const unsigned long long* sytag_end;
  float* gpart;                // per group: [2 buffers][split ranks][TT tokens][PART_STRIDE]
  const float* gpart_end;      // end of the exchange area (bounds of the checked build)
  int N;
  int tt;                      // tokens per tile (a multiple of 8, <= TT); rows >= tt are idle
  int d;
  int split;
  int slice;
  int nsteps;
  int iters;
  float hc_eps;
  float norm_eps;
  float neg_zero;              // -0.0: the run-time zero addend of the rounded products (hc_arith.cuh)
  unsigned flags;
};

// Bounds checks of the checked build (MHC_CHECKED=1): the producer's copies, the X'/y stores,
// the exchange-area accesses, the finisher's stores and the MXFP8 scale stores test their
// indexes first; a failed test records STATUS_BOUNDS for mhc_get_status and the access is
// skipped (never a trap). Other builds compile the tests away.
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
// n floats at p lie inside the exchange area.
__device__ __forceinline__ bool in_gpart(const StepParams& P, const float* p, int n) {
  return p >= P.gpart && p + n <= P.gpart_end;
}
// Row offset planted by FLAG_PLANT_OOB (checked builds only): N rows past the end.
__device__ __forceinline__ int planted_rows(const StepParams& P, bool here) {
#if MHC_CHECKED
  return here && (P.flags & FLAG_PLANT_OOB) != 0 ? P.N : 0;
#else
  (void)P;
  (void)here;
  return 0;
#endif
}

// Fold accumulation group `gg` (TMEM accumulator gg & 1) into this thread's 12 running sums
// (the tile's first group sets them).
// The packed weight rows are ordered so that half h of the 24 mix numbers, all three planes,
// lands in accumulator columns [36h, 36h + 36): 12 hi, then 12 mid, then 12 lo.
__device__ __forceinline__ void fold_group(uint32_t tmem_lane, int gg, int h, float* run,
                                           bool first) {
  const uint32_t col = static_cast<uint32_t>((gg & 1) * ACC_COLS + 36 * h);
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
    const float4 v = first ? make_float4(0.f, 0.f, 0.f, 0.f) : rp[q];
    float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = 4 * q + e;
      vv[e] += (lo[r] + __uint_as_float(a[12 + r])) + __uint_as_float(a[r]);
    }
    rp[q] = make_float4(vv[0], vv[1], vv[2], vv[3]);
  }
}

// y = bf16(gain * (y_hat * r)) for 8 columns whose gains are g0, g1.
__device__ __forceinline__ uint4 rms_scale8(const uint32_t* w, float4 g0, float4 g1, f2 r2) {
  const f2 gp[4] = {f2{g0.x, g0.y}, f2{g0.z, g0.w}, f2{g1.x, g1.y}, f2{g1.z, g1.w}};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) o[e] = f2_to_bf2(mul2(gp[e], mul2(bf2_to_f2(w[e]), r2)));
  return make_uint4(o[0], o[1], o[2], o[3]);
}
// ... for the 8 columns starting at `col`.
__device__ __forceinline__ uint4 rms_scale8(const uint32_t* w, const float* __restrict__ gain,
                                            int col, f2 r2) {
  return rms_scale8(w, __ldg(reinterpret_cast<const float4*>(gain + col)),
                    __ldg(reinterpret_cast<const float4*>(gain + col + 4)), r2);
}

// MXFP8 y (OCP Microscaling formats v1.0: E4M3 elements, blocks of 32 features of a token that
// share one E8M0 scale 2^(floor(log2 amax) - 8)), encoded from the bf16 y: the codes equal an
// MXFP8 pass over the y that the bf16 path writes. A slot row is one block; each of the token's
// two consumer threads holds 16 of its features.
// This thread's 16 bf16 y values, packed in pairs: those of the bf16 path.
__device__ __forceinline__ void y_bf16x16(const uint32_t* w, const float4* g, f2 r2, uint32_t* y) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 v = rms_scale8(w + 4 * q, g[2 * q], g[2 * q + 1], r2);
    y[4 * q] = v.x;
    y[4 * q + 1] = v.y;
    y[4 * q + 2] = v.z;
    y[4 * q + 3] = v.w;
  }
}
// Biased exponent of the largest |y| of 16 bf16 values (0 for zeros and subnormals):
// floor(log2 amax) + 127. Non-negative bf16 bit patterns order like their values.
__device__ __forceinline__ uint32_t amax_exponent16(const uint32_t* y) {
  uint32_t m = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = max(m, max(y[k] & 0x7fffu, (y[k] >> 16) & 0x7fffu));
  return m >> 7;
}
// E8M0 code of a block whose largest magnitude has biased exponent e: floor(log2 amax) - 8 + 127,
// at least 0 (an all-zero block takes 0).
__device__ __forceinline__ uint32_t mx_scale_code(uint32_t e) { return e > 8 ? e - 8 : 0; }
// 16 bf16 values divided by the block scale 2^(code - 127) (a power of two: exact) and rounded to
// E4M3, nearest even, saturating at +-448; bytes in feature order.
__device__ __forceinline__ uint4 mx_encode16(const uint32_t* y, uint32_t code) {
  const float inv = __uint_as_float((254u - code) << 23);   // 2^(127 - code)
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p0 = y[2 * i], p1 = y[2 * i + 1];       // features 4i, 4i+1 | 4i+2, 4i+3
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__uint_as_float(p0 << 16) * inv, __uint_as_float(p0 & 0xffff0000u) * inv),
        __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__uint_as_float(p1 << 16) * inv, __uint_as_float(p1 & 0xffff0000u) * inv),
        __NV_SATFINITE, __NV_E4M3);
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Staging of one slot of E4M3 codes in shared memory: the codes of tile quarter q (tokens
// 32q .. 32q + 31, held by one pair of consumer warps) fill the first kilobyte of the 2 KB
// at base + 2048 q, [32 rows][32 bytes] with the 32-byte swizzle, so that each pair writes only
// bytes that it alone read before. One TMA store per full quarter (32-row boxes), 8-row boxes
// for the rows of a partial last quarter.
__device__ __forceinline__ uint32_t code_offset(int tl, int part) {
  return static_cast<uint32_t>((tl >> 5) * 2048) + swizzled_chunk_offset(tl & 31, part, 32);
}
__device__ __forceinline__ void store_codes(const CUtensorMap* m32, const CUtensorMap* m8,
                                            const uint8_t* base, int col, int row0, int rows,
                                            uint64_t pol) {
  for (int q = 0; 32 * q < rows; ++q) {
    const int n = min(32, rows - 32 * q);
    if (n == 32) {
      tma_store_2d_hint(m32, base + 2048 * q, col, row0 + 32 * q, pol);
    } else {
      for (int j = 0; j < n; j += 8)
        tma_store_2d_hint(m8, base + 2048 * q + 32 * j, col, row0 + 32 * q + j, pol);
    }
  }
}

// One pass's y_hat (PASS_COLS packed bf16 pairs) to or from the TMEM stash.
__device__ __forceinline__ void stash_load(uint32_t taddr, uint32_t (&w)[PASS_COLS]) { tmem_ld_x8(taddr, w); }
__device__ __forceinline__ void stash_load_nowait(uint32_t taddr, uint32_t (&w)[PASS_COLS]) {
  tmem_ld_x8_nowait(taddr, w);
}
__device__ __forceinline__ void stash_store(uint32_t taddr, const uint32_t (&w)[PASS_COLS]) { tmem_st_x8(taddr, w); }

// Persistent: group c of gridDim.x / split groups handles tiles c, c + #groups, ... The TMA ring,
// the accumulation groups and the barrier phases run on across tiles.
// FUSED: the whole step (else the mix numbers of X alone); MX: y as MXFP8 codes and scales.
template <bool FUSED, bool MX = false>
__global__ void __launch_bounds__(NTHREADS, 1)
    step_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_f,
                const __grid_constant__ CUtensorMap tm_xo, const __grid_constant__ CUtensorMap tm_y,
                const __grid_constant__ CUtensorMap tm_y8, const StepParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + OFF_BARS);
  uint64_t* empty = full + NSTAGE;
  uint64_t* xready = empty + NSTAGE;
  uint64_t* wfull = xready + NSTAGE;        // [NW]: the block in weight entry e has landed
  uint64_t* wempty = wfull + NW;            // [NW]: the MMAs that read weight entry e are done
  uint64_t* accready = wempty + NW;         // [2]: an accumulation group finished in buffer i
  uint64_t* mposted = accready + 2;         // [2]: the folding warps wrote a tile's mix sums
  uint64_t* pfreed = mposted + 2;           // [2]: the group's finishers released an exchange buffer
  uint64_t* cfull = pfreed + 2;             // [2]: a tile's coefficients are in its sums buffer
  uint64_t* drained = cfull + 2;            // the last X'/y stores have left the ring
  uint64_t* never = drained + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = P.split;
  const uint32_t g = blockIdx.x % split;              // rank within the group
  const int tt = P.tt;
  const int ntiles = (P.N + tt - 1) / tt;
  const int nclust = gridDim.x / split;               // groups
  const int c0 = blockIdx.x / split;                  // this CTA's group = its first tile
  // group exchange (global memory): counters and the partial sums of every rank
  unsigned* const pready = P.counters + 8 * c0 + 2;   // [2]: consumer warps that posted mix sums
  unsigned* const pfree = pready + 2;                 // [2]: finishers done reading a buffer
  auto gpart = [&](int pb, int rank) {
    return P.gpart + ((static_cast<size_t>(c0) * 2 + pb) * split + rank) * (TT * PART_STRIDE);
  };
  // the tagged S_y words of token row tl, rank 0 (the ranks follow)
  auto sytag = [&](int pb, int tl_) {
    return P.sytag + ((static_cast<size_t>(c0) * 2 + pb) * TT + tl_) * split;
  };
  const int col0 = static_cast<int>(g) * DC;          // first column of this CTA's slice
  const int cstride = DC * split;                     // stride between its slots' columns
  const int S = P.nsteps;                             // slots per tile
  const int G = (S + PG - 1) / PG;                    // accumulation groups per tile (the last
                                                      // may hold fewer slots)
  const int R = S + RLAG;                             // y_hat stash ring slots
  const int d = P.d;
  bool timed_out = false;
  auto limit = [&]() { return timed_out ? 0ull : WAIT_LIMIT_NS; };

  // optional phase trace, one record per (tile, rank): slot 0 absolute tile start; slots 1..6
  // ns since then: producer done, loop done, partials posted, (unused), finisher
  // done, consumers' tile end; slot 7 = SM id << 40 | ns to the kernel end.
  auto trace_rec = [&](int tile) -> unsigned long long* {
    return P.trace == nullptr ? nullptr : P.trace + 8ull * (static_cast<unsigned long long>(tile) * split + g);
  };

  if (threadIdx.x == 0) {
    for (int b = 0; b < NSTAGE; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], FUSED ? 2 : 1 + NCONS);
      mbar_init(&xready[b], NCONS);
    }
    for (int e = 0; e < NW; ++e) {
      mbar_init(&wfull[e], 1);
      mbar_init(&wempty[e], 1);
    }
    mbar_init(&accready[0], 1);
    mbar_init(&accready[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&mposted[i], NFOLD);
      mbar_init(&pfreed[i], 1);
      mbar_init(&cfull[i], 1);
    }
    mbar_init(drained, 1);
    mbar_init(never, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
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
      if (FUSED) {
        tma_prefetch_desc(&tm_f);
        tma_prefetch_desc(&tm_xo);
        tma_prefetch_desc(&tm_y);
      }
      const uint64_t stream_pol = policy_evict_first();
      const uint32_t bytes = (FUSED ? 5u : 4u) * static_cast<uint32_t>(tt * ROWB);   // tt-row boxes
      int gs = 0;
      for (int tile = c0; tile < ntiles; tile += nclust) {
        const int t0 = tile * tt;
        for (int s = 0; s < S; ++s, ++gs) {
          const int b = gs % NSTAGE;
          if (gs >= NSTAGE) {
            if (!mbar_wait(&empty[b], ((gs / NSTAGE) - 1) & 1, limit())) timed_out = true;
          }
          const int i0 = col0 + s * cstride;
          if (checked(i0 >= 0 && i0 + DC <= d && t0 >= 0 && t0 < P.N, P.status)) {
            mbar_arrive_expect_tx(&full[b], bytes);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tma_load_3d_hint(sm + xtile(b, k), &tm_x, &full[b], i0, k, t0, stream_pol);
            if (FUSED) tma_load_2d_hint(sm + ftile(b), &tm_f, &full[b], i0, t0, stream_pol);
          } else {
            mbar_arrive(&full[b]);      // the slot completes without data
          }
        }
        if (auto tr = trace_rec(tile)) tr[1] = global_timer_ns();
      }
    } else if (lane == 1) {
      // ---------------------------------------------------------------- poster
      // The CTA's link to its group's counters in global memory, so that no consumer warp waits
      // on an L2 round trip: a gpu-scope release waits for the writes to reach L2, and every
      // acquire load of a counter is an L2 round trip too, several microseconds each under full
      // memory load. Per tile, in order:
      //   1. (from the third tile) wait until the group's finishers have released exchange
      //      buffer it & 1, then tell the consumers (pfreed);
      //   2. once the folding warps wrote the tile's mix sums and S_x (mposted; every consumer
      //      warp folds), release pready.
      // (The tile's S_y goes to the group through tagged words the consumers post and poll
      // themselves.)
      // Causality runs through this lane: the peers' release, its acquire, its CTA-scope
      // arrive, the consumers' wait.
      // It also copies each tile's coefficients into the tile's running-sum buffer, one and a
      // half tiles ahead (the buffer of tile it + 2 is free once the folders posted tile it's
      // mix sums), so the consumers never wait on those loads at a tile start.
      const uint64_t coef_pol = policy_evict_first();
      auto coef_copy = [&](int it_) {
        const int tile = c0 + it_ * nclust;
        if (!FUSED || tile >= ntiles) return;
        const int t0 = tile * tt;
        const uint32_t cnt = static_cast<uint32_t>(min(tt, P.N - t0));
        uint8_t* buf = sm + OFF_PART + (it_ & 1) * RUN_BYTES;
        if (!checked(t0 >= 0 && cnt >= 1 && cnt <= static_cast<uint32_t>(TT) &&
                     t0 + static_cast<int>(cnt) <= P.N, P.status)) {
          mbar_arrive(&cfull[it_ & 1]);
          return;
        }
        mbar_arrive_expect_tx(&cfull[it_ & 1], cnt * 96u);
        bulk_load_hint(buf, P.post_prev + static_cast<size_t>(t0) * 4, cnt * 16u, &cfull[it_ & 1], coef_pol);
        bulk_load_hint(buf + COEF_PRE, P.pre_prev + static_cast<size_t>(t0) * 4, cnt * 16u, &cfull[it_ & 1], coef_pol);
        bulk_load_hint(buf + COEF_COMB, P.comb_prev + static_cast<size_t>(t0) * 16, cnt * 64u, &cfull[it_ & 1], coef_pol);
      };
      coef_copy(0);
      coef_copy(1);
      int it = 0;
      for (int tile = c0; tile < ntiles; tile += nclust, ++it) {
        if (it >= 2) {
          if (!gwait(&pfree[it & 1], static_cast<unsigned>((it >> 1) * split), limit()))
            timed_out = true;
          mbar_arrive(&pfreed[it & 1]);
        }
        if (!mbar_wait(&mposted[it & 1], (it >> 1) & 1, limit())) timed_out = true;
        gcount_release_n(&pready[it & 1], NFOLD);
        coef_copy(it + 2);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // It also runs the weight ring, whose only reader it is: global weight block u (block
    // u % HALVES of slot u / HALVES) goes to entry u % NW, and an entry is refilled with block
    // u + NW once the MMAs that read block u have completed. The X/F producer never waits on it.
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(MMA_M, STEP_MMA_N);
      const uint64_t weight_pol = policy_evict_last();
      const int nblocks = ((ntiles - c0 + nclust - 1) / nclust) * S * HALVES;
      auto load_block = [&](int u) {
        const int e = u % NW;
        const int slot_in_tile = (u / HALVES) % S;
        const int blk = (col0 + slot_in_tile * cstride) / WDC + u % HALVES;
        if (!checked(blk >= 0 && (blk + 1) * WDC <= d, P.status)) {
          mbar_arrive(&wfull[e]);
          return;
        }
        mbar_arrive_expect_tx(&wfull[e], STEP_WBLOCK_BYTES);
        bulk_load_hint(sm + wtile(e, 0), P.w_packed + static_cast<size_t>(blk) * STEP_WBLOCK_BYTES,
                       STEP_WBLOCK_BYTES, &wfull[e], weight_pol);
      };
      for (int u = 0; u < NW && u < nblocks; ++u) load_block(u);
      int gs = 0;
      for (int tile = c0, it = 0; tile < ntiles; tile += nclust, ++it) {
        for (int s = 0; s < S; ++s, ++gs) {
          const int b = gs % NSTAGE;
          if (!mbar_wait(FUSED ? &xready[b] : &full[b], (gs / NSTAGE) & 1, limit())) timed_out = true;
          tc_fence_after();
          // accumulation groups of PG slots (numbered across tiles) alternate between the two
          // accumulators
          const int gg = it * G + s / PG;
          const uint32_t acc = tmem + static_cast<uint32_t>((gg & 1) * ACC_COLS);
#pragma unroll
          for (int j = 0; j < HALVES; ++j) {
            const int u = gs * HALVES + j, e = u % NW;
            if (!mbar_wait(&wfull[e], (u / NW) & 1, limit())) timed_out = true;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t a0 = smem_u32(sm + xtile(b, k));
              const uint32_t b0 = smem_u32(sm + wtile(e, k));
#pragma unroll
              for (int kk = 0; kk < KSTEPS; ++kk) {
                umma_bf16(acc, sdesc_kmajor_swizzled(a0 + 32 * (j * KSTEPS + kk), ROWB),
                          sdesc_kmajor_swizzled(b0 + 32 * kk, STEP_WROW_BYTES), idesc,
                          (s % PG != 0 || j != 0 || k != 0 || kk != 0) ? 1u : 0u);
              }
            }
            umma_commit(&wempty[e]);
          }
          umma_commit(&empty[b]);
          if (s % PG == PG - 1 || s == S - 1) umma_commit(&accready[gg & 1]);
          // refill this slot's weight entries with the blocks NW ahead once its MMAs are done
#pragma unroll
          for (int j = 0; j < HALVES; ++j) {
            const int u = gs * HALVES + j;
            if (u + NW < nblocks) {
              if (!mbar_wait(&wempty[u % NW], (u / NW) & 1, limit())) timed_out = true;
              load_block(u + NW);
            }
          }
        }
      }
    }
  } else if (warp == STORE_WARP) {
    // ------------------------------------------------------------------ X'/y store issuer
    if (FUSED && lane == 0) {
      const uint64_t stream_pol = policy_evict_first();
      int gs = 0;
      for (int tile = c0; tile < ntiles; tile += nclust) {
        const int t0 = tile * tt;
        for (int s = 0; s < S; ++s, ++gs) {
          const int b = gs % NSTAGE;
          if (!mbar_wait(&xready[b], (gs / NSTAGE) & 1, limit())) timed_out = true;
          const int i0 = col0 + s * cstride;
          if (checked(i0 >= 0 && i0 + DC <= d && t0 >= 0 && t0 < P.N, P.status)) {
#pragma unroll
            for (int k = 0; k < 4; ++k) tma_store_3d_hint(&tm_xo, sm + xtile(b, k), i0, k, t0, stream_pol);
          }
          if (gs >= R) {
            // the y the consumers normalised into the F tile: global slot gs - R
            const int src = gs - R;
            const int ytile = c0 + (src / S) * nclust;
            const int ycol = col0 + (src % S) * cstride;
            if (checked(ycol >= 0 && ycol + DC <= d && ytile >= 0 && ytile * tt < P.N, P.status)) {
              if constexpr (MX)
                store_codes(&tm_y, &tm_y8, sm + ftile(b), ycol, ytile * tt, tt, stream_pol);
              else
                tma_store_2d_hint(&tm_y, sm + ftile(b), ycol, ytile * tt, stream_pol);
            }
          }
          bulk_commit();
          bulk_wait_read<0>();          // the slot's tiles have been read: free the slot
          mbar_arrive(&empty[b]);
        }
      }
    }
    if (lane == 0) mbar_arrive(drained);
  } else if (warp < STORE_WARP) {
    // ------------------------------------------------------------------ consumers
    const int c = warp - NROLE;
    const int sub = warp & 3;           // TMEM lane quarter this warp may access
    const int h = c >> 2;               // which of the quarter's two warps; a folder's 12 mix numbers
    const int tl = (sub % QPT) * 32 + lane;             // token row within a tile
    const int part = (sub / QPT) * 2 + h;               // which CPH chunks of each slot row
    const bool folder = sub < QPT;      // its TMEM lane holds the token's accumulator row
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    const int chunk0 = part * CPH;      // this thread's 16-byte chunks: chunk0 + q, q < CPH
    uint32_t row_off[CPH];
#pragma unroll
    for (int q = 0; q < CPH; ++q) row_off[q] = tile_chunk_offset(tl, chunk0 + q);
    // the y_hat stash, in this thread's own TMEM lane: a ring of R slots of PASS_COLS columns;
    // global slot gs uses ring slot gs % R
    const uint32_t stash = lane_base + STASH_COL + static_cast<uint32_t>(h * R * PASS_COLS);
    auto slot_addr = [&](int slot) { return stash + static_cast<uint32_t>(slot * PASS_COLS); };

    f2 cu[4], cc[4][4], cp[4];
    const f2 nz2{P.neg_zero, P.neg_zero};
    // this token's coefficients of tile iteration it_, from the tile's sums buffer (copied in by
    // the poster lane)
    auto load_coeffs = [&](int it_, int tile) {
      const int token = tile * tt + tl;
      const bool valid = FUSED && tl < tt && token < P.N;
      const bool row_dest = (P.flags & 1u) != 0;
      const float* buf = reinterpret_cast<const float*>(sm + OFF_PART + (it_ & 1) * RUN_BYTES);
      const float* cb = buf + tl * 4;
      const float* pb = buf + COEF_PRE / 4 + tl * 4;
      const float* mb = buf + COEF_COMB / 4 + tl * 16;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float uk = valid ? cb[k] : 0.f;
        const float pk = valid ? pb[k] : 0.f;
        cu[k] = f2{uk, uk};
        cp[k] = f2{pk, pk};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // cc[j][k]: coefficient of input stream j in output stream k
          const float v = valid ? mb[row_dest ? (k * 4 + j) : (j * 4 + k)] : 0.f;
          cc[j][k] = f2{v, v};
        }
      }
    };
    auto part_of = [&](int it_) {   // running sums of this thread for tile iteration it_
      return reinterpret_cast<float*>(sm + OFF_PART + (it_ & 1) * RUN_BYTES) + tl * RUN_STRIDE;
    };
    // RMS factor of tile iteration it_ for this token, from the group's tagged S_y words (one per
    // rank, tag it_ + 1). In two halves, so that the L2 round trip overlaps other work:
    // rms_issue loads the words of the last eight ranks (earlier ranks, if any, are summed at
    // once); rms_finish polls again any word whose tag was not there yet and adds them up, in
    // rank order. Rows at and past the tile height have no words and take no factor.
    float rms_sy = 0.f;
    uint64_t rms_w[8];
    auto rms_sum8 = [&](int it_, int rk0) {   // the words of ranks rk0.., polled until complete
      const uint32_t want = static_cast<uint32_t>(it_) + 1u;
      const unsigned long long* row = sytag(it_ & 1, tl) + rk0;
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        v[u] = 0.f;
        if (rk0 + u < split && tl < tt && (!MHC_CHECKED || (row + u >= P.sytag && row + u < P.sytag_end))) {
          uint64_t w = rms_w[u];
          if (word_tag(w) != want) {
            const uint64_t t0 = global_timer_ns();
            const uint64_t lim = limit();
            do {
              w = tagged_load(row + u);
              if (word_tag(w) == want) break;
              if (global_timer_ns() - t0 > lim) {
                timed_out = true;
                break;
              }
            } while (true);
          }
          v[u] = word_value(w);
        }
      }
      return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    };
    auto rms_load8 = [&](int it_, int rk0) {
      const unsigned long long* row = sytag(it_ & 1, tl) + rk0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        rms_w[u] = 0;
        if (rk0 + u < split && tl < tt && checked(row + u >= P.sytag && row + u < P.sytag_end, P.status))
          rms_w[u] = tagged_load(row + u);
      }
    };
    int rms_last = 0;                      // first rank of the words loaded by rms_issue
    auto rms_issue = [&](int it_) {
      rms_sy = 0.f;
      for (int rk0 = 0; rk0 < split; rk0 += 8) {
        if (rk0 > 0) rms_sy += rms_sum8(it_, rk0 - 8);
        rms_load8(it_, rk0);
        rms_last = rk0;
      }
    };
    auto rms_finish = [&](int it_) {
      const float sy = rms_sy + rms_sum8(it_, rms_last);
      const float r = __frsqrt_rn(__fdiv_rn(sy, static_cast<float>(d)) + P.norm_eps);
      return f2{r, r};
    };
    // fold accumulation group gg (global numbering) into its tile's running sums; after a
    // tile's last group, post the tile's partials to the group
    auto fold = [&](int gg) {
      if (!mbar_wait(&accready[gg & 1], (gg >> 1) & 1, limit())) timed_out = true;
      tc_fence_after();
      const int it_ = gg / G;
      float* run = part_of(it_) + 12 * h;
      fold_group(lane_base, gg, h, run, gg % G == 0);
      if (gg % G == G - 1) {
        // this thread's 12 mix sums of the tile are final: publish them to the group (the
        // counter's release orders what the warp wrote before __syncwarp)
        float4* dst = reinterpret_cast<float4*>(gpart(it_ & 1, g) + tl * PART_STRIDE + 12 * h);
        const float4* src = reinterpret_cast<const float4*>(run);
        if (checked(in_gpart(P, reinterpret_cast<const float*>(dst), 12), P.status)) {
          dst[0] = src[0];
          dst[1] = src[1];
          dst[2] = src[2];
        }
        // the sums buffer is free now: the poster's bulk copy of a later tile's coefficients
        // will write it (async proxy after these generic accesses)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&mposted[it_ & 1]);   // published by the poster (warp 0)
        if (warp == NROLE && lane == 0) {
          if (auto tr = trace_rec(c0 + it_ * nclust)) tr[3] = global_timer_ns() - tr[0];
        }
      }
    };

    // RMS factors: r_old for tile it-2 (consumed in slots s < RLAG), r_new for tile it-1 (from
    // slot RLAG on; computed after slot RLAG - 1)
    f2 r_old{0.f, 0.f}, r_new{0.f, 0.f};
    int gs = 0, it = 0, folded = 0;
    int slot = 0;                        // gs % R, kept incrementally
    // this token's coefficients of tile iteration it_, once the poster's copy has landed
    auto take_coeffs = [&](int it_) {
      const int tile = c0 + it_ * nclust;
      if (!FUSED || tile >= ntiles) return;
      if (!mbar_wait(&cfull[it_ & 1], (it_ >> 1) & 1, limit())) timed_out = true;
      load_coeffs(it_, tile);
    };
    take_coeffs(0);
    for (int tile = c0; tile < ntiles; tile += nclust, ++it) {
      unsigned long long* tr = trace_rec(tile);
      if (warp == NROLE && lane == 0 && tr) tr[0] = global_timer_ns();
      r_old = r_new;
      // tokens of the y written in this tile's slots: tile it-1's from slot RLAG on, before that
      // tile it-2's
      const int ytok1 = (tile - nclust) * tt + tl, ytok2 = (tile - 2 * nclust) * tt + tl;

      f2 sx2{0.f, 0.f}, sy2{0.f, 0.f};
      for (int s = 0; s < S; ++s, ++gs) {
        const int b = gs % NSTAGE;
        // the ring slot this slot writes holds the y_hat of global slot gs - R (tile it-1, or
        // it-2 in slots s < RLAG): read it now, normalise it into the F tile once F has been read; the
        // store warp writes it out with this slot's X'
        const bool consume = FUSED && gs >= R;
        uint32_t prev[PASS_COLS];
        if (consume) stash_load_nowait(slot_addr(slot), prev);
        if (!mbar_wait(&full[b], (gs / NSTAGE) & 1, limit())) timed_out = true;
        if (consume) tmem_ld_wait();
        f2 lx{0.f, 0.f};   // this slot's sum of squares, added to the running sum once
        if (FUSED) {
          const int ycol = col0 + (s >= RLAG ? s - RLAG : s + S - RLAG) * cstride;   // slot of gs - R
          f2 ly{0.f, 0.f};
          {
            uint32_t ywall[PASS_COLS];
#pragma unroll
            for (int q = 0; q < CPH; ++q) {
              uint32_t xw[4][4], fw[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint4 v = *reinterpret_cast<const uint4*>(sm + xtile(b, k) + row_off[q]);
                xw[k][0] = v.x;
                xw[k][1] = v.y;
                xw[k][2] = v.z;
                xw[k][3] = v.w;
              }
              {
                const uint4 v = *reinterpret_cast<const uint4*>(sm + ftile(b) + row_off[q]);
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
                  // X'_k: rounded products summed in stream order (hc_arith.cuh)
                  const f2 ck[4] = {cc[0][k], cc[1][k], cc[2][k], cc[3][k]};
                  ow[k][w] = f2_to_bf2(hc_post_pair(ck, cu[k], x, f, nz2));
                  xp[k] = bf2_to_f2(ow[k][w]);
                  lx = fma2(xp[k], xp[k], lx);
                }
                ywall[4 * q + w] = f2_to_bf2(hc_pre_pair(cp, xp, nz2));
                const f2 yr = bf2_to_f2(ywall[4 * q + w]);
                ly = fma2(yr, yr, ly);
              }
#pragma unroll
              for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4*>(sm + xtile(b, k) + row_off[q]) =
                    make_uint4(ow[k][0], ow[k][1], ow[k][2], ow[k][3]);
            }
            stash_store(slot_addr(slot), ywall);
          }
          // the previous tile's RMS factor: its loads were issued after slot RLAG - 1
          if (s == RLAG && it > 0) r_new = rms_finish(it - 1);
          if (consume) {
            // y of global slot gs - R into the F tile (read above)
            const f2 r_src = s >= RLAG ? r_new : r_old;
            if constexpr (MX) {
              // the block's scale needs the partner thread's maximum (the other warp of this
              // TMEM quarter); after their barrier both have also read their F rows, which then
              // take the quarter's codes (code_offset)
              uint32_t yv[8];
              float4 gv[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                gv[i] = __ldg(reinterpret_cast<const float4*>(P.gain + ycol + chunk0 * 8) + i);
              y_bf16x16(prev, gv, r_src, yv);
              const uint32_t e_own = amax_exponent16(yv);
              uint8_t* xch = sm + OFF_XCH + (gs & 1) * (2 * TT);
              xch[part * TT + tl] = static_cast<uint8_t>(e_own);
              named_bar_sync(3 + sub, 64);   // the quarter's two warps (ids 3..6)
              const uint32_t code = mx_scale_code(max(e_own, static_cast<uint32_t>(xch[(part ^ 1) * TT + tl])));
              *reinterpret_cast<uint4*>(sm + ftile(b) + code_offset(tl, part)) = mx_encode16(yv, code);
              const int token = s >= RLAG ? ytok1 : ytok2;
              if (part == 0 && tl < tt && token < P.N) {
                const int row = token + planted_rows(P, blockIdx.x == 0 && tl == 0 && gs == R);
                if (checked(row >= 0 && row < P.N && ycol >= 0 && ycol + DC <= d, P.status))
                  P.y_scale[static_cast<size_t>(row) * (P.d / 32) + ycol / 32] = static_cast<uint8_t>(code);
              }
            } else {
#pragma unroll
              for (int q = 0; q < CPH; ++q)
                *reinterpret_cast<uint4*>(sm + ftile(b) + row_off[q]) =
                    rms_scale8(prev + 4 * q, P.gain, ycol + (chunk0 + q) * 8, r_src);
            }
          }
          sy2 = add2(sy2, ly);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&xready[b]);
        } else {
#pragma unroll
          for (int q = 0; q < CPH; ++q) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 v = *reinterpret_cast<const uint4*>(sm + xtile(b, k) + row_off[q]);
              const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const f2 x = bf2_to_f2(wv[w]);
                lx = fma2(x, x, lx);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[b]);
        }
        sx2 = add2(sx2, lx);
        slot = slot + 1 == R ? 0 : slot + 1;
        // Fold group q in the last slot of group q+1 (global numbering, across tiles): the MMA
        // that reuses q's accumulator (group q+2) starts only after this warp's xready of a
        // later slot.
        if (folder && (s % PG == PG - 1 || s == S - 1) && it * G + s / PG >= 1) fold(folded++);
        // the previous tile's RMS factor, needed from slot RLAG on: its loads are issued after
        // slot RLAG-1's work is published and summed in slot RLAG after the X' work
        if (FUSED && s == RLAG - 1 && it > 0) rms_issue(it - 1);
      }
      if (FUSED) tmem_wait_st();
      if (tr && warp == NROLE && lane == 0) tr[2] = global_timer_ns() - tr[0];
      take_coeffs(it + 1);

      // ------------------------------------------------------------ post this slice's sums
      // S_y: the token's two parts are added (part 0 + part 1, through shared memory between
      // the two warps of this TMEM quarter) and posted as one tagged word, tag it + 1, which
      // the group's consumers poll from slot RLAG - 1 of their next tile. Its buffer it & 1 is
      // rewritten two tiles later, after every rank has read it: no rank gets past slot RLAG of
      // tile it + 1 before all ranks posted tile it, which they do after reading tile it - 1.
      if (FUSED) {
        float* syx = reinterpret_cast<float*>(sm + OFF_SYX);
        syx[part * TT + tl] = sy2.x + sy2.y;
        named_bar_sync(3 + sub, 64);
        if (part == 0 && tl < tt) {
          unsigned long long* w = sytag(it & 1, tl) + g;
          if (checked(w >= P.sytag && w < P.sytag_end, P.status))
            tagged_store(w, syx[tl] + syx[TT + tl], static_cast<uint32_t>(it) + 1u);
        }
        named_bar_sync(3 + sub, 64);      // syx is free for the next tile
      }
      // exchange row layout: [0..23] mix sums (folder half h owns 12h..12h+11), [24 + part] S_x.
      // The group buffer it & 1 was last read (by every finisher) two tiles ago.
      if (it >= 2 && !mbar_wait(&pfreed[it & 1], ((it >> 1) - 1) & 1, limit())) timed_out = true;
      {
        float* pt = gpart(it & 1, g) + tl * PART_STRIDE;
        if (checked(in_gpart(P, pt, PART_STRIDE), P.status)) pt[24 + part] = sx2.x + sx2.y;
      }
      __syncwarp();
      if (tr && warp == NROLE && lane == 0) tr[6] = global_timer_ns() - tr[0];
    }

    // ---------------------------------------------------------------- after the last tile
    const int ngroups_total = it * G;
    while (folder && folded < ngroups_total) fold(folded++);
    if (FUSED && it > 0) {
      // y still in the stash: the last R global slots (tile it-1's slots and, before them, the
      // last RLAG slots of tile it-2)
      // The gains of the CTA's S column blocks go to the last staging tile, in the idle weight
      // ring (this thread has folded the last group, so every MMA is done); their loads are in
      // flight during the RMS-factor wait.
      float* gsm = reinterpret_cast<float*>(sm + yslot(NYSLOTS - 1));
      const int ct = static_cast<int>(threadIdx.x) - NROLE * 32;
      float gl[GAIN_PER_THREAD];
#pragma unroll
      for (int k = 0; k < GAIN_PER_THREAD; ++k) {
        const int i = ct + k * NCONS * 32;
        gl[k] = i < S * DC ? __ldg(P.gain + col0 + (i / DC) * cstride + i % DC) : 0.f;
      }
      rms_issue(it - 1);
      const f2 r_last = rms_finish(it - 1);
      const f2 r_before = r_new;    // tile it-2's factor (computed during tile it-1)
#pragma unroll
      for (int k = 0; k < GAIN_PER_THREAD; ++k) {
        const int i = ct + k * NCONS * 32;
        if (i < S * DC) gsm[i] = gl[k];
      }
      if (!mbar_wait(drained, 0, limit())) timed_out = true;   // the ring is idle now
      named_bar_sync(1, NCONS * 32);                            // and the gains are in place
      const uint64_t stream_pol = policy_evict_first();
      const int first = std::max(0, gs - R);
      const int boundary = (it - 1) * S;    // slots below it are tile it-2's
      int ring = first % R, sidx = first % S;
      for (int g0 = first; g0 < gs; g0 += NYSLOTS) {
        const int g1 = std::min(gs, g0 + NYSLOTS);
        if constexpr (MX) {
          // EB stash slots per TMEM wait. As in the main loop, the block maxima go through the
          // spare kilobyte of each staged slot's quarter: one pair barrier per EB slots.
          for (int b0 = g0; b0 < g1; b0 += EB) {
            uint32_t w[EB][PASS_COLS], yv[EB][8], e_own[EB], col[EB];
#pragma unroll
            for (int e = 0; e < EB; ++e) {
              col[e] = 0;
              if (b0 + e < g1) {
                stash_load_nowait(slot_addr(ring), w[e]);
                col[e] = sidx;
                ring = ring + 1 == R ? 0 : ring + 1;
                sidx = sidx + 1 == S ? 0 : sidx + 1;
              }
            }
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < EB; ++e) {
              const int src = b0 + e;
              if (src < g1) {
                y_bf16x16(w[e], reinterpret_cast<const float4*>(gsm + col[e] * DC + chunk0 * 8),
                          src >= boundary ? r_last : r_before, yv[e]);
                e_own[e] = amax_exponent16(yv[e]);
                sm[yslot(src - g0) + sub * 2048 + 1024 + part * 32 + lane] = static_cast<uint8_t>(e_own[e]);
              }
            }
            named_bar_sync(3 + sub, 64);
#pragma unroll
            for (int e = 0; e < EB; ++e) {
              const int src = b0 + e;
              if (src < g1) {
                const uint32_t other = sm[yslot(src - g0) + sub * 2048 + 1024 + (part ^ 1) * 32 + lane];
                const uint32_t code = mx_scale_code(max(e_own[e], other));
                *reinterpret_cast<uint4*>(sm + yslot(src - g0) + code_offset(tl, part)) = mx_encode16(yv[e], code);
                const int token = (c0 + (src / S) * nclust) * tt + tl;
                const int scol = col0 + static_cast<int>(col[e]) * cstride;
                const int row = token + planted_rows(P, blockIdx.x == 0 && tl == 0 && src == first);
                if (part == 0 && tl < tt && token < P.N &&
                    checked(row >= 0 && row < P.N && scol >= 0 && scol + DC <= d, P.status))
                  P.y_scale[static_cast<size_t>(row) * (P.d / 32) + scol / 32] = static_cast<uint8_t>(code);
              }
            }
          }
        } else {
          for (int src = g0; src < g1; ++src) {
            uint32_t w[PASS_COLS];
            stash_load(slot_addr(ring), w);
            const float4* gp = reinterpret_cast<const float4*>(gsm + sidx * DC + chunk0 * 8);
            const f2 r = src >= boundary ? r_last : r_before;
#pragma unroll
            for (int q = 0; q < CPH; ++q)
              *reinterpret_cast<uint4*>(sm + yslot(src - g0) + row_off[q]) =
                  rms_scale8(w + 4 * q, gp[2 * q], gp[2 * q + 1], r);
            ring = ring + 1 == R ? 0 : ring + 1;
            sidx = sidx + 1 == S ? 0 : sidx + 1;
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, NCONS * 32);
        if constexpr (MX) {
          // four or more stores per staged slot: every consumer warp issues those of every
          // NCONS-th slot (measured 10% faster at 4,096 tokens than one issuing thread)
          if (lane == 0) {
            for (int src = g0 + (warp - NROLE); src < g1; src += NCONS) {
              const int ytile = c0 + (src / S) * nclust;
              const int ycol = col0 + (src % S) * cstride;
              if (checked(ycol >= 0 && ycol + DC <= d && ytile >= 0 && ytile * tt < P.N, P.status))
                store_codes(&tm_y, &tm_y8, sm + yslot(src - g0), ycol, ytile * tt, tt, stream_pol);
            }
            bulk_commit();
            bulk_wait_read<0>();
          }
        } else if (warp == NROLE && lane == 0) {
          for (int src = g0; src < g1; ++src) {
            const int ytile = c0 + (src / S) * nclust;
            const int ycol = col0 + (src % S) * cstride;
            if (checked(ycol >= 0 && ycol + DC <= d && ytile >= 0 && ytile * tt < P.N, P.status))
              tma_store_2d_hint(&tm_y, sm + yslot(src - g0), ycol, ytile * tt, stream_pol);
          }
          bulk_commit();
          bulk_wait_read<0>();
        }
        named_bar_sync(1, NCONS * 32);
      }
    }
  } else {
    // ------------------------------------------------------------------ finisher
    // Tokens [g*per, (g+1)*per) of each tile: scale, split, Sinkhorn. Two layouts, by tokens per
    // CTA (uniform over the launch):
    //   * per >= 8: the finisher runs beside the main loop, so it is kept lean. 16 tokens per
    //     pass; lane 4q + j serves tokens q and q + 8 and owns comb row j; it sums, rank by rank,
    //     only the 16 partial sums its row needs; the token's four lanes run Sinkhorn together
    //     (split_sinkhorn_row, shuffles for the column sums).
    //   * per < 8: few tokens per CTA, the finisher is on the critical path. TP tokens per pass
    //     (up to 8), L = 32 / TP lanes per token: lane r of a token adds the rows of ranks r,
    //     r + L, ... (two ranks' loads in flight at a time), a shuffle butterfly combines the L
    //     sums (the same total in every lane), and every lane runs the whole Sinkhorn
    //     (split_sinkhorn_all, no shuffle latency); lanes r < 4 write row r.
    // the split parameters, read by every token's split: into L1 before the first tile
    if (lane < 24) prefetch_l1(P.base + lane);
    if (lane == 24) prefetch_l1(P.scale);
    const int q = lane >> 2;
    const int j = lane & 3;
    const int per = tt / split;
    int TP = 8;
    while (TP > 1 && TP > per) TP >>= 1;
    const int L = 32 / TP;
    const int lq = lane / L;
    const int lr = lane % L;
    int it = 0;
    for (int tile = c0; tile < ntiles; tile += nclust, ++it) {
      const int pb = it & 1;
      if (!gwait(&pready[pb], static_cast<unsigned>(((it >> 1) + 1) * split * NFOLD), limit()))
        timed_out = true;
      const int t0 = tile * tt;
      if (per >= 8) {
        // 16 tokens per pass (two per lane group); after the last pass's reads the peers may
        // reuse their partials buffers
        for (int base_t = 0; base_t < per; base_t += 16) {
          float4 s0[2], s1[2], s2[2], s6[2];
          int tl2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            s0[u] = s1[u] = s2[u] = s6[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            tl2[u] = static_cast<int>(g) * per + min(base_t + 8 * u + q, per - 1);
          }
          // two ranks' rows of both tokens in flight per round trip; added in rank order
          for (int rk = 0; rk < split; rk += 2) {
            float4 v[2][2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
              for (int o = 0; o < 2; ++o) {
                const float4* row = reinterpret_cast<const float4*>(
                    gpart(pb, min(rk + o, split - 1)) + tl2[u] * PART_STRIDE);
                if (!checked(in_gpart(P, reinterpret_cast<const float*>(row), PART_STRIDE), P.status)) {
                  v[u][o][0] = v[u][o][1] = v[u][o][2] = v[u][o][3] = make_float4(0.f, 0.f, 0.f, 0.f);
                  continue;
                }
                v[u][o][0] = __ldcg(row);
                v[u][o][1] = __ldcg(row + 1);
                v[u][o][2] = __ldcg(row + 2 + j);
                v[u][o][3] = __ldcg(row + 6);
              }
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
              for (int o = 0; o < 2; ++o) {
                if (rk + o >= split) continue;
                const float4 v0 = v[u][o][0], v1 = v[u][o][1], v2 = v[u][o][2], v6 = v[u][o][3];
                s0[u].x += v0.x; s0[u].y += v0.y; s0[u].z += v0.z; s0[u].w += v0.w;
                s1[u].x += v1.x; s1[u].y += v1.y; s1[u].z += v1.z; s1[u].w += v1.w;
                s2[u].x += v2.x; s2[u].y += v2.y; s2[u].z += v2.z; s2[u].w += v2.w;
                s6[u].x += TPT == 4 ? (v6.x + v6.y) + (v6.z + v6.w) : v6.x + v6.y;   // S_x parts
              }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int tk = base_t + 8 * u + q;
            const bool in_range = tk < per;
            const int token2 = t0 + static_cast<int>(g) * per + tk;
            const float rs = __frsqrt_rn(__fdiv_rn(s6[u].x, static_cast<float>(4 * d)) + P.norm_eps);
            const float m0[4] = {s0[u].x * rs, s0[u].y * rs, s0[u].z * rs, s0[u].w * rs};
            const float m1[4] = {s1[u].x * rs, s1[u].y * rs, s1[u].z * rs, s1[u].w * rs};
            const float mrow[4] = {s2[u].x * rs, s2[u].y * rs, s2[u].z * rs, s2[u].w * rs};
            float pj, uj, crow[4];
            split_sinkhorn_row(mrow, m0[j], m1[j], j, __ldg(P.scale), __ldg(P.scale + 1),
                               __ldg(P.scale + 2), P.base, P.iters, P.hc_eps, pj, uj, crow);
            const int row = token2 + planted_rows(P, blockIdx.x == 0 && it == 0 && base_t == 0 && u == 0 && q == 0);
            if (in_range && token2 < P.N && checked(row >= 0 && row < P.N, P.status)) {
              P.pre_out[static_cast<size_t>(row) * 4 + j] = pj;
              P.post_out[static_cast<size_t>(row) * 4 + j] = uj;
              reinterpret_cast<float4*>(P.comb_out + static_cast<size_t>(row) * 16)[j] =
                  make_float4(crow[0], crow[1], crow[2], crow[3]);
              if (P.mixes_out != nullptr) {
                float4* mo = reinterpret_cast<float4*>(P.mixes_out + static_cast<size_t>(row) * 24);
                mo[2 + j] = make_float4(mrow[0], mrow[1], mrow[2], mrow[3]);
                if (j == 0) mo[0] = make_float4(m0[0], m0[1], m0[2], m0[3]);
                if (j == 1) mo[1] = make_float4(m1[0], m1[1], m1[2], m1[3]);
              }
            }
          }
        }
      } else {
        for (int base_t = 0; base_t < per; base_t += TP) {
          const int tt_ = base_t + lq;
          const bool in_range = tt_ < per;
          const int tl2 = static_cast<int>(g) * per + min(tt_, per - 1);
          constexpr int NACC = 24 + TPT;   // 24 mix sums, then the S_x parts
          constexpr int NV = PART_STRIDE / 4;
          float acc[NACC];
#pragma unroll
          for (int e = 0; e < NACC; ++e) acc[e] = 0.f;
          for (int rk = lr; rk < split; rk += 2 * L) {
            const bool two = rk + L < split;
            const float4* r0 = reinterpret_cast<const float4*>(gpart(pb, rk) + tl2 * PART_STRIDE);
            const float4* r1 = reinterpret_cast<const float4*>(gpart(pb, two ? rk + L : rk) + tl2 * PART_STRIDE);
            if (!checked(in_gpart(P, reinterpret_cast<const float*>(r0), PART_STRIDE) &&
                             in_gpart(P, reinterpret_cast<const float*>(r1), PART_STRIDE), P.status))
              continue;
            float4 v0[NV], v1[NV];
#pragma unroll
            for (int e = 0; e < NV; ++e) {
              v0[e] = __ldcg(r0 + e);
              v1[e] = two ? __ldcg(r1 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int e = 0; e < NV; ++e) {
              const float a4[4] = {v0[e].x + v1[e].x, v0[e].y + v1[e].y, v0[e].z + v1[e].z, v0[e].w + v1[e].w};
#pragma unroll
              for (int c = 0; c < 4; ++c)
                if (4 * e + c < NACC) acc[4 * e + c] += a4[c];
            }
          }
          for (int off = 1; off < L; off <<= 1)
#pragma unroll
            for (int e = 0; e < NACC; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
          const int token2 = t0 + static_cast<int>(g) * per + tt_;
          float sxt = 0.f;
#pragma unroll
          for (int e = 24; e < NACC; ++e) sxt += acc[e];
          const float rs = __frsqrt_rn(__fdiv_rn(sxt, static_cast<float>(4 * d)) + P.norm_eps);
          float m[24];
#pragma unroll
          for (int e = 0; e < 24; ++e) m[e] = acc[e] * rs;
          float pv[4], uv[4], cv[16];
          split_sinkhorn_all(m, __ldg(P.scale), __ldg(P.scale + 1), __ldg(P.scale + 2), P.base,
                             P.iters, P.hc_eps, pv, uv, cv);
          // lane r < 4 writes row r
          const int jr = lr & 3;
          const float pj = jr == 0 ? pv[0] : jr == 1 ? pv[1] : jr == 2 ? pv[2] : pv[3];
          const float uj = jr == 0 ? uv[0] : jr == 1 ? uv[1] : jr == 2 ? uv[2] : uv[3];
          float crow[4], mrow[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            crow[k] = jr == 0 ? cv[k] : jr == 1 ? cv[4 + k] : jr == 2 ? cv[8 + k] : cv[12 + k];
            mrow[k] = jr == 0 ? m[8 + k] : jr == 1 ? m[12 + k] : jr == 2 ? m[16 + k] : m[20 + k];
          }
          const int row = token2 + planted_rows(P, blockIdx.x == 0 && it == 0 && base_t == 0 && lq == 0);
          if (in_range && lr < 4 && token2 < P.N && checked(row >= 0 && row < P.N, P.status)) {
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
      }
      // every read of exchange buffer pb is done: the group may reuse it for tile it + 2 (if
      // any). Released after the tile's outputs, off the path to them: the release waits for
      // this lane's earlier memory operations.
      if (tile + 2 * nclust < ntiles) {
        __syncwarp();
        if (lane == 0) gcount_release(&pfree[pb]);
      }
      if (lane == 0) {
        if (auto tr = trace_rec(tile)) tr[5] = global_timer_ns();
      }
    }
  }

  if ((P.flags & 2u) != 0 && threadIdx.x == 0) {
    if (!mbar_wait(never, 0, DEBUG_WAIT_NS)) timed_out = true;
  }
  if (timed_out) atomicOr(P.status, STATUS_TIMEOUT);

  // ------------------------------------------------------------------ leave together
  // (every warp, all its lanes included, has arrived: the TMEM is free after this)
  tc_fence_before();
  block_sync();
  if (threadIdx.x == 0 && P.trace != nullptr) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    for (int tile = c0; tile < ntiles; tile += nclust) {
      unsigned long long* tr = trace_rec(tile);
      const unsigned long long t_tile = tr[0];
      tr[1] -= t_tile;
      tr[5] -= t_tile;
      tr[7] = (static_cast<unsigned long long>(smid) << 40) | (global_timer_ns() - t_tile);
    }
  }
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// host side

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  constexpr CUtensorMapSwizzle swz = ROWB == 32   ? CU_TENSOR_MAP_SWIZZLE_32B
                                     : ROWB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// MXFP8 codes of y [N, d], one byte each: boxes of DC bytes x box_rows, 32-byte swizzle.
bool map_codes(CUtensorMap* m, const void* p, int64_t N, int d, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N)};
  const cuuint64_t str[1] = {static_cast<cuuint64_t>(d)};
  const cuuint32_t box[2] = {DC, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(p), dims, str, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool map_streams(CUtensorMap* m, const void* p, int64_t N, int d, uint32_t box_rows) {   // [N, 4, d]
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), 4, static_cast<cuuint64_t>(N)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 8};
  const cuuint32_t box[3] = {DC, 1, box_rows};
  return make_map(m, p, 3, dims, str, box);
}
bool map_rows(CUtensorMap* m, const void* p, int64_t rows, int64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t str[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {DC, box_rows};
  return make_map(m, p, 2, dims, str, box);
}


// CTAs of the step kernel the current device holds at once (one per SM), cached per device.
template <typename Kern>
cudaError_t resident_ctas(Kern kern, int* ctas) {
  constexpr int kDevices = 64;
  static std::atomic<int> cache[3][kDevices] = {};
  const int which = (kern == step_kernel<true>) ? 1 : (kern == step_kernel<true, true>) ? 2 : 0;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
  const int cached = cache[which][dev].load(std::memory_order_relaxed);
  if (cached > 0) {
    *ctas = cached;
    return cudaSuccess;
  }
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NTHREADS, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cache[which][dev].store(sms * per_sm, std::memory_order_relaxed);
  *ctas = sms * per_sm;
  return cudaSuccess;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

bool split_ok(int d, int s) {
  // slices of whole slots, at least 128 columns (the previous tile's RMS factor
  // is taken after slot RLAG - 1), and a stash ring of S + RLAG slots that fits TMEM
  return d > 0 && s >= 1 && s <= kMaxSplit && d % (DC * s) == 0 && d / s <= MAX_SLICE &&
         d / s >= 4 * WDC;
}

int choose_split(int d, int forced) {
  if (forced != 0) return split_ok(d, forced) ? forced : 0;
  for (int s = 1; s <= kMaxSplit; s *= 2)
    if (split_ok(d, s)) return s;
  return 0;
}

StepShape choose_shape(int64_t N, int d, int ctas, int forced_split, int forced_tile) {
  // Every tile runs d / (DC * split) pipeline slots, each costing about (tt + kTileCostTokens)
  // tokens' worth of time; a group handles ceil(tiles / groups) tiles. Minimise the busiest
  // group's total; ties go to the smaller split and then the taller tile.
  StepShape best{0, 0, 0};
  int64_t best_cost = INT64_MAX;
  const int64_t n = std::max<int64_t>(N, 1);
  for (int s = 1; s <= kMaxSplit; s *= 2) {
    if ((forced_split != 0 && s != forced_split) || !split_ok(d, s) || ctas < s) continue;
    const int groups = ctas / s;
    const int64_t slots = d / (DC * s);
    for (int tt = TT; tt >= 8; tt -= 8) {
      if ((forced_tile != 0 && tt != forced_tile) || tt % s != 0) continue;
      const int64_t tiles = (n + tt - 1) / tt;
      const int64_t rounds = (tiles + groups - 1) / groups;
      const int64_t cost = rounds * slots * (tt + kTileCostTokens);
      if (cost < best_cost) {
        best_cost = cost;
        best = StepShape{s, tt, static_cast<int>(std::min<int64_t>(tiles, groups))};
      }
    }
  }
  return best;
}

size_t step_scratch_bytes() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  // per CTA (at most one per SM): its group's counters (32 bytes, shared by the group), two
  // buffers of its tagged S_y words and two of its partial sums
  return 256 + static_cast<size_t>(sms) * (32 + 2 * TT * 8 + 2 * PART_BYTES);
}

cudaError_t launch_step(bool fused, const StepArgs& a, cudaStream_t stream) {
  const bool mx = fused && a.y_scale != nullptr;
  // small batches: one thread-block cluster per tile (cluster.cu)
  if (const int cl = cluster_path(a.N, a.d, a.flags, fused && !mx)) return launch_cluster_step(a, cl, stream);
  if ((a.flags & FLAG_PATH_CLUSTER) != 0) return cudaErrorInvalidConfiguration;
  auto kern = mx ? step_kernel<true, true> : fused ? step_kernel<true> : step_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int ctas = 0;
  e = resident_ctas(kern, &ctas);
  if (e != cudaSuccess) return e;
  const StepShape shape = choose_shape(a.N, a.d, ctas, split_flag_value(a.flags), tile_flag(a.flags));
  if (shape.split == 0) return cudaErrorInvalidConfiguration;
  const int split = shape.split;
  const int tt = shape.tt;
  const int ngroups = std::max(1, shape.groups);
  const int tiles = static_cast<int>((a.N + tt - 1) / tt);
  CUtensorMap tx, tf, txo, ty, ty8;
  if (!map_streams(&tx, a.X, a.N, a.d, tt)) return cudaErrorInvalidValue;
  if (fused) {
    if (!map_rows(&tf, a.F, a.N, a.d, tt)) return cudaErrorInvalidValue;
    if (!map_streams(&txo, a.X_out, a.N, a.d, tt)) return cudaErrorInvalidValue;
    if (!(mx ? map_codes(&ty, a.y_out, a.N, a.d, std::min(tt, 32)) : map_rows(&ty, a.y_out, a.N, a.d, tt)))
      return cudaErrorInvalidValue;
    if (mx ? !map_codes(&ty8, a.y_out, a.N, a.d, 8) : false) return cudaErrorInvalidValue;
    if (!mx) ty8 = ty;
  } else {
    tf = tx;
    txo = tx;
    ty = tx;
    ty8 = tx;
  }

  StepParams P{};
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
  P.y_scale = mx ? a.y_scale : nullptr;
  P.status = status_word();
  if (P.status == nullptr) return cudaErrorInvalidDevice;
  P.trace = trace_buffer(static_cast<int64_t>(split) * tiles);
  // scratch: the group counters (32 B per group), the tagged S_y words (both zeroed by one
  // memset per launch), then the partial sums
  uint8_t* scratch = static_cast<uint8_t*>(a.scratch);
  const size_t counter_bytes = (static_cast<size_t>(ngroups) * 32 + 255) / 256 * 256;
  const size_t sytag_bytes = static_cast<size_t>(ngroups) * 2 * TT * split * 8;
  P.counters = reinterpret_cast<unsigned*>(scratch);
  P.sytag = reinterpret_cast<unsigned long long*>(scratch + counter_bytes);
  P.sytag_end = P.sytag + sytag_bytes / 8;
  P.gpart = reinterpret_cast<float*>(scratch + counter_bytes + sytag_bytes);
  P.gpart_end = P.gpart + static_cast<size_t>(ngroups) * split * 2 * (PART_BYTES / 4);
  if (counter_bytes + sytag_bytes + static_cast<size_t>(ngroups) * split * 2 * PART_BYTES > a.scratch_bytes)
    return cudaErrorInvalidValue;
  P.N = static_cast<int>(a.N);
  P.tt = tt;
  P.d = a.d;
  P.split = split;
  P.slice = a.d / split;
  P.nsteps = P.slice / DC;
  P.iters = a.iters;
  P.hc_eps = a.hc_eps;
  P.norm_eps = a.norm_eps;
  P.neg_zero = -0.0f;
  P.flags = a.flags;

  e = cudaMemsetAsync(P.counters, 0, counter_bytes + sytag_bytes, stream);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ngroups * split, 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: groups wait on each other
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tx, tf, txo, ty, ty8, P);
}

cudaError_t step_resident_ctas(int* ctas) {
  auto kern = step_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return resident_ctas(kern, ctas);
}

}  // namespace mhc

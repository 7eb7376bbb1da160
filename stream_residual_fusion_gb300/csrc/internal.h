// internal.h -- host-side declarations shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "layout.cuh"

namespace mhc {

// Device address of the library's status word on the current device (see mhc_get_status).
unsigned* status_word();
// The trace buffer set by mhc_set_trace if it holds `ctas` CTAs' records, else nullptr.
unsigned long long* trace_buffer(int64_t ctas);

constexpr unsigned STATUS_TIMEOUT = 1u;
// Set by the bounds-checked build (MHC_CHECKED=1) when an index test fails; the access is skipped.
constexpr unsigned STATUS_BOUNDS = 2u;
// Flag bit of the checked build only: plant one out-of-range row index in a finisher store and
// in an MXFP8 scale store, to show that the checks catch it (MHC_ERR_SHAPE elsewhere).
constexpr unsigned FLAG_PLANT_OOB = 0x4u;

#ifndef MHC_CHECKED
#define MHC_CHECKED 0
#endif

struct StepArgs {
  const void* X;
  const void* F;            // fused step only
  const float* pre_prev;    // fused step only
  const float* post_prev;   // fused step only
  const float* comb_prev;   // fused step only
  const void* W_packed;     // bf16 [72, 4d]
  const float* scale;
  const float* base;
  const float* gain;        // fused step only
  void* X_out;              // fused step only
  void* y_out;              // fused step only: bf16 [N, d], or E4M3 codes [N, d] with y_scale
  uint8_t* y_scale;         // MXFP8 y only: E8M0 scale codes [N, d / 32]; null for bf16 y
  float* pre_out;
  float* post_out;
  float* comb_out;
  float* mixes_out;         // nullable
  void* scratch;            // group exchange area, >= step_scratch_bytes()
  size_t scratch_bytes;
  int64_t N;
  int d;
  int split;                // CTAs per token tile (cluster size)
  int iters;
  float hc_eps;
  float norm_eps;
  unsigned flags;
};

// Largest number of CTAs that share a tile.
constexpr int kMaxSplit = 32;
// Whether `split` CTAs can share a tile of width d.
bool split_ok(int d, int split);
// The smallest split that fits width d (or `forced` if it fits); 0 if none.
int choose_split(int d, int forced);
// Launch shape of the step kernel: CTAs per tile, tokens per tile (a multiple of 8 and of the
// split, <= STEP_TT) and groups launched. `forced_*` != 0 pins a value; split 0 if nothing fits.
struct StepShape {
  int split;
  int tt;
  int groups;
};
StepShape choose_shape(int64_t N, int d, int ctas, int forced_split, int forced_tile);
// Cost of one pipeline slot of the step kernel in tokens of streaming work: a slot of a tile of
// tt tokens takes about (tt + kTileCostTokens) units (every slot pays load latency). Measured on
// GB300 at d = 5120, 20 slots per tile: 685 us for 256 tiles of 128 tokens, 955 us for 512
// tiles of 64.
constexpr int kTileCostTokens = 96;
// Tile height forced by the flags (MHC_TILE_SHIFT bits), 0 if automatic; -1 if invalid (over
// the STEP_TT rows a tile holds).
inline int tile_flag(unsigned flags) {
  const int v = static_cast<int>((flags >> 16) & 0x1Fu);
  return v == 0 ? 0 : (8 * v <= STEP_TT ? 8 * v : -1);
}
// Split forced by the flags (MHC_SPLIT_SHIFT bits hold log2(split) + 1), 0 if automatic; -1 if
// invalid.
inline int split_flag_value(unsigned flags) {
  const int v = static_cast<int>((flags >> 8) & 0xFu);
  return v == 0 ? 0 : (v <= 6 ? 1 << (v - 1) : -1);
}
constexpr int kMaxTokens = 65535 * 128;

// Launch-path flags (MHC_PATH_PERSISTENT, MHC_PATH_CLUSTER).
constexpr unsigned FLAG_PATH_PERSISTENT = 0x8u;
constexpr unsigned FLAG_PATH_CLUSTER = 0x10u;
// The cluster kernel (cluster.cu): CTAs per cluster (16 or 8, `forced` if nonzero) whose tiles
// fit width d, 0 if none; clusters of that size the current device runs at once (0 if it cannot
// run one); the cluster size the step takes for (N, d, flags) (0: the persistent kernel), with
// fused_bf16 false for the mixes-only and MXFP8 forms; and the launch.
int cluster_size_for(int d, int forced);
int cluster_capacity(int cl);
int cluster_path(int64_t N, int d, unsigned flags, bool fused_bf16);
cudaError_t launch_cluster_step(const StepArgs& a, int cl, cudaStream_t stream);
// Automatic choice: the cluster kernel while the tiles need at most this many waves of clusters.
constexpr int kClusterWaves = 1;
// Tokens per tile of the cluster kernel.
constexpr int kClusterTile = 40;

// The driver's tensor-map encoder (cuTensorMapEncodeTiled), looked up once; nullptr if absent.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

cudaError_t launch_step(bool fused, const StepArgs& a, cudaStream_t stream);
// CTAs of the step kernel the current device holds at once (one per SM).
cudaError_t step_resident_ctas(int* ctas);
// Scratch the step kernel needs on the current device (0 if the device cannot be queried).
size_t step_scratch_bytes();
cudaError_t launch_pack(const float* W, void* packed, int d, cudaStream_t stream);
cudaError_t launch_sinkhorn(const float* mixes, const float* scale, const float* base, float* pre,
                            float* post, float* comb, int64_t N, int iters, float eps,
                            cudaStream_t stream);
cudaError_t launch_rmsnorm(const void* x, const float* gain, void* y, int64_t N, int d, float eps,
                           cudaStream_t stream);
cudaError_t launch_hc_post(const void* X, const void* F, const float* post, const float* comb,
                           void* X_out, int64_t N, int d, bool row_dest, cudaStream_t stream);
cudaError_t launch_hc_pre(const void* Xp, const float* pre, void* y_hat, int64_t N, int d,
                          cudaStream_t stream);

// Gradients of the step (backward.cu).
struct BwdArgs {
  const void* X;          // bf16 [N, 4, d]
  const void* F;          // bf16 [N, d]
  const void* Xp;         // bf16 [N, 4, d], the forward's X'
  const float* mixes;     // [N, 24], the forward's m
  const float* pre_prev;
  const float* post_prev;
  const float* comb_prev;
  const float* W;         // fp32 [24, 4d]
  const float* scale;
  const float* base;
  const float* gain;
  const void* gXp;        // bf16 [N, 4, d]
  const void* gy;         // bf16 [N, d]
  const float* gpre;
  const float* gpost;
  const float* gcomb;
  void* gX;               // bf16 [N, 4, d]
  void* gF;               // bf16 [N, d]
  float* gpre_prev;
  float* gpost_prev;
  float* gcomb_prev;
  float* gW;              // [24, 4d]
  float* gbase;           // [24]
  float* gscale;          // [3]
  float* ggain;           // [d]
  void* workspace;
  size_t workspace_bytes;
  int64_t N;
  int d;
  int iters;
  float hc_eps;
  float norm_eps;
  unsigned flags;
};
// Workspace of the backward on the current device: byte offsets of its parts and the total.
struct BwdLayout {
  size_t off_wt, off_gm, off_rec, off_gsf, off_gpl, off_part0, off_partW, off_partG, bytes;
  int ranges;    // token ranges of the weight-gradient partial sums
  int64_t per;   // tokens per range
  int blocks0;   // blocks of the mix-gradient kernel (its partial sums)
};
// bytes == 0 if d is not a multiple of 64 or the device cannot be queried.
BwdLayout bwd_layout(int64_t N, int d);
cudaError_t launch_backward(const BwdArgs& a, cudaStream_t stream);

// Address ranges of the tensors of a call, for the overlap checks of the entry points.
struct Span {
  uintptr_t lo, hi;
  bool empty() const { return hi <= lo; }
};
inline Span span(const void* p, uint64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Span{a, a + static_cast<uintptr_t>(bytes)};
}
inline bool overlap(Span a, Span b) { return !a.empty() && !b.empty() && a.lo < b.hi && b.lo < a.hi; }

// Outputs must not overlap inputs or each other; output `same_out` may be exactly equal (same
// start and size) to input `same_in` (an in-place update).
template <int NO, int NI>
inline bool aliasing_ok(const Span (&outs)[NO], const Span (&ins)[NI], int same_out = -1, int same_in = -1) {
  for (int i = 0; i < NO; ++i) {
    for (int j = 0; j < NI; ++j) {
      if (i == same_out && j == same_in && outs[i].lo == ins[j].lo && outs[i].hi == ins[j].hi) continue;
      if (overlap(outs[i], ins[j])) return false;
    }
    for (int j = i + 1; j < NO; ++j)
      if (overlap(outs[i], outs[j])) return false;
  }
  return true;
}

}  // namespace mhc

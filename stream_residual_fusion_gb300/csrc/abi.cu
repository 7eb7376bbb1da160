// abi.cu -- the exported C ABI: argument validation, launches, status word.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "layout.cuh"
#include "mhc.h"

namespace mhc {
namespace {

// The status word: set by device-side bounded waits that give up, read and cleared by
// mhc_get_status. One per device that loaded the library (static, never allocated).
__device__ unsigned g_status;

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;
unsigned long long* g_trace = nullptr;
int64_t g_trace_ctas = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_code(cudaError_t e) { return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA; }

}  // namespace

unsigned* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

unsigned long long* trace_buffer(int64_t ctas) {
  return (g_trace != nullptr && ctas <= g_trace_ctas) ? g_trace : nullptr;
}

}  // namespace mhc

using namespace mhc;

namespace {

// Checks shared by the fused step and the mixes call. Returns MHC_OK and the split, or a code.
// cluster_ok: the call has the cluster kernel (the fused step with bf16 y); MHC_PATH_CLUSTER is
// MHC_ERR_SHAPE elsewhere, and where d fits no cluster size (its split bits then pick 8 or 16).
int check_step_shape(int64_t N, int n, int d, int iters, unsigned flags, int* split,
                     bool cluster_ok = false) {
  if (n != 4 || N < 0 || N > kMaxTokens || iters < 1 || d <= 0) return MHC_ERR_SHAPE;
  if (!MHC_CHECKED && (flags & FLAG_PLANT_OOB) != 0) return MHC_ERR_SHAPE;   // checked build only
  const int fs = split_flag_value(flags), ft = tile_flag(flags);
  if (fs < 0 || ft < 0) return MHC_ERR_SHAPE;
  if ((flags & FLAG_PATH_CLUSTER) != 0) {
    if (!cluster_ok || (flags & FLAG_PATH_PERSISTENT) != 0 || ft != 0) return MHC_ERR_SHAPE;
    *split = cluster_size_for(d, fs);
    return *split != 0 ? MHC_OK : MHC_ERR_SHAPE;
  }
  *split = choose_split(d, fs);
  if (*split == 0) return MHC_ERR_SHAPE;
  // some split that fits d must also divide a forced tile height
  for (int s = 1; s <= kMaxSplit; s *= 2)
    if ((fs == 0 || s == fs) && split_ok(d, s) && (ft == 0 || ft % s == 0)) return MHC_OK;
  return MHC_ERR_SHAPE;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// workspace = [packed weights | scratch]; W_mix given: pack into the workspace first.
int fused_common(const void* X, const void* F, const float* pre_prev, const float* post_prev,
                 const float* comb_prev, const void* W_packed, const float* scale,
                 const float* base, const float* gain, void* X_out, void* y_out, float* pre_out,
                 float* post_out, float* comb_out, float* mixes_out, int64_t N, int n, int d,
                 int iters, float hc_eps, float norm_eps, unsigned flags, const void* workspace,
                 uint64_t ws_bytes, void* scratch, uint64_t scratch_bytes, const float* W_mix,
                 void* stream, uint8_t* y_scale = nullptr) {
  // y_scale set: y_out receives MXFP8 E4M3 codes [N, d] (one byte each) and y_scale the E8M0
  // block scales [N, d / 32]; otherwise y_out is bf16 [N, d].
  int split = 0;
  int rc = check_step_shape(N, n, d, iters, flags, &split, y_scale == nullptr);
  if (rc != MHC_OK) return rc;
  if (N == 0) return MHC_OK;  // nothing to read or write (empty tensors may have no address)
  if (!X || !F || !pre_prev || !post_prev || !comb_prev || !W_packed || !scale || !base || !gain ||
      !X_out || !y_out || !pre_out || !post_out || !comb_out)
    return MHC_ERR_NULL;
  if (!scratch) return MHC_ERR_WORKSPACE;
  const void* ptrs[] = {X, F, pre_prev, post_prev, comb_prev, W_packed, scale, base, gain,
                        X_out, y_out, pre_out, post_out, comb_out, scratch};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MHC_ERR_ALIGN;
  if (mixes_out && !aligned16(mixes_out)) return MHC_ERR_ALIGN;
  if (W_mix && !aligned16(W_mix)) return MHC_ERR_ALIGN;
  if (y_scale && !aligned16(y_scale)) return MHC_ERR_ALIGN;

  const uint64_t nt = static_cast<uint64_t>(N);
  const uint64_t K = 4ull * d;
  const uint64_t y_bytes = nt * d * (y_scale ? 1 : 2);
  const Span ins[] = {span(X, nt * K * 2),     span(F, nt * d * 2),      span(pre_prev, nt * 16),
                      span(post_prev, nt * 16), span(comb_prev, nt * 64), span(scale, 12),
                      span(base, 96),          span(gain, 4ull * d),     span(W_mix, W_mix ? 96 * K : 0)};
  const Span outs[] = {span(X_out, nt * K * 2), span(y_out, y_bytes), span(pre_out, nt * 16),
                       span(post_out, nt * 16), span(comb_out, nt * 64),
                       span(mixes_out, mixes_out ? nt * 96 : 0),
                       span(workspace, workspace ? ws_bytes : 0),
                       span(scratch, workspace ? 0 : scratch_bytes),
                       span(y_scale, y_scale ? nt * (d / 32) : 0)};
  if (!aliasing_ok(outs, ins, 0, 0)) return MHC_ERR_ALIAS;
  if (!workspace) {  // pre-packed weights are an input too
    const Span packed_in[] = {span(W_packed, mhc_packed_weights_bytes(4, d))};
    if (!aliasing_ok(outs, packed_in)) return MHC_ERR_ALIAS;
  }
  const size_t need = step_scratch_bytes();
  if (need == 0) return MHC_ERR_CUDA;
  if (scratch_bytes < need) return MHC_ERR_WORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (W_mix) {
    rc = cuda_code(launch_pack(W_mix, const_cast<void*>(W_packed), d, s));
    if (rc != MHC_OK) return rc;
  }
  StepArgs a{};
  a.X = X;
  a.F = F;
  a.pre_prev = pre_prev;
  a.post_prev = post_prev;
  a.comb_prev = comb_prev;
  a.W_packed = W_packed;
  a.scale = scale;
  a.base = base;
  a.gain = gain;
  a.X_out = X_out;
  a.y_out = y_out;
  a.y_scale = y_scale;
  a.pre_out = pre_out;
  a.post_out = post_out;
  a.comb_out = comb_out;
  a.mixes_out = mixes_out;
  a.scratch = scratch;
  a.scratch_bytes = scratch_bytes;
  a.N = N;
  a.d = d;
  a.split = split;
  a.iters = iters;
  a.hc_eps = hc_eps;
  a.norm_eps = norm_eps;
  a.flags = flags;
  return cuda_code(launch_step(true, a, s));
}

}  // namespace

extern "C" {

size_t mhc_packed_weights_bytes(int n, int d) {
  if (n != 4 || d <= 0 || d % STEP_WDC != 0) return 0;
  return static_cast<size_t>(d / STEP_WDC) * STEP_WBLOCK_BYTES;
}

size_t mhc_step_scratch_bytes(int n, int d) {
  if (mhc_packed_weights_bytes(n, d) == 0) return 0;
  return step_scratch_bytes();
}

size_t mhc_workspace_bytes(int n, int d) {
  const size_t packed = mhc_packed_weights_bytes(n, d);
  if (packed == 0) return 0;
  return align256(packed) + step_scratch_bytes();
}

int mhc_packed_block_columns(void) { return STEP_WDC; }

int mhc_pack_weights(const float* W_mix, void* W_packed, int n, int d, void* stream) {
  if (!W_mix || !W_packed) return MHC_ERR_NULL;
  if (n != 4 || d <= 0 || d % STEP_WDC != 0) return MHC_ERR_SHAPE;
  if (!aligned16(W_mix) || !aligned16(W_packed)) return MHC_ERR_ALIGN;
  const uint64_t K = 4ull * d;
  if (overlap(span(W_mix, 96 * K), span(W_packed, mhc_packed_weights_bytes(4, d)))) return MHC_ERR_ALIAS;
  return cuda_code(launch_pack(W_mix, W_packed, d, static_cast<cudaStream_t>(stream)));
}

int mhc_fused_step(const void* X, const void* F, const float* pre_prev, const float* post_prev,
                   const float* comb_prev, const float* W_mix, const float* scale,
                   const float* base, const float* gain, void* X_out, void* y_out,
                   float* pre_out, float* post_out, float* comb_out, float* mixes_out,
                   int64_t N, int n, int d, int sinkhorn_iters, float hc_eps, float norm_eps,
                   unsigned flags, void* workspace, size_t workspace_bytes, void* stream) {
  int split = 0;
  const int rc = check_step_shape(N, n, d, sinkhorn_iters, flags, &split, true);
  if (rc != MHC_OK) return rc;
  if (N == 0) return MHC_OK;
  if (!W_mix) return MHC_ERR_NULL;
  const size_t packed = align256(mhc_packed_weights_bytes(n, d));
  if (!workspace || workspace_bytes < packed) return MHC_ERR_WORKSPACE;
  return fused_common(X, F, pre_prev, post_prev, comb_prev, workspace, scale, base, gain, X_out,
                      y_out, pre_out, post_out, comb_out, mixes_out, N, n, d, sinkhorn_iters,
                      hc_eps, norm_eps, flags, workspace, workspace_bytes,
                      static_cast<uint8_t*>(workspace) + packed, workspace_bytes - packed, W_mix,
                      stream);
}

int mhc_fused_step_packed(const void* X, const void* F, const float* pre_prev,
                          const float* post_prev, const float* comb_prev, const void* W_packed,
                          const float* scale, const float* base, const float* gain, void* X_out,
                          void* y_out, float* pre_out, float* post_out, float* comb_out,
                          float* mixes_out, int64_t N, int n, int d, int sinkhorn_iters,
                          float hc_eps, float norm_eps, unsigned flags, void* scratch,
                          size_t scratch_bytes, void* stream) {
  return fused_common(X, F, pre_prev, post_prev, comb_prev, W_packed, scale, base, gain, X_out,
                      y_out, pre_out, post_out, comb_out, mixes_out, N, n, d, sinkhorn_iters,
                      hc_eps, norm_eps, flags, nullptr, 0, scratch, scratch_bytes, nullptr,
                      stream);
}

int mhc_fused_step_mxfp8(const void* X, const void* F, const float* pre_prev,
                         const float* post_prev, const float* comb_prev, const void* W_packed,
                         const float* scale, const float* base, const float* gain, void* X_out,
                         void* y_codes, void* y_scale, float* pre_out, float* post_out,
                         float* comb_out, float* mixes_out, int64_t N, int n, int d,
                         int sinkhorn_iters, float hc_eps, float norm_eps, unsigned flags,
                         void* scratch, size_t scratch_bytes, void* stream) {
  if (N > 0 && !y_scale) return MHC_ERR_NULL;
  return fused_common(X, F, pre_prev, post_prev, comb_prev, W_packed, scale, base, gain, X_out,
                      y_codes, pre_out, post_out, comb_out, mixes_out, N, n, d, sinkhorn_iters,
                      hc_eps, norm_eps, flags, nullptr, 0, scratch, scratch_bytes, nullptr,
                      stream, static_cast<uint8_t*>(y_scale));
}

int mhc_mixes(const void* X, const float* W_mix, const float* scale, const float* base,
              float* mixes_out, float* pre_out, float* post_out, float* comb_out, int64_t N,
              int n, int d, int sinkhorn_iters, float hc_eps, float norm_eps, unsigned flags,
              void* workspace, size_t workspace_bytes, void* stream) {
  int split = 0;
  int rc = check_step_shape(N, n, d, sinkhorn_iters, flags, &split);
  if (rc != MHC_OK) return rc;
  if (N == 0) return MHC_OK;
  if (!X || !W_mix || !scale || !base || !pre_out || !post_out || !comb_out) return MHC_ERR_NULL;
  if (!workspace) return MHC_ERR_WORKSPACE;
  const size_t packed = align256(mhc_packed_weights_bytes(n, d));
  const size_t need = step_scratch_bytes();
  if (need == 0) return MHC_ERR_CUDA;
  if (workspace_bytes < packed + need) return MHC_ERR_WORKSPACE;
  const void* ptrs[] = {X, W_mix, scale, base, pre_out, post_out, comb_out, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MHC_ERR_ALIGN;
  if (mixes_out && !aligned16(mixes_out)) return MHC_ERR_ALIGN;
  const uint64_t nt = static_cast<uint64_t>(N), K = 4ull * d;
  const Span ins[] = {span(X, nt * K * 2), span(W_mix, 96 * K), span(scale, 12), span(base, 96)};
  const Span outs[] = {span(pre_out, nt * 16), span(post_out, nt * 16), span(comb_out, nt * 64),
                       span(mixes_out, mixes_out ? nt * 96 : 0), span(workspace, workspace_bytes)};
  if (!aliasing_ok(outs, ins)) return MHC_ERR_ALIAS;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = cuda_code(launch_pack(W_mix, workspace, d, s));
  if (rc != MHC_OK) return rc;
  StepArgs a{};
  a.X = X;
  a.W_packed = workspace;
  a.scale = scale;
  a.base = base;
  a.pre_out = pre_out;
  a.post_out = post_out;
  a.comb_out = comb_out;
  a.mixes_out = mixes_out;
  a.scratch = static_cast<uint8_t*>(workspace) + packed;
  a.scratch_bytes = workspace_bytes - packed;
  a.N = N;
  a.d = d;
  a.split = split;
  a.iters = sinkhorn_iters;
  a.hc_eps = hc_eps;
  a.norm_eps = norm_eps;
  a.flags = flags;
  return cuda_code(launch_step(false, a, s));
}

int mhc_sinkhorn(const float* mixes, const float* scale, const float* base, float* pre_out,
                 float* post_out, float* comb_out, int64_t N, int n, int sinkhorn_iters,
                 float hc_eps, void* stream) {
  if (n != 4 || N < 0 || sinkhorn_iters < 1 || N > (int64_t(1) << 40)) return MHC_ERR_SHAPE;
  if (N == 0) return MHC_OK;
  if (!mixes || !scale || !base || !pre_out || !post_out || !comb_out) return MHC_ERR_NULL;
  const void* ptrs[] = {mixes, scale, base, pre_out, post_out, comb_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MHC_ERR_ALIGN;
  const uint64_t nt = static_cast<uint64_t>(N);
  const Span ins[] = {span(mixes, nt * 96), span(scale, 12), span(base, 96)};
  const Span outs[] = {span(pre_out, nt * 16), span(post_out, nt * 16), span(comb_out, nt * 64)};
  if (!aliasing_ok(outs, ins)) return MHC_ERR_ALIAS;
  return cuda_code(launch_sinkhorn(mixes, scale, base, pre_out, post_out, comb_out, N,
                                   sinkhorn_iters, hc_eps, static_cast<cudaStream_t>(stream)));
}

int mhc_rmsnorm(const void* x, const float* gain, void* y, int64_t N, int d, float eps,
                void* stream) {
  if (N < 0 || d <= 0 || d % 8 != 0) return MHC_ERR_SHAPE;
  if (N == 0) return MHC_OK;
  if (!x || !gain || !y) return MHC_ERR_NULL;
  if (!aligned16(x) || !aligned16(gain) || !aligned16(y)) return MHC_ERR_ALIGN;
  const uint64_t nt = static_cast<uint64_t>(N);
  const Span ins[] = {span(x, nt * d * 2), span(gain, 4ull * d)};
  const Span outs[] = {span(y, nt * d * 2)};
  if (!aliasing_ok(outs, ins, 0, 0)) return MHC_ERR_ALIAS;
  return cuda_code(launch_rmsnorm(x, gain, y, N, d, eps, static_cast<cudaStream_t>(stream)));
}

int mhc_hc_post(const void* X, const void* F, const float* post, const float* comb, void* X_out,
                int64_t N, int n, int d, unsigned flags, void* stream) {
  if (n != 4 || N < 0 || d <= 0 || d % 8 != 0) return MHC_ERR_SHAPE;
  if (N == 0) return MHC_OK;
  if (!X || !F || !post || !comb || !X_out) return MHC_ERR_NULL;
  const void* ptrs[] = {X, F, post, comb, X_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MHC_ERR_ALIGN;
  const uint64_t nt = static_cast<uint64_t>(N), K = 4ull * d;
  const Span ins[] = {span(X, nt * K * 2), span(F, nt * d * 2), span(post, nt * 16), span(comb, nt * 64)};
  const Span outs[] = {span(X_out, nt * K * 2)};
  if (!aliasing_ok(outs, ins, 0, 0)) return MHC_ERR_ALIAS;
  return cuda_code(launch_hc_post(X, F, post, comb, X_out, N, d, (flags & MHC_COMB_ROW_DEST) != 0,
                                  static_cast<cudaStream_t>(stream)));
}

int mhc_hc_pre(const void* Xp, const float* pre, void* y_hat, int64_t N, int n, int d,
               void* stream) {
  if (n != 4 || N < 0 || d <= 0 || d % 8 != 0) return MHC_ERR_SHAPE;
  if (N == 0) return MHC_OK;
  if (!Xp || !pre || !y_hat) return MHC_ERR_NULL;
  if (!aligned16(Xp) || !aligned16(pre) || !aligned16(y_hat)) return MHC_ERR_ALIGN;
  const uint64_t nt = static_cast<uint64_t>(N);
  const Span ins[] = {span(Xp, nt * 8ull * d), span(pre, nt * 16)};
  const Span outs[] = {span(y_hat, nt * d * 2)};
  if (!aliasing_ok(outs, ins)) return MHC_ERR_ALIAS;
  return cuda_code(launch_hc_pre(Xp, pre, y_hat, N, d, static_cast<cudaStream_t>(stream)));
}

int mhc_get_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MHC_ERR_CUDA;
  unsigned* p = status_word();
  if (p == nullptr) return MHC_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MHC_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MHC_ERR_CUDA;
  }
  if (v & STATUS_BOUNDS) return MHC_ERR_BOUNDS;
  return (v & STATUS_TIMEOUT) ? MHC_ERR_TIMEOUT : MHC_OK;
}

const char* mhc_strerror(int code) {
  switch (code) {
    case MHC_OK: return "ok";
    case MHC_ERR_NULL: return "a required pointer is NULL";
    case MHC_ERR_SHAPE: return "unsupported shape (n must be 4; d, N or sinkhorn_iters out of range)";
    case MHC_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case MHC_ERR_ALIAS: return "an output overlaps an input or another output";
    case MHC_ERR_CUDA: return "a CUDA call failed";
    case MHC_ERR_TIMEOUT: return "a device-side bounded wait gave up";
    case MHC_ERR_WORKSPACE: return "workspace missing or too small";
    case MHC_ERR_BOUNDS: return "an index check of the bounds-checked build failed (access skipped)";
    default: return "unknown status code";
  }
}

int mhc_step_path(int64_t N, int n, int d, unsigned flags) {
  int sp = 0;
  const int rc = check_step_shape(N, n, d, 1, flags, &sp, true);
  if (rc != MHC_OK) return rc;
  return cluster_path(N, d, flags, true) != 0 ? static_cast<int>(MHC_PATH_CLUSTER)
                                              : static_cast<int>(MHC_PATH_PERSISTENT);
}

int mhc_step_config(int64_t N, int n, int d, unsigned flags, int* split, int* tile, int* groups) {
  if (!split || !tile || !groups) return MHC_ERR_NULL;
  int sp = 0, ctas = 0;
  const int rc = check_step_shape(N, n, d, 1, flags, &sp, true);
  if (rc != MHC_OK) return rc;
  if (const int cl = cluster_path(N, d, flags, true)) {
    *split = cl;
    *tile = kClusterTile;
    *groups = static_cast<int>((std::max<int64_t>(N, 1) + kClusterTile - 1) / kClusterTile);
    return MHC_OK;
  }
  if (step_resident_ctas(&ctas) != cudaSuccess) return MHC_ERR_CUDA;
  const StepShape sh = choose_shape(N, d, ctas, split_flag_value(flags), tile_flag(flags));
  if (sh.split == 0) return MHC_ERR_CUDA;
  *split = sh.split;
  *tile = sh.tt;
  *groups = sh.groups;
  return MHC_OK;
}

// ---------------------------------------------------------------------------------------------
// Allocation-free fused step.
//
// Some callers cannot allocate device memory at the point they run the step: a serving loop
// running under a fixed device-memory budget, or one whose caching allocator it may not enter
// there, or a plain C host that links this library and has no device allocator of its own. This entry point runs the same fused step with its
// scratch (the packed weights and the step's exchange area) in one fixed array that the
// library holds on every GPU that loads it, until the process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the fixed scratch on the current device (set up once per device).
void* noalloc_scratch(int* rc) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *rc = MHC_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *rc = MHC_ERR_CUDA;
      return nullptr;
    }
    g_noalloc_ptr[dev] = p;
  }
  *rc = MHC_OK;
  return g_noalloc_ptr[dev];
}

}  // namespace

size_t mhc_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int mhc_fused_step_noalloc(const void* X, const void* F, const float* pre_prev,
                           const float* post_prev, const float* comb_prev, const float* W_mix,
                           const float* scale, const float* base, const float* gain, void* X_out,
                           void* y_out, float* pre_out, float* post_out, float* comb_out,
                           float* mixes_out, int64_t N, int n, int d, int sinkhorn_iters,
                           float hc_eps, float norm_eps, unsigned flags, void* stream) {
  int split = 0;
  int rc = check_step_shape(N, n, d, sinkhorn_iters, flags, &split, true);
  if (rc != MHC_OK) return rc;
  if (N == 0) return MHC_OK;
  if (!W_mix) return MHC_ERR_NULL;
  const size_t need = mhc_workspace_bytes(n, d);
  if (need == 0) return MHC_ERR_CUDA;
  if (need > kNoAllocScratchBytes) return MHC_ERR_WORKSPACE;   // beyond the fixed scratch
  void* ws = noalloc_scratch(&rc);
  if (ws == nullptr) return rc;
  const size_t packed = align256(mhc_packed_weights_bytes(n, d));
  return fused_common(X, F, pre_prev, post_prev, comb_prev, ws, scale, base, gain, X_out, y_out,
                      pre_out, post_out, comb_out, mixes_out, N, n, d, sinkhorn_iters, hc_eps,
                      norm_eps, flags, ws, kNoAllocScratchBytes,
                      static_cast<uint8_t*>(ws) + packed, kNoAllocScratchBytes - packed, W_mix,
                      stream);
}

// ---------------------------------------------------------------------------------------------
// Gradients of the step.

size_t mhc_backward_workspace_bytes(int64_t N, int n, int d) {
  if (n != 4 || N < 0 || N > kMaxTokens || d <= 0 || d % 64 != 0) return 0;
  return bwd_layout(N, d).bytes;
}

int mhc_fused_step_backward(const void* X, const void* F, const void* Xp, const float* mixes,
                            const float* pre_prev, const float* post_prev, const float* comb_prev,
                            const float* W_mix, const float* scale, const float* base,
                            const float* gain, const void* gXp, const void* gy, const float* gpre,
                            const float* gpost, const float* gcomb, void* gX, void* gF,
                            float* gpre_prev, float* gpost_prev, float* gcomb_prev, float* gW,
                            float* gbase, float* gscale, float* ggain, int64_t N, int n, int d,
                            int sinkhorn_iters, float hc_eps, float norm_eps, unsigned flags,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (n != 4 || N < 0 || N > kMaxTokens || d <= 0 || d % 64 != 0 || sinkhorn_iters < 1)
    return MHC_ERR_SHAPE;
  if ((flags & ~MHC_COMB_ROW_DEST) != 0) return MHC_ERR_SHAPE;
  if (!W_mix || !scale || !base || !gain || !gW || !gbase || !gscale || !ggain) return MHC_ERR_NULL;
  const void* params[] = {W_mix, scale, base, gain, gW, gbase, gscale, ggain};
  for (const void* p : params)
    if (!aligned16(p)) return MHC_ERR_ALIGN;
  const uint64_t nt = static_cast<uint64_t>(N), K = 4ull * d;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {   // sums over no tokens
    const Span pin[] = {span(W_mix, 96 * K), span(scale, 12), span(base, 96), span(gain, 4ull * d)};
    const Span pout[] = {span(gW, 96 * K), span(gbase, 96), span(gscale, 12), span(ggain, 4ull * d)};
    if (!aliasing_ok(pout, pin)) return MHC_ERR_ALIAS;
    cudaError_t e = cudaMemsetAsync(gW, 0, 96 * K, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(gbase, 0, 96, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(gscale, 0, 12, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ggain, 0, 4ull * d, s);
    return cuda_code(e);
  }
  const void* ptrs[] = {X, F, Xp, mixes, pre_prev, post_prev, comb_prev, gXp, gy, gpre, gpost,
                        gcomb, gX, gF, gpre_prev, gpost_prev, gcomb_prev};
  for (const void* p : ptrs)
    if (!p) return MHC_ERR_NULL;
  for (const void* p : ptrs)
    if (!aligned16(p)) return MHC_ERR_ALIGN;
  if (!workspace) return MHC_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MHC_ERR_ALIGN;
  const Span ins[] = {span(X, nt * K * 2),      span(F, nt * d * 2),       span(Xp, nt * K * 2),
                      span(mixes, nt * 96),     span(pre_prev, nt * 16),   span(post_prev, nt * 16),
                      span(comb_prev, nt * 64), span(W_mix, 96 * K),       span(scale, 12),
                      span(base, 96),           span(gain, 4ull * d),      span(gXp, nt * K * 2),
                      span(gy, nt * d * 2),     span(gpre, nt * 16),       span(gpost, nt * 16),
                      span(gcomb, nt * 64)};
  const Span outs[] = {span(gX, nt * K * 2),      span(gF, nt * d * 2),     span(gpre_prev, nt * 16),
                       span(gpost_prev, nt * 16), span(gcomb_prev, nt * 64), span(gW, 96 * K),
                       span(gbase, 96),           span(gscale, 12),         span(ggain, 4ull * d),
                       span(workspace, workspace_bytes)};
  if (!aliasing_ok(outs, ins)) return MHC_ERR_ALIAS;
  const size_t need = bwd_layout(N, d).bytes;
  if (need == 0) return MHC_ERR_CUDA;
  if (workspace_bytes < need) return MHC_ERR_WORKSPACE;
  BwdArgs a{};
  a.X = X;
  a.F = F;
  a.Xp = Xp;
  a.mixes = mixes;
  a.pre_prev = pre_prev;
  a.post_prev = post_prev;
  a.comb_prev = comb_prev;
  a.W = W_mix;
  a.scale = scale;
  a.base = base;
  a.gain = gain;
  a.gXp = gXp;
  a.gy = gy;
  a.gpre = gpre;
  a.gpost = gpost;
  a.gcomb = gcomb;
  a.gX = gX;
  a.gF = gF;
  a.gpre_prev = gpre_prev;
  a.gpost_prev = gpost_prev;
  a.gcomb_prev = gcomb_prev;
  a.gW = gW;
  a.gbase = gbase;
  a.gscale = gscale;
  a.ggain = ggain;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.N = N;
  a.d = d;
  a.iters = sinkhorn_iters;
  a.hc_eps = hc_eps;
  a.norm_eps = norm_eps;
  a.flags = flags;
  return cuda_code(launch_backward(a, s));
}

int mhc_set_trace(void* buffer, int64_t bytes) {
  if (buffer != nullptr && (!aligned16(buffer) || bytes < 64)) return MHC_ERR_ALIGN;
  g_trace = static_cast<unsigned long long*>(buffer);
  g_trace_ctas = buffer == nullptr ? 0 : bytes / 64;
  return MHC_OK;
}

int mhc_version(void) { return 101; }

int mhc_checked_build(void) { return MHC_CHECKED; }

}  // extern "C"

// host_pipeline.cu -- the fused step on host-resident tensors: token chunks flow through three
// device staging slots so that host->device copies, the fused kernel and device->host copies of
// consecutive chunks overlap (three internal streams joined to the caller's stream by events).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "mhc.h"

namespace mhc {
namespace {

constexpr int kMaxDevices = 64;
// Staging slots. With two, the copy-in of chunk i would wait for the copy-out of chunk i-2, which
// trails the copy-in of chunk i-1 by one step kernel: a bubble per chunk. Three leave a chunk of
// slack.
constexpr int kSlots = 3;

struct Lanes {
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_ready[kSlots] = {}, computed[kSlots] = {}, out_done[kSlots] = {};
  bool ok = false;
};
Lanes g_lanes[kMaxDevices];
std::mutex g_lanes_mu;

// Streams and events of the current device, created on its first use.
Lanes* lanes() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_lanes_mu);
  Lanes& L = g_lanes[dev];
  if (!L.ok) {
    bool good = cudaStreamCreateWithFlags(&L.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&L.comp, cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&L.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                cudaEventCreateWithFlags(&L.start, cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&L.done, cudaEventDisableTiming) == cudaSuccess;
    for (int b = 0; good && b < kSlots; ++b)
      good = cudaEventCreateWithFlags(&L.in_ready[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&L.computed[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&L.out_done[b], cudaEventDisableTiming) == cudaSuccess;
    if (!good) return nullptr;
    L.ok = true;
  }
  return &L;
}

// Bytes of one staging slot for `chunk` tokens (inputs then outputs), each piece 256-aligned.
struct SlotLayout {
  size_t X, F, pre, post, comb, Xo, y, po, uo, co, mo, bytes;
};
size_t a256(size_t v) { return (v + 255) / 256 * 256; }
SlotLayout slot_layout(int64_t chunk, int d, bool with_mixes) {
  SlotLayout s{};
  const size_t c = static_cast<size_t>(chunk);
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += a256(bytes); return at; };
  s.X = take(c * 4 * d * 2);
  s.F = take(c * d * 2);
  s.pre = take(c * 16);
  s.post = take(c * 16);
  s.comb = take(c * 64);
  s.Xo = take(c * 4 * d * 2);
  s.y = take(c * d * 2);
  s.po = take(c * 16);
  s.uo = take(c * 16);
  s.co = take(c * 64);
  s.mo = with_mixes ? take(c * 96) : 0;
  s.bytes = o;
  return s;
}

// Token count of chunk i. The first and the last chunks ramp (c/8, c/4, c/2) so that the
// copy-in before the first step and the copy-out after the last one, which overlap nothing, are
// short; the rest are c tokens, the last full-size one taking the remainder. Batches under
// 2(c/8 + c/4 + c/2) + c tokens use plain chunks of c.
struct ChunkPlan {
  int64_t N, c, ramp[3] = {}, ramp_sum = 0;
  bool ramped = false;
  ChunkPlan(int64_t n_tok, int64_t chunk) : N(n_tok), c(chunk) {
    for (int k = 0; k < 3; ++k) {
      ramp[k] = chunk >> (3 - k);
      ramp_sum += ramp[k];
    }
    ramped = ramp[0] >= 1 && N >= 2 * ramp_sum + c;
  }
  // Calls f(start, count) for every chunk in order.
  template <class Fn>
  int each(Fn&& f) const {
    int64_t t = 0;
    int rc = 0;
    if (!ramped) {
      for (; t < N && rc == 0; t += c) rc = f(t, N - t < c ? N - t : c);
      return rc;
    }
    for (int k = 0; k < 3 && rc == 0; ++k) {
      rc = f(t, ramp[k]);
      t += ramp[k];
    }
    const int64_t mid_end = N - ramp_sum;
    for (; t < mid_end && rc == 0; t += c) rc = f(t, mid_end - t < c ? mid_end - t : c);
    t = mid_end;
    for (int k = 2; k >= 0 && rc == 0; --k) {
      rc = f(t, ramp[k]);
      t += ramp[k];
    }
    return rc;
  }
};

}  // namespace
}  // namespace mhc

using namespace mhc;

extern "C" {

size_t mhc_host_staging_bytes(int n, int d, int64_t chunk_tokens, int with_mixes) {
  const size_t ws = mhc_workspace_bytes(n, d);
  if (ws == 0 || chunk_tokens <= 0) return 0;
  return a256(ws) + kSlots * slot_layout(chunk_tokens, d, with_mixes != 0).bytes;
}

int64_t mhc_host_chunks(int64_t N, int64_t chunk_tokens, int64_t* counts, int64_t max_chunks) {
  if (N < 0 || chunk_tokens <= 0) return MHC_ERR_SHAPE;
  int64_t k = 0;
  ChunkPlan(N, chunk_tokens).each([&](int64_t, int64_t c) -> int {
    if (counts != nullptr && k < max_chunks) counts[k] = c;
    ++k;
    return MHC_OK;
  });
  return k;
}

int mhc_fused_step_host(const void* X, const void* F, const float* pre_prev,
                        const float* post_prev, const float* comb_prev, const float* W_mix,
                        const float* scale, const float* base, const float* gain, void* X_out,
                        void* y_out, float* pre_out, float* post_out, float* comb_out,
                        float* mixes_out, int64_t N, int n, int d, int sinkhorn_iters,
                        float hc_eps, float norm_eps, unsigned flags, void* staging,
                        size_t staging_bytes, int64_t chunk_tokens, void* stream) {
  if (chunk_tokens <= 0) return MHC_ERR_SHAPE;
  // the shape rules of the device step (it validates without launching when N == 0)
  int rc = mhc_fused_step_packed(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, N < 0 ? N : 0, n, d, sinkhorn_iters, hc_eps, norm_eps,
                                 flags, nullptr, 0, stream);
  if (rc != MHC_OK) return rc;
  if (N == 0) return MHC_OK;
  if (!X || !F || !pre_prev || !post_prev || !comb_prev || !W_mix || !scale || !base || !gain ||
      !X_out || !y_out || !pre_out || !post_out || !comb_out)
    return MHC_ERR_NULL;
  const uint64_t nt = static_cast<uint64_t>(N), K = 4ull * d;
  const Span ins[] = {span(X, nt * K * 2), span(F, nt * d * 2), span(pre_prev, nt * 16),
                      span(post_prev, nt * 16), span(comb_prev, nt * 64)};
  const Span outs[] = {span(X_out, nt * K * 2), span(y_out, nt * d * 2), span(pre_out, nt * 16),
                       span(post_out, nt * 16), span(comb_out, nt * 64),
                       span(mixes_out, mixes_out ? nt * 96 : 0)};
  if (!aliasing_ok(outs, ins, 0, 0)) return MHC_ERR_ALIAS;
  if (!staging) return MHC_ERR_WORKSPACE;
  const bool with_mixes = mixes_out != nullptr;
  const size_t need = mhc_host_staging_bytes(n, d, chunk_tokens, with_mixes ? 1 : 0);
  if (need == 0) return MHC_ERR_SHAPE;
  if (staging_bytes < need) return MHC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0) return MHC_ERR_ALIGN;
  Lanes* L = lanes();
  if (L == nullptr) return MHC_ERR_CUDA;

  uint8_t* base_ptr = static_cast<uint8_t*>(staging);
  const size_t ws_bytes = a256(mhc_workspace_bytes(n, d));
  const size_t packed = a256(mhc_packed_weights_bytes(n, d));
  uint8_t* ws = base_ptr;
  const SlotLayout lay = slot_layout(chunk_tokens, d, with_mixes);
  uint8_t* slot[kSlots];
  for (int b = 0; b < kSlots; ++b) slot[b] = base_ptr + ws_bytes + b * lay.bytes;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);

  auto ck = [](cudaError_t e) { return e == cudaSuccess; };
  // fork: the internal streams start after what the caller enqueued so far
  if (!ck(cudaEventRecord(L->start, caller)) || !ck(cudaStreamWaitEvent(L->h2d, L->start, 0)) ||
      !ck(cudaStreamWaitEvent(L->comp, L->start, 0)) || !ck(cudaStreamWaitEvent(L->d2h, L->start, 0)))
    return MHC_ERR_CUDA;
  rc = mhc_pack_weights(W_mix, ws, n, d, L->comp);
  if (rc != MHC_OK) return rc;

  const uint8_t* hX = static_cast<const uint8_t*>(X);
  const uint8_t* hF = static_cast<const uint8_t*>(F);
  uint8_t* hXo = static_cast<uint8_t*>(X_out);
  uint8_t* hy = static_cast<uint8_t*>(y_out);
  const size_t rowX = static_cast<size_t>(4) * d * 2, rowF = static_cast<size_t>(d) * 2;
  int64_t i = 0;
  rc = ChunkPlan(N, chunk_tokens).each([&](int64_t t0, int64_t c) -> int {
    const int b = static_cast<int>(i % kSlots);
    const size_t cc = static_cast<size_t>(c), tt = static_cast<size_t>(t0);
    uint8_t* S = slot[b];
    // inputs of chunk i into slot b once chunk i-kSlots has left it
    if (i >= kSlots && !ck(cudaStreamWaitEvent(L->h2d, L->out_done[b], 0))) return MHC_ERR_CUDA;
    ++i;
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    if (!ck(cudaMemcpyAsync(S + lay.X, hX + tt * rowX, cc * rowX, h2d, L->h2d)) ||
        !ck(cudaMemcpyAsync(S + lay.F, hF + tt * rowF, cc * rowF, h2d, L->h2d)) ||
        !ck(cudaMemcpyAsync(S + lay.pre, pre_prev + tt * 4, cc * 16, h2d, L->h2d)) ||
        !ck(cudaMemcpyAsync(S + lay.post, post_prev + tt * 4, cc * 16, h2d, L->h2d)) ||
        !ck(cudaMemcpyAsync(S + lay.comb, comb_prev + tt * 16, cc * 64, h2d, L->h2d)) ||
        !ck(cudaEventRecord(L->in_ready[b], L->h2d)))
      return MHC_ERR_CUDA;
    // the step on slot b
    if (!ck(cudaStreamWaitEvent(L->comp, L->in_ready[b], 0))) return MHC_ERR_CUDA;
    const int r = mhc_fused_step_packed(
        S + lay.X, S + lay.F, reinterpret_cast<float*>(S + lay.pre),
        reinterpret_cast<float*>(S + lay.post), reinterpret_cast<float*>(S + lay.comb), ws, scale,
        base, gain, S + lay.Xo, S + lay.y, reinterpret_cast<float*>(S + lay.po),
        reinterpret_cast<float*>(S + lay.uo), reinterpret_cast<float*>(S + lay.co),
        with_mixes ? reinterpret_cast<float*>(S + lay.mo) : nullptr, c, n, d, sinkhorn_iters,
        hc_eps, norm_eps, flags, ws + packed, ws_bytes - packed, L->comp);
    if (r != MHC_OK) return r;
    if (!ck(cudaEventRecord(L->computed[b], L->comp))) return MHC_ERR_CUDA;
    // outputs of chunk i back to the host
    if (!ck(cudaStreamWaitEvent(L->d2h, L->computed[b], 0)) ||
        !ck(cudaMemcpyAsync(hXo + tt * rowX, S + lay.Xo, cc * rowX, d2h, L->d2h)) ||
        !ck(cudaMemcpyAsync(hy + tt * rowF, S + lay.y, cc * rowF, d2h, L->d2h)) ||
        !ck(cudaMemcpyAsync(pre_out + tt * 4, S + lay.po, cc * 16, d2h, L->d2h)) ||
        !ck(cudaMemcpyAsync(post_out + tt * 4, S + lay.uo, cc * 16, d2h, L->d2h)) ||
        !ck(cudaMemcpyAsync(comb_out + tt * 16, S + lay.co, cc * 64, d2h, L->d2h)) ||
        (with_mixes && !ck(cudaMemcpyAsync(mixes_out + tt * 24, S + lay.mo, cc * 96, d2h, L->d2h))) ||
        !ck(cudaEventRecord(L->out_done[b], L->d2h)))
      return MHC_ERR_CUDA;
    return MHC_OK;
  });
  if (rc != MHC_OK) return rc;
  // join: the caller's stream continues once the last outputs are on the host
  if (!ck(cudaEventRecord(L->done, L->d2h)) || !ck(cudaStreamWaitEvent(caller, L->done, 0)))
    return MHC_ERR_CUDA;
  return MHC_OK;
}

}  // extern "C"

/*
 * mhc.h -- C ABI of libmhc.so, the GB300 (sm_103a) single-pass mHC step.
 *
 * The multi-stream hyper-connection (mHC) residual step of a 4-stream block, as defined on the
 * pages "DeepSeek V4.1 · Stream weights for the feed-forward" (sections "Why", "All 5 steps",
 * "Parameters", "Code") and "DeepSeek V4.1 · MoE RMSNorm" (formula block, "Code").
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous, row-major, with
 *     the token axis flattened (N = B*T). bf16 tensors are passed as void*. The library never
 *     frees or keeps them. (mhc_fused_step_host takes its per-token tensors as HOST pointers.)
 *   - Every pointer must be 16-byte aligned (MHC_ERR_ALIGN otherwise).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream). The library never synchronises, except in mhc_get_status.
 *   - The library allocates no device memory. Calls that need scratch take a caller-owned
 *     `workspace` of at least the size the matching *_workspace_bytes() call returns.
 *     (mhc_fused_step_host creates three streams and a few events per device on its first call
 *     there and keeps them until the process exits.)
 *   - Arguments are validated on the host before anything is launched; a negative return code
 *     means nothing was launched (except MHC_ERR_CUDA, which reports a launch failure).
 *   - Only n = 4 streams is built (the shape of the pages' block; (2+n)n = 24 mix numbers).
 */
#ifndef MHC_H
#define MHC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------------ */
#define MHC_OK             0
#define MHC_ERR_NULL      -1  /* a required pointer is NULL                                     */
#define MHC_ERR_SHAPE     -2  /* n != 4, d out of range / not a multiple of the tile, N < 0, iters < 1 */
#define MHC_ERR_ALIGN     -3  /* a pointer is not 16-byte aligned                                */
#define MHC_ERR_ALIAS     -4  /* an output overlaps an input or another output (X_out == X allowed) */
#define MHC_ERR_CUDA      -5  /* a CUDA runtime/driver call failed (launch, tensor map, attribute) */
#define MHC_ERR_TIMEOUT   -6  /* a device-side bounded wait gave up (see mhc_get_status)         */
#define MHC_ERR_WORKSPACE -7  /* workspace missing or smaller than *_workspace_bytes()           */
#define MHC_ERR_BOUNDS    -8  /* bounds-checked build only: an index check failed and its access
                                 was skipped (see mhc_get_status, mhc_checked_build)           */

/* ---- flags ------------------------------------------------------------------------------- */
/* Reading of comb in hc_post. Default (0): the pages' code, X'_k = u_k F + sum_j C_jk X_j
 * (Stream weights for the feed-forward, Code: hc_post sums over comb's first stream index).
 * MHC_COMB_ROW_DEST: X'_j = u_j F + sum_k C_jk X_k (element (i,j) = "from stream j into stream i",
 * "2A · Single-Pass mHC", section 3).                                                        */
#define MHC_COMB_ROW_DEST        0x1u
/* Test hook: one thread per CTA waits on a barrier that nothing completes, with a ~2 ms limit;
 * the wait gives up, records MHC_ERR_TIMEOUT for mhc_get_status, and the call completes.      */
#define MHC_DEBUG_NEVER_ARRIVE   0x2u
/* Test hook of the bounds-checked build only (MHC_ERR_SHAPE in other builds): one finisher
 * store and one MXFP8 scale store of the first CTA get a row index N rows past the end; the
 * index checks skip both and mhc_get_status reports MHC_ERR_BOUNDS.                          */
#define MHC_DEBUG_PLANT_OOB      0x4u
/* Bits 8..11: log2 + 1 of the number of CTAs (1, 2, 4, 8, 16 or 32) that split the width d of
 * each token tile between them (a group of co-resident CTAs); values above 6 are MHC_ERR_SHAPE.
 * 0 = automatic: with the tile height (below), the shape that minimises the busiest group's
 * work: wider groups for few tokens, the fewest CTAs per tile for many.                       */
#define MHC_SPLIT_SHIFT          8
#define MHC_SPLIT_MASK           (0xFu << MHC_SPLIT_SHIFT)
/* Bits 16..20: tokens per tile of the step kernel / 8 (1..16, i.e. 8..128 tokens; larger values
 * are MHC_ERR_SHAPE; the height must be a multiple of the split). 0 = automatic (above).      */
#define MHC_TILE_SHIFT           16
#define MHC_TILE_MASK            (0x1Fu << MHC_TILE_SHIFT)
/* Launch path of the fused step with bf16 y (mhc_fused_step, _packed, _noalloc). Two kernels
 * compute the same step (X' bit for bit; the other outputs within the stated tolerances, their
 * partial sums being added in another order):
 *   the persistent kernel: one cooperative launch, one CTA per SM; groups of `split` CTAs walk
 *     128-token tiles and sum their partial results through the step scratch (L2);
 *   the cluster kernel: one thread-block cluster of 16 CTAs (8 where d needs it) per tile of
 *     40 tokens, summing through distributed shared memory; d / (32 x cluster size) <= 10
 *     (d = 5120: 16 CTAs of 320 columns). Made for small batches (decode).
 * Default (neither bit): the cluster kernel when d fits it and every tile's cluster runs at once
 * on the device (up to 280 tokens at d = 5120 on a 152-SM GB300: 7 clusters of 16 CTAs), the
 * persistent kernel otherwise, and
 * always the persistent kernel when the split or tile bits are set.
 * MHC_PATH_PERSISTENT: always the persistent kernel.
 * MHC_PATH_CLUSTER: always the cluster kernel, for any N (clusters beyond what the device runs
 *   at once wait for a free place); the split bits then choose its cluster size (0: 16 where d
 *   fits, else 8; 4 = 8 CTAs; 5 = 16 CTAs); MHC_ERR_SHAPE with the tile bits, with
 *   MHC_PATH_PERSISTENT, where d fits no cluster size, or in calls without bf16 y (mhc_mixes,
 *   mhc_fused_step_mxfp8). The cluster kernel ignores the step scratch.                      */
#define MHC_PATH_PERSISTENT      0x8u
#define MHC_PATH_CLUSTER         0x10u

/* ---- sizes ------------------------------------------------------------------------------- */
/* Bytes of the packed projection weights (3 bf16 planes of W_mix plus padding, in the layout
 * described at mhc_pack_weights). 0 if (n, d) cannot be packed.                             */
size_t mhc_packed_weights_bytes(int n, int d);
/* Columns of d per block of the packed weights (B below).                                    */
int mhc_packed_block_columns(void);
/* Scratch of the step kernel on the CURRENT device: the exchange area through which the CTAs
 * that share a token tile sum their partial results (counters and partial sums; it grows with
 * the device's SM count, about 4.4 MB on a 152-SM GB300). 0 if no device can be queried.     */
size_t mhc_step_scratch_bytes(int n, int d);
/* Workspace of mhc_fused_step / mhc_mixes on the current device: the packed weights (rounded
 * up to 256 bytes) followed by the step scratch.                                             */
size_t mhc_workspace_bytes(int n, int d);

/* ---- the fused single-pass step ------------------------------------------------------------
 * One sublayer of the single-pass mHC step (MoE RMSNorm, Code: Block.forward, FFN half;
 * Stream weights for the feed-forward, "Why" and "All 5 steps"), in ONE kernel pass over the
 * streams:
 *   X'   = hc_post(X, F, post_prev, comb_prev)                  -> X_out  (bf16, rounded)
 *   m    = (flatten(X') W_mix^T) / sqrt(mean(flatten(X')^2) + norm_eps)      -> mixes_out
 *   pre  = sigmoid(scale[0] m[0:n] + base[0:n]) + hc_eps                     -> pre_out
 *   post = 2 sigmoid(scale[1] m[n:2n] + base[n:2n])                          -> post_out
 *   comb = Sinkhorn(softmax_k(scale[2] m[2n:] + base[2n:]) ), sinkhorn_iters rounds -> comb_out
 *   y    = RMSNorm(hc_pre(X', pre_prev); gain, norm_eps)                     -> y_out (bf16)
 * hc_post and hc_pre are evaluated in float32 as the pages' code spells them out (Code:
 * hc_post, hc_pre: every product a float32 tensor, summed over the stream index), each product
 * and each addition rounded to float32, the sums in stream order, then rounded to bf16
 * (fl = one float32 rounding):
 *   X'_k  = fl(u_k F) + (((fl(C_0k X_0) + fl(C_1k X_1)) + fl(C_2k X_2)) + fl(C_3k X_3))
 *   y_hat = ((fl(p_0 X'_0) + fl(p_1 X'_1)) + fl(p_2 X'_2)) + fl(p_3 X'_3)
 *
 *   X         bf16 [N, n, d]      residual streams                      (read once)
 *   F         bf16 [N, d]         sublayer output                        (read once)
 *   pre_prev  fp32 [N, n]         previous reading weights (used by hc_pre)
 *   post_prev fp32 [N, n]         previous writing weights (used by hc_post)
 *   comb_prev fp32 [N, n, n]      previous stream combination (used by hc_post)
 *   W_mix     fp32 [(2+n)n, n*d]  projection, flat index k*d + i (stream-major)
 *   scale     fp32 [3], base fp32 [(2+n)n], gain fp32 [d]
 *   X_out     bf16 [N, n, d]      may equal X (in place); no other overlap
 *   y_out     bf16 [N, d]
 *   pre_out, post_out fp32 [N, n]; comb_out fp32 [N, n, n]; mixes_out fp32 [N, (2+n)n] or NULL
 *   d: for some split of 1, 2, 4, 8, 16 or 32 CTAs per tile, d/split is a multiple of B
 *      (B = mhc_packed_block_columns()) between 4B and 640; d = 5120 runs with 8, 16 or 32
 *      CTAs per tile, d <= 20480 at most.
 *   workspace: >= mhc_workspace_bytes(n, d) device bytes; W_mix is packed into its start each
 *      call and the rest is the step scratch. Calls that share a workspace or scratch buffer
 *      must not overlap in time on the GPU (put them on one stream).
 * The launch is cooperative (one CTA per SM, all resident); MHC_ERR_CUDA if the device cannot
 * hold it (for example while other work occupies SMs of an MPS partition).
 * Returns MHC_OK or a negative code. N == 0 returns MHC_OK once the shape is valid, without
 * looking at the pointers (empty tensors may have none) and without launching.               */
int mhc_fused_step(const void* X, const void* F, const float* pre_prev, const float* post_prev,
                   const float* comb_prev, const float* W_mix, const float* scale,
                   const float* base, const float* gain, void* X_out, void* y_out,
                   float* pre_out, float* post_out, float* comb_out, float* mixes_out,
                   int64_t N, int n, int d, int sinkhorn_iters, float hc_eps, float norm_eps,
                   unsigned flags, void* workspace, size_t workspace_bytes, void* stream);

/* Same step with W_mix already packed by mhc_pack_weights (no per-call packing); `scratch` is
 * >= mhc_step_scratch_bytes(n, d) device bytes.                                              */
int mhc_fused_step_packed(const void* X, const void* F, const float* pre_prev,
                          const float* post_prev, const float* comb_prev, const void* W_packed,
                          const float* scale, const float* base, const float* gain, void* X_out,
                          void* y_out, float* pre_out, float* post_out, float* comb_out,
                          float* mixes_out, int64_t N, int n, int d, int sinkhorn_iters,
                          float hc_eps, float norm_eps, unsigned flags, void* scratch,
                          size_t scratch_bytes, void* stream);

/* ---- the fused step with y quantised for the next sublayer ----------------------------------
 * The pages name an FP4/FP8 MoE as a consumer of y ("2A · Single-Pass mHC", section 2, the flow
 * diagram) but define no quantised format; this entry writes y in the OCP Microscaling (MX) v1.0
 * format MXFP8 instead of bf16, fused into the same single pass. It runs the persistent kernel;
 * everything else is as in mhc_fused_step_packed with MHC_PATH_PERSISTENT (same X', p, u, C and
 * optional mixes, bit for bit).
 *   y_codes  uint8 [N, d]       E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
 *                                no infinities)
 *   y_scale  uint8 [N, d / 32]  E8M0 codes: block b of token t (features 32b .. 32b + 31) has
 *                                scale X = 2^(y_scale[t, b] - 127)
 * The encoded values are the bf16 y that mhc_fused_step_packed returns with MHC_PATH_PERSISTENT
 * for the same inputs (bit for bit), so the codes equal a separate MXFP8 pass over that y: X = 2^(floor(log2(amax)) - 8)
 * with amax the block's largest |y| (code clamped to >= 0; an all-zero block takes code 0); each
 * code is y / X rounded to the nearest E4M3 value, ties to even, saturating at +-448.
 * Dequantised: y ~= value(code) * X.
 * Both pointers 16-byte aligned, neither overlapping another argument.                       */
int mhc_fused_step_mxfp8(const void* X, const void* F, const float* pre_prev,
                         const float* post_prev, const float* comb_prev, const void* W_packed,
                         const float* scale, const float* base, const float* gain, void* X_out,
                         void* y_codes, void* y_scale, float* pre_out, float* post_out,
                         float* comb_out, float* mixes_out, int64_t N, int n, int d,
                         int sinkhorn_iters, float hc_eps, float norm_eps, unsigned flags,
                         void* scratch, size_t scratch_bytes, void* stream);

/* ---- gradients of the step (training) -------------------------------------------------------
 * The pages define the forward step only; no page describes a backward pass. The gradients
 * computed are those of reverse-mode differentiation of the pages' forward code (Stream weights
 * for the feed-forward, Code: hc_post, hc_mixes, hc_pre, hc_split_sinkhorn; MoE RMSNorm, Code:
 * RMSNorm, Block.forward) with its casts to bf16 passed straight through, every derivative taken
 * at the values the forward computed. Per token, with x = flat(X'), K = 4d,
 * r = (|x|^2/K + norm_eps)^(-1/2), r_y = (|y_hat|^2/d + norm_eps)^(-1/2), T = sum gain gy y_hat:
 *   g_m (24) from (gpre, gpost, gcomb) through the split and every Sinkhorn round;
 *   g_y_hat = r_y gain gy - (r_y^3 T / d) y_hat;
 *   g_X'_k = gXp_k + p_k g_y_hat + (W^T (r g_m))_k - (r^2/K)(g_m . m) X'_k;
 *   gX_j = sum_k C_jk g_X'_k; gF = sum_k u_k g_X'_k; gpost_prev_k = g_X'_k . F;
 *   gcomb_prev_jk = g_X'_k . X_j; gpre_prev_j = g_y_hat . X'_j;
 *   gW = sum over tokens of (r g_m) x^T; ggain = sum of r_y gy y_hat; gbase, gscale from the split.
 * (MHC_COMB_ROW_DEST: the other comb reading, as in the forward.)
 * Inputs (device, layouts as for mhc_fused_step):
 *   X, F, pre_prev, post_prev, comb_prev, W_mix [24, 4d] fp32, scale, base, gain   the forward's inputs
 *   Xp    bf16 [N, 4, d]   the forward's X' output (saved activation)
 *   mixes fp32 [N, 24]     the forward's mixes output m (saved activation)
 *   gXp bf16 [N, 4, d], gy bf16 [N, d], gpre, gpost fp32 [N, 4], gcomb fp32 [N, 4, 4]
 *                          gradients of the forward's outputs X', y, p, u, C
 * Outputs (device): gX bf16 [N, 4, d], gF bf16 [N, d], gpre_prev, gpost_prev fp32 [N, 4],
 *   gcomb_prev fp32 [N, 4, 4]; gW fp32 [24, 4d], gbase fp32 [24], gscale fp32 [3],
 *   ggain fp32 [d] (sums over the N tokens; written, not accumulated; zero when N = 0).
 * workspace: >= mhc_backward_workspace_bytes(N, n, d) device bytes, 16-byte aligned.
 * Shapes: n = 4, d a multiple of 64, sinkhorn_iters >= 1 (MHC_ERR_SHAPE); flags other than
 * MHC_COMB_ROW_DEST are MHC_ERR_SHAPE. No output may overlap an input or another output.
 * Five kernels run in order on `stream`.                                                      */
int mhc_fused_step_backward(const void* X, const void* F, const void* Xp, const float* mixes,
                            const float* pre_prev, const float* post_prev, const float* comb_prev,
                            const float* W_mix, const float* scale, const float* base,
                            const float* gain, const void* gXp, const void* gy, const float* gpre,
                            const float* gpost, const float* gcomb, void* gX, void* gF,
                            float* gpre_prev, float* gpost_prev, float* gcomb_prev, float* gW,
                            float* gbase, float* gscale, float* ggain, int64_t N, int n, int d,
                            int sinkhorn_iters, float hc_eps, float norm_eps, unsigned flags,
                            void* workspace, size_t workspace_bytes, void* stream);
/* Workspace bytes of mhc_fused_step_backward on the current device (0 if the shape is
 * unsupported).                                                                               */
size_t mhc_backward_workspace_bytes(int64_t N, int n, int d);

/* ---- the fused step without any allocation --------------------------------------------------
 * No counterpart in the paper: an addition for callers that cannot allocate device memory when
 * they run the step -- a serving loop that runs under a fixed device-memory budget, or whose
 * caching allocator it may not enter from that point, or a plain C host that links this library
 * and has no device allocator of its own. Same arguments and results as mhc_fused_step, without the workspace:
 * the packed weights and the step scratch live in one fixed array of
 * mhc_noalloc_scratch_bytes() (8 MiB) that the library keeps on every GPU that loads it until
 * the process exits. No device memory is allocated or freed, by this call or by anything it
 * calls. Returns MHC_ERR_WORKSPACE when the packed weights for d plus the step scratch for the
 * current device do not fit that array (n = 4: d <= 5120 fits on devices of up to 178 SMs).
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture. All calls on a device share the array and leave
 * the last call's contents in it (the step clears what it needs zeroed), so calls that overlap
 * on the GPU -- on different streams, or from different threads -- race: serialise them.   */
int mhc_fused_step_noalloc(const void* X, const void* F, const float* pre_prev,
                           const float* post_prev, const float* comb_prev, const float* W_mix,
                           const float* scale, const float* base, const float* gain, void* X_out,
                           void* y_out, float* pre_out, float* post_out, float* comb_out,
                           float* mixes_out, int64_t N, int n, int d, int sinkhorn_iters,
                           float hc_eps, float norm_eps, unsigned flags, void* stream);
/* Bytes of the fixed per-device array mhc_fused_step_noalloc uses.                          */
size_t mhc_noalloc_scratch_bytes(void);

/* ---- the fused step on host-resident streams -------------------------------------------------
 * No counterpart in the paper (its step runs on device tensors): the same step as
 * mhc_fused_step for a caller whose per-token tensors are in HOST memory. The tokens are cut
 * into chunks (see mhc_host_chunks); chunk i is copied into device staging slot i%3, stepped,
 * and copied back, on three internal streams of the current device, so that the host->device copy
 * of chunk i+1, the step on chunk i and the device->host copy of chunk i-1 overlap. The
 * internal streams start after the work already queued on `stream`, and `stream` continues only
 * after the last output has reached the host: synchronise `stream` before reading the outputs
 * or reusing the inputs.
 *   X, F, pre_prev, post_prev, comb_prev   HOST pointers, layouts as for mhc_fused_step
 *   X_out, y_out, pre_out, post_out, comb_out, mixes_out (or NULL)   HOST pointers, same layouts;
 *        X_out may equal X (chunk i's inputs are read before its outputs are written), no other
 *        overlap (not checked on the host side). Page-locked (pinned) host memory is needed for
 *        the copies to overlap; pageable memory gives the same results, serialised.
 *   W_mix, scale, base, gain   DEVICE pointers (parameters stay resident on the GPU).
 *   staging: >= mhc_host_staging_bytes(n, d, chunk_tokens, mixes_out != NULL) device bytes,
 *        256-byte aligned (MHC_ERR_ALIGN otherwise): the workspace of mhc_fused_step followed by
 *        three slots of chunk_tokens tokens' inputs and outputs.
 * The internal streams and events are shared by all calls on a device: calls that overlap in
 * time -- from different threads, or on different caller streams -- must be serialised.
 * Returns MHC_OK or a negative code (as mhc_fused_step; MHC_ERR_SHAPE also for chunk_tokens
 * < 1). An error returned part way leaves the chunks already queued to complete.          */
int mhc_fused_step_host(const void* X, const void* F, const float* pre_prev,
                        const float* post_prev, const float* comb_prev, const float* W_mix,
                        const float* scale, const float* base, const float* gain, void* X_out,
                        void* y_out, float* pre_out, float* post_out, float* comb_out,
                        float* mixes_out, int64_t N, int n, int d, int sinkhorn_iters,
                        float hc_eps, float norm_eps, unsigned flags, void* staging,
                        size_t staging_bytes, int64_t chunk_tokens, void* stream);
/* Device bytes of the staging buffer of mhc_fused_step_host; 0 for an invalid shape or chunk. */
size_t mhc_host_staging_bytes(int n, int d, int64_t chunk_tokens, int with_mixes);
/* The chunks mhc_fused_step_host cuts N tokens into, in order: writes the first min(count,
 * max_chunks) token counts to `counts` (may be NULL) and returns the count, or MHC_ERR_SHAPE for
 * N < 0 or chunk_tokens < 1. When N >= 2(c/8 + c/4 + c/2) + c (c = chunk_tokens, c >= 8), the
 * first three chunks are c/8, c/4, c/2 tokens and the last three c/2, c/4, c/8, so that the
 * copy-in before the first step and the copy-out after the last, which overlap nothing, stay
 * short; the chunks between hold c tokens, the last of them the remainder. Otherwise every chunk
 * holds c tokens but the last.                                                                */
int64_t mhc_host_chunks(int64_t N, int64_t chunk_tokens, int64_t* counts, int64_t max_chunks);

/* ---- hc_mixes alone ------------------------------------------------------------------------
 * Stream weights for the feed-forward, Code: hc_mixes (+ the hc_split_sinkhorn kernel): from
 * bf16 streams X [N,n,d], the 24 mix numbers m (optional output) and pre/post/comb as above.
 * Same shape rules and workspace as mhc_fused_step.                                          */
int mhc_mixes(const void* X, const float* W_mix, const float* scale, const float* base,
              float* mixes_out, float* pre_out, float* post_out, float* comb_out, int64_t N,
              int n, int d, int sinkhorn_iters, float hc_eps, float norm_eps, unsigned flags,
              void* workspace, size_t workspace_bytes, void* stream);

/* ---- split + Sinkhorn alone ----------------------------------------------------------------
 * Stream weights for the feed-forward, Code: hc_split_sinkhorn kernel. mixes fp32 [N,(2+n)n]
 * -> pre, post fp32 [N,n], comb fp32 [N,n,n]. Any N >= 0, sinkhorn_iters >= 1.            */
int mhc_sinkhorn(const float* mixes, const float* scale, const float* base, float* pre_out,
                 float* post_out, float* comb_out, int64_t N, int n, int sinkhorn_iters,
                 float hc_eps, void* stream);

/* ---- RMSNorm alone -------------------------------------------------------------------------
 * MoE RMSNorm, formula block and Code: RMSNorm. x bf16 [N,d] -> y = bf16(gain * x /
 * sqrt(mean(x^2) + eps)) [N,d]. d multiple of 8; y may equal x.                              */
int mhc_rmsnorm(const void* x, const float* gain, void* y, int64_t N, int d, float eps,
                void* stream);

/* ---- the unfused form, one op per kernel ---------------------------------------------------
 * The earlier form the page "Stream weights for the feed-forward" ("Why") compares against:
 * hc_post, hc_mixes and hc_pre as separate kernels (plus RMSNorm), each a full pass over the
 * streams. Same arithmetic as the fused step; used to measure the (4n+4)d vs (2n+2)d traffic.
 * mhc_hc_post: X, F, post, comb -> X_out bf16 [N,n,d] (flags: MHC_COMB_ROW_DEST).
 * mhc_hc_pre:  X' bf16 [N,n,d], pre fp32 [N,n] -> y_hat bf16 [N,d].  d multiple of 8.        */
int mhc_hc_post(const void* X, const void* F, const float* post, const float* comb, void* X_out,
                int64_t N, int n, int d, unsigned flags, void* stream);
int mhc_hc_pre(const void* Xp, const float* pre, void* y_hat, int64_t N, int n, int d,
               void* stream);

/* ---- weights packing -----------------------------------------------------------------------
 * Split fp32 W_mix [(2+n)n, n*d] into three bf16 planes hi + mid + lo (each the bf16 rounding
 * of what the previous planes left); the three planes carry W to float32 accuracy for the
 * tensor cores. The packed buffer is the fused kernel's shared-memory image, d/B blocks of B
 * columns (B = mhc_packed_block_columns()): block b = [n streams][80 rows][B columns] bf16 of
 * columns [b*B, (b+1)*B) of each stream; plane pl (0 hi, 1 mid, 2 lo) of mix row r is row
 * 36*(r/12) + 12*pl + r%12, rows 72..79 are zero, and the 16-byte chunks of each row are
 * swizzled: chunk c of row r is stored at chunk c ^ ((r*2B/128) mod (B/8)).
 * d must be a multiple of B.                                                                 */
int mhc_pack_weights(const float* W_mix, void* W_packed, int n, int d, void* stream);

/* ---- status --------------------------------------------------------------------------------
 * Synchronises `stream`, then returns and clears the device status word: MHC_OK,
 * MHC_ERR_BOUNDS if an index check of the bounds-checked build failed since the last call,
 * else MHC_ERR_TIMEOUT if a bounded device-side wait gave up, or MHC_ERR_CUDA if the
 * synchronisation itself failed.                                                              */
int mhc_get_status(void* stream);
/* 1 for the bounds-checked build of the library (libmhc_checked.so: every copy, store and
 * exchange access of the fused step tests its index first and skips it on failure, reporting
 * MHC_ERR_BOUNDS), 0 for the regular build (the tests compiled away).                          */
int mhc_checked_build(void);
/* The kernel mhc_fused_step runs for N tokens of width d with `flags` on the current device:
 * MHC_PATH_PERSISTENT or MHC_PATH_CLUSTER (see the flags above), or a negative code.          */
int mhc_step_path(int64_t N, int n, int d, unsigned flags);

/* Launch shape of the fused step (and of mhc_mixes) for N tokens of width d with `flags` on
 * the current device: CTAs that share a tile, tokens per tile, and groups launched (each group
 * is `split` CTAs, one per SM). On the cluster path (mhc_step_path): the cluster size, 40, and
 * the number of clusters. Diagnostic; needs a GPU.                                           */
int mhc_step_config(int64_t N, int n, int d, unsigned flags, int* split, int* tile, int* groups);
/* Phase tracing of the fused step's persistent kernel (off by default; the cluster kernel
 * records nothing). With a device buffer set, every later launch whose grid fits records, per
 * (tile, rank in its group), 8 uint64 values from the GPU's nanosecond timer: slot 0 the tile's
 * start; slots 1..6 nanoseconds since then at: the producer issued the tile's loads, the
 * consumers' main loop done, the tile's partial sums posted, (unused), the finisher done, the
 * consumers' tile end; slot 7 the nanoseconds to the kernel's end, with the SM id in bits 40
 * and up. Record index = tile * split + rank. Launches with more records than the buffer holds
 * (64 bytes each) record nothing. NULL turns tracing off. The buffer stays caller-owned; it
 * must outlive the launches that write it. Not thread-safe.                                  */
int mhc_set_trace(void* buffer, int64_t bytes);
/* Static text for a status code.                                                              */
const char* mhc_strerror(int code);
/* Library ABI version (major*100 + minor): 101.                                               */
int mhc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MHC_H */

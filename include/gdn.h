/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet layer core.
 *
 * The core is the linear-attention block of Qwen3-Next / Qwen3.5-style models
 * as defined by "mlex 0.1.2, src/models/gated_delta.rs" (GatedDeltaNet::load and
 * GatedDeltaNet::forward) and by "mlx-bun 0.4.0 -> 1.0.0,
 * package/src/model/qwen3-delta.ts" (the numerics table at its head, the
 * gated_delta_step kernel and its masked specialization, computeG,
 * gatedDeltaUpdate):
 *
 *   conv window   X = [conv_state || qkv] along time, conv_state' = last K-1 rows
 *   conv + SiLU   u[t,c] = sum_j w[c,j] X[t+j,c] (tap K-1 = current token); x = u*sigmoid(u)
 *   q/k norm      q = rms(x_q)/Dk, k = rms(x_k)/sqrt(Dk), v = x_v; rms(x) = x/sqrt(mean(x^2)+eps)
 *   gates         g = exp(-exp(A_log) * softplus(a + dt_bias)), beta = sigmoid(b)
 *   recurrence    per (b, hv), hk = hv / (Hv/Hk):  S <- g S;  delta = beta (v - S k);
 *                 S <- S + delta k^T;  y = S q          (S is [Dv, Dk], f32)
 *   mask          a step with mask 0 writes zero y (and zero q/k/v), does not enter
 *                 the conv window and leaves both states untouched.
 *
 * Conventions shared by every entry point
 *   - Memory: every pointer is a DEVICE pointer owned by the caller.  The library
 *     allocates nothing and keeps no state between calls except one device error
 *     word per device (see gdn_device_status).
 *   - Types: "bf16" buffers hold bfloat16 bit patterns (uint16_t); "f32" is IEEE
 *     single.  Every tensor is dense and row-major with the shape given.
 *   - Alignment: every tensor pointer must be 16-byte aligned, else
 *     GDN_ERR_INVALID_ARG.
 *   - Streams: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and the call returns without waiting.  Argument errors are
 *     reported before anything is enqueued; GDN_ERR_CUDA reports a launch error.
 *   - Supported sizes: Dk, Dv in {32, 64, 128}; Hv % Hk == 0; 2 <= K <= 4;
 *     B, T >= 0 (a zero size is a no-op).  Others give GDN_ERR_UNSUPPORTED.
 *   - Channel order of qkv / conv_state / conv_w: C = 2*Hk*Dk + Hv*Dv channels,
 *     q heads [0, Hk*Dk), k heads [Hk*Dk, 2*Hk*Dk), v heads [2*Hk*Dk, C), each
 *     head's channels contiguous.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols keep default visibility even when the library is built
 * with hidden visibility. */
#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st *gdn_stream;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, negative size, Hv % Hk != 0 */
    GDN_ERR_UNSUPPORTED = 2,   /* a size outside the supported set above */
    GDN_ERR_CUDA = 3,          /* a CUDA launch or attribute call failed */
    GDN_ERR_TIMEOUT = 4        /* a bounded on-device wait gave up (see gdn_device_status) */
} gdn_status;

/* Problem sizes: the fields of GatedDeltaConfig (mlex gated_delta.rs) plus the
 * batch B and the number of time steps T of this call.  eps_qk is the q/k
 * rms-norm epsilon (1e-6 on the pages). */
typedef struct gdn_dims {
    int32_t B, T, Hk, Hv, Dk, Dv, K;
    float eps_qk;
} gdn_dims;

/* Causal depthwise conv + SiLU + q/k rms-norm and scaling, with the rolling
 * conv state.  (mlex gated_delta.rs, GatedDeltaNet::forward: the conv_state
 * concat/slice, conv1d with groups = conv_dim, silu, split into q/k/v, rms_norm
 * and the inv_scale factors.)
 *   qkv        bf16 [B, T, C]      pre-conv input (in)
 *   conv_w     bf16 [C, K]         depthwise weights, tap K-1 = current token (in)
 *   conv_state bf16 [B, K-1, C]    in/out: the K-1 most recent valid raw inputs,
 *                                  oldest first; NULL = zeros and not returned
 *   mask       u8   [B, T]         nonzero = valid step; NULL = all valid
 *   q, k       bf16 [B, T, Hk, Dk] out; v bf16 [B, T, Hv, Dv] out.  One
 *                                  round-to-nearest-even rounding of the f32
 *                                  result; masked steps are written as zeros.
 * qkv must not alias any output. */
GDN_API gdn_status gdn_conv_update(const gdn_dims *dims, const uint16_t *qkv, const uint16_t *conv_w,
                           uint16_t *conv_state, const uint8_t *mask,
                           uint16_t *q, uint16_t *k, uint16_t *v, gdn_stream stream);

/* Gates. (mlex gated_delta.rs, GatedDeltaNet::forward: beta and g; mlx-bun
 * qwen3-delta.ts, computeG.)
 *   a, b        bf16 [B, T, Hv] (in);  A_log, dt_bias f32 [Hv] (in)
 *   g, beta     f32  [B, T, Hv] (out): g = exp(-exp(A_log) softplus(a + dt_bias)),
 *               beta = sigmoid(b), softplus(x) = max(x,0) + log1p(exp(-|x|)). */
GDN_API gdn_status gdn_gating(const gdn_dims *dims, const uint16_t *a, const uint16_t *b,
                      const float *A_log, const float *dt_bias, float *g, float *beta,
                      gdn_stream stream);

/* One decode step (dims->T must be 1), fully fused: conv window + conv + SiLU
 * + q/k norm, gates, and the recurrence step, in one kernel that streams the
 * f32 state once.  (mlx-bun qwen3-delta.ts, gated_delta_step at T = 1;
 * mlex gated_delta.rs, GatedDeltaNet::forward with a one-token input.)
 *   qkv        bf16 [B, C] (in)            conv_w bf16 [C, K] (in)
 *   conv_state bf16 [B, K-1, C] in/out (required)
 *   a, b       bf16 [B, Hv] (in)           A_log, dt_bias f32 [Hv] (in)
 *   state      f32  [B, Hv, Dv, Dk] in/out, updated in place
 *   row_mask   u8   [B] or NULL: a zero row writes y = 0 and leaves both of its
 *              states untouched
 *   y          bf16 [B, Hv, Dv] (out)
 * Supports Hv/Hk <= 16. */
GDN_API gdn_status gdn_recurrent_decode(const gdn_dims *dims, const uint16_t *qkv, const uint16_t *conv_w,
                                uint16_t *conv_state, const uint16_t *a, const uint16_t *b,
                                const float *A_log, const float *dt_bias, float *state,
                                const uint8_t *row_mask, uint16_t *y, gdn_stream stream);

/* Decode steps fed from and returned to host memory: n_steps consecutive
 * tokens of gdn_recurrent_decode (same arithmetic, same kernel), with each
 * step's inputs copied in from host buffers and its y copied out to a host
 * buffer inside the call, as a serving loop does.  (Same definitions as
 * gdn_recurrent_decode.)
 *   qkv_h      bf16 [n_steps, B, C]       host (in), step i's qkv at row i
 *   a_h, b_h   bf16 [n_steps, B, Hv]      host (in)
 *   y_h        bf16 [n_steps, B, Hv, Dv]  host (out)
 *   conv_w, conv_state, A_log, dt_bias, state, row_mask: device, as in
 *              gdn_recurrent_decode (row_mask applies to every step)
 *   staging    device workspace of gdn_decode_host_staging_size(dims) bytes,
 *              16-byte aligned: four slots of qkv, a, b and y, so that the
 *              next steps' inputs travel and earlier steps' y return while
 *              step i runs
 * Host buffers should be page-locked (cudaHostAlloc / pinned): pageable
 * memory is accepted but its copies do not overlap the kernels.  The copies
 * run on two copy streams of the library (cudaMemcpyAsync, one per tensor and
 * step) and are ordered against `stream` with events; the streams and events
 * are created on a device's first call and kept until the process exits, and
 * calls from several host threads enqueue one after the other (a lock per
 * device; their copies then share the two streams).  Everything is enqueued
 * before the call returns and `stream` completes after the last y has
 * arrived, so synchronise `stream` before reading y_h.  Neither host buffer
 * may be written (inputs) or read (y_h) before that.  n_steps = 0 is a no-op.
 * Errors: GDN_ERR_INVALID_ARG for a bad argument or a short staging buffer,
 * GDN_ERR_CUDA for a failed CUDA call (work already enqueued still runs). */
GDN_API gdn_status gdn_recurrent_decode_host_steps(const gdn_dims *dims, int n_steps, const uint16_t *qkv_h,
                                                   const uint16_t *a_h, const uint16_t *b_h, uint16_t *y_h,
                                                   const uint16_t *conv_w, uint16_t *conv_state,
                                                   const float *A_log, const float *dt_bias, float *state,
                                                   const uint8_t *row_mask, void *staging, size_t staging_bytes,
                                                   gdn_stream stream);

/* Bytes of device staging gdn_recurrent_decode_host_steps needs (0 for bad
 * dims). */
GDN_API size_t gdn_decode_host_staging_size(const gdn_dims *dims);

/* gdn_recurrent_decode followed by the layer's RMSNormGated.  The norm runs
 * in the decode kernel's epilogue when one CTA holds all Dv rows of a head
 * (for example Hv/Hk = 16 or Dv = 32 with few heads); when a head's rows are
 * spread over several CTAs, the decode kernel writes y into `out` and a
 * second kernel normalises it in place, which measured faster than an
 * exchange of partial sums between the CTAs.  (mlex gated_delta.rs,
 * GatedDeltaNet::forward: the f32 rms_norm of y over Dv with norm_eps, times
 * the norm weight, times silu(z), cast to bf16.)  Per (b, hv):
 *   out = bf16( silu(z) * norm_w * yb / sqrt(mean_Dv(yb^2) + norm_eps) )
 * where yb is the bf16-rounded recurrence output (the y gdn_recurrent_decode
 * would write), so the result equals gdn_recurrent_decode followed by
 * gdn_rmsnorm_gated up to f32 summation order.
 *   z          bf16 [B, Hv, Dv] (in): the in_proj_z output of the token
 *   norm_w     f32  [Dv] (in);  norm_eps >= 0
 *   out        bf16 [B, Hv, Dv] (out); a zero row of row_mask gives zeros
 *              (its y is 0; the sign of a zero follows silu(z) * norm_w)
 * Other arguments and limits as gdn_recurrent_decode. */
GDN_API gdn_status gdn_recurrent_decode_gated(const gdn_dims *dims, const uint16_t *qkv,
                                              const uint16_t *conv_w, uint16_t *conv_state,
                                              const uint16_t *a, const uint16_t *b, const float *A_log,
                                              const float *dt_bias, float *state, const uint8_t *row_mask,
                                              const uint16_t *z, const float *norm_w, float norm_eps,
                                              uint16_t *out, gdn_stream stream);

/* Multi-token decode window for speculative verification: dims->T (1..8)
 * new tokens per row, fused like gdn_recurrent_decode (one pass over the f32
 * state).  y is written for all T tokens; conv_state and state are advanced by
 * exactly keep[b] leading tokens of row b, so a verify call with keep = NULL
 * (all tokens) or a commit call with the accepted counts gives the state after
 * the accepted prefix.  (mlx-bun qwen3-delta.ts, SsmSpecRound and
 * specRoundRollback: a window of S tokens whose first `keep` are kept, the
 * state after them being the same arithmetic prefix; gated_delta_step.)
 *   qkv        bf16 [B, T, C] (in)          conv_w bf16 [C, K] (in)
 *   conv_state bf16 [B, K-1, C] in/out      a, b bf16 [B, T, Hv] (in)
 *   A_log, dt_bias f32 [Hv] (in)            state f32 [B, Hv, Dv, Dk] in/out
 *   keep       int32 [B] or NULL (= T); values are clamped to [0, T]; 0 leaves
 *              both states untouched (y is still produced)
 *   y          bf16 [B, T, Hv, Dv] (out)
 * Supports Hv/Hk <= 16; dims->T outside 1..8 gives GDN_ERR_UNSUPPORTED. */
GDN_API gdn_status gdn_decode_window(const gdn_dims *dims, const uint16_t *qkv, const uint16_t *conv_w,
                                     uint16_t *conv_state, const uint16_t *a, const uint16_t *b,
                                     const float *A_log, const float *dt_bias, float *state,
                                     const int32_t *keep, uint16_t *y, gdn_stream stream);

/* The recurrence over T steps (prefill).  (mlx-bun qwen3-delta.ts,
 * gatedDeltaUpdate and the gated_delta_step kernel with its masked
 * specialization; mlex gated_delta.rs, the per-timestep loop.)
 *   q, k       bf16 [B, T, Hk, Dk] (in)    v bf16 [B, T, Hv, Dv] (in)
 *   g, beta    f32  [B, T, Hv] (in)
 *   state_in   f32  [B, Hv, Dv, Dk] or NULL (= zeros)
 *   state_out  f32  [B, Hv, Dv, Dk] (out); may equal state_in
 *   mask       u8   [B, T] or NULL
 *   y          bf16 [B, T, Hv, Dv] (out)
 *   chunk      0 = sequential form (state resident on chip across all T);
 *              64 = chunked (WY / UT-transform) form on the tensor cores
 *   workspace  optional device scratch of at least gdn_prefill_workspace_size()
 *              bytes, 16-byte aligned, or NULL.  With a mask, the call first
 *              writes there the order in which rows are handed to the kernel's
 *              CTAs (most chunks holding a valid step first), so that the
 *              longest rows of a ragged batch do not start last; with NULL the
 *              rows go in index order.  With chunk = 64 and fewer heads
 *              (B * Hv) than the GPU has SMs, the size also covers the
 *              two-pass chunked form (about 145 KiB per head and chunk of 64
 *              steps): the state-independent work of all chunks first runs
 *              over the whole GPU and is kept there, then one pass per head
 *              applies it to the state.  The results are the same, bit for
 *              bit, whichever way the call runs.  A workspace smaller than
 *              the two-pass size but at least the row-order size runs the
 *              single pass; a smaller or misaligned one gives
 *              GDN_ERR_INVALID_ARG.  It must not be in use by another call
 *              still running on another stream.
 * Wholly masked 64-step chunks cost only their zero y stores.
 * The chunked form reads q, k, v of masked steps (their contribution is then
 * cancelled exactly), so those entries must hold finite values; the zeros
 * gdn_conv_update writes there qualify.  It supports every Dk, Dv in
 * {32, 64, 128}: smaller heads run in the same 128-wide tiles, the channels
 * past the head read as zeros and are never written, so a chunk costs what it
 * costs at 128 and the results are those of the true sizes.
 */
GDN_API gdn_status gdn_prefill(const gdn_dims *dims, const uint16_t *q, const uint16_t *k,
                       const uint16_t *v, const float *g, const float *beta,
                       const float *state_in, float *state_out, const uint8_t *mask,
                       uint16_t *y, int chunk, void *workspace, size_t ws_bytes,
                       gdn_stream stream);

/* gdn_prefill with the layer's RMSNormGated applied to y before it is
 * stored.  (mlex gated_delta.rs, GatedDeltaNet::forward: the f32 rms_norm of
 * y over Dv with norm_eps, times the norm weight, times silu(z), cast to bf16.)
 * Per (b, t, hv):
 *   out = bf16( silu(z) * norm_w * yb / sqrt(mean_Dv(yb^2) + norm_eps) )
 * with yb the bf16 y that gdn_prefill would write (so a masked step, yb = 0,
 * gives a zero).  chunk = 64 runs the norm in the chunked kernel's epilogue
 * (y never goes to memory) when B * Hv is at least the GPU's SM count; with
 * fewer heads, and for chunk = 0 (whose kernel spreads a head's rows over
 * several CTAs), y is written to `out` and a second kernel normalises it in
 * place, which measured faster there.
 *   z          bf16 [B, T, Hv, Dv] (in): the in_proj_z output
 *   norm_w     f32  [Dv] (in);  norm_eps >= 0
 *   out        bf16 [B, T, Hv, Dv] (out)
 * Other arguments, the workspace and the limits as gdn_prefill. */
GDN_API gdn_status gdn_prefill_gated(const gdn_dims *dims, const uint16_t *q, const uint16_t *k,
                                     const uint16_t *v, const float *g, const float *beta,
                                     const float *state_in, float *state_out, const uint8_t *mask,
                                     const uint16_t *z, const float *norm_w, float norm_eps, uint16_t *out,
                                     int chunk, void *workspace, size_t ws_bytes, gdn_stream stream);

/* RMSNormGated output of the layer, applied to the recurrence output y.
 * (mlex gated_delta.rs, GatedDeltaNet::forward: rms_norm of y in f32 with
 * norm_eps, times the norm weight, times silu(z), cast to the activation dtype.)
 *   y, z       bf16 [B, T, Hv, Dv] (in); z is the in_proj_z output
 *   norm_w     f32  [Dv] (in)
 *   out        bf16 [B, T, Hv, Dv] (out), per (b, t, hv) row:
 *              out = bf16( silu(z) * w * y / sqrt(mean_Dv(y^2) + norm_eps) )
 * Only dims->B, T, Hv, Dv are used (the others must still be valid).  out may
 * alias y. */
GDN_API gdn_status gdn_rmsnorm_gated(const gdn_dims *dims, const uint16_t *y, const uint16_t *z,
                                     const float *norm_w, float norm_eps, uint16_t *out, gdn_stream stream);

/* The recurrence with vectorized gating: one decay factor per key channel,
 * S <- S diag(g_t) in place of S <- g_t S (the variant the qwen3-delta.ts
 * page of mlx-bun names beside the scalar one; the rest of the step as in
 * gdn_prefill).  Sequential form.
 *   g_vec      f32  [B, T, Hv, Dk] (in): the per-channel decay factors
 *   other arguments as gdn_prefill (q, k, v, beta, state_in, state_out, mask, y) */
GDN_API gdn_status gdn_prefill_vec(const gdn_dims *dims, const uint16_t *q, const uint16_t *k,
                                   const uint16_t *v, const float *g_vec, const float *beta,
                                   const float *state_in, float *state_out, const uint8_t *mask,
                                   uint16_t *y, gdn_stream stream);

/* gdn_prefill for callers that cannot allocate device memory.  Not an
 * operation of the method (the pages have no counterpart): a variant of the
 * call above for code that may not call cudaMalloc, such as a runtime that
 * hands out all device memory from its own pool, a loop that must never
 * synchronise the device, or a binding with no device allocator.  Same
 * arguments, results and errors as gdn_prefill, minus the workspace: the
 * row-order scratch lives in a fixed 32 KiB array inside the library, held on
 * every GPU that loads the library until the process exits.
 *   dims->B above GDN_NOALLOC_MAX_ROWS gives GDN_ERR_UNSUPPORTED.
 * The first call on each device looks up that array's device address
 * (cudaGetSymbolAddress, with that device current); make it before capturing
 * any stream.  The address is kept for the life of the process: a device
 * reset (cudaDeviceReset, or a reset of the primary context) between calls
 * leaves it stale and is not supported.  All calls share the array: calls that
 * overlap on the GPU (other streams, other host threads) race on it, so order
 * them.  Nothing in it needs clearing between calls.  No allocation is made by
 * this call.
 * Speed: the array holds only the row order, not the per-chunk images of the
 * two-pass chunked form, so with chunk = 64 this call always runs the single
 * pass.  Results are bit-identical to gdn_prefill's, but when B * Hv is below
 * the number of SMs the single pass keeps only B * Hv SMs busy: at B = 1,
 * Hv = 32, T = 8192 it takes about 3.1 times as long as gdn_prefill given
 * its full workspace (1.25 against 0.40 ms).  With B * Hv at or above the SM count both calls run
 * the same kernels. */
#define GDN_NOALLOC_MAX_ROWS 4096
GDN_API gdn_status gdn_prefill_noalloc(const gdn_dims *dims, const uint16_t *q, const uint16_t *k,
                                       const uint16_t *v, const float *g, const float *beta,
                                       const float *state_in, float *state_out, const uint8_t *mask,
                                       uint16_t *y, int chunk, gdn_stream stream);

/* Backward pass of the recurrence (training): the gradients of y and of the
 * final state with respect to q, k, v, g, beta and the initial state.  The
 * pages define the forward step only (mlex gated_delta.rs, the per-timestep
 * loop; mlx-bun qwen3-delta.ts, gated_delta_step); this is its exact
 * derivative.  A masked step has zero gradients for its inputs and passes the
 * state gradient through.  Sequential form, every step in f32.
 *   q, k, v, g, beta, state_in, mask  as gdn_prefill (the forward inputs)
 *   dy         bf16 [B, T, Hv, Dv] (in): gradient of y
 *   dstate_out f32  [B, Hv, Dv, Dk] (in) or NULL (= 0): gradient of the final state
 *   dq, dk     f32  [B, T, Hk, Dk] (out): summed over the Hv/Hk v-heads of each k-head
 *   dv         f32  [B, T, Hv, Dv] (out)
 *   dg, dbeta  f32  [B, T, Hv] (out)
 *   dstate_in  f32  [B, Hv, Dv, Dk] (out): gradient of the initial state (also
 *              when state_in is NULL); may equal dstate_out
 *   workspace  device scratch of gdn_prefill_backward_workspace_size() bytes,
 *              16-byte aligned (required when B * T > 0): a longest-first
 *              row order for masked batches, the forward state
 *              at the start of every 32-step chunk (16 KiB per 32 state rows
 *              and chunk at Dk = 128), for batches with fewer than two row
 *              slices of 32 rows per SM also its gradient at every chunk's
 *              end, and one 32-step history per CTA of the pass that
 *              reverses the chunks (one per row slice, or at most two per SM
 *              of the current device, so query the size on the device that
 *              runs it)
 * The outputs are summed with atomics, so for Hv/Hk > 2 or Dv > 32 their
 * last bits can differ between runs.  Supports Dk, Dv in {32, 64, 128}. */
GDN_API size_t gdn_prefill_backward_workspace_size(const gdn_dims *dims);
GDN_API gdn_status gdn_prefill_backward(const gdn_dims *dims, const uint16_t *q, const uint16_t *k,
                                        const uint16_t *v, const float *g, const float *beta,
                                        const float *state_in, const uint8_t *mask, const uint16_t *dy,
                                        const float *dstate_out, float *dq, float *dk, float *dv, float *dg,
                                        float *dbeta, float *dstate_in, void *workspace, size_t ws_bytes,
                                        gdn_stream stream);

/* The same gradients in chunked form on the tensor cores (Dk, Dv in {32, 64,
 * 128}, all on 128-wide tiles whose padding is exact zeros): the derivative of the chunked
 * forward's products (chunks of 64 steps, tf32 operands with f32
 * accumulation, like gdn_prefill with chunk = 64), with the gradient of the
 * state carried backwards from chunk to chunk.  The call runs the chunked
 * forward first, keeping every chunk's start state and D^T, then the chain
 * images and the reverse chain (one cooperative launch when B * Hv is at
 * most a quarter of the SM count, else two) and two gradient passes.
 * Arguments, outputs and mask semantics as gdn_prefill_backward; the
 * gradients agree with the sequential form within the tf32 rounding of the
 * products (about 3e-4 relative L2 against an f64 reference).
 *   workspace  device scratch of gdn_prefill_backward_chunked_workspace_size()
 *              bytes, 16-byte aligned (required when B * T > 0): the row
 *              order, then per chunk of each (b, hv) head
 *              161 KiB of chain images and 192 KiB of f32 records (start
 *              state, D^T, state gradient, dZ^T), and, when B * Hv is below
 *              the SM count, the two-pass forward's chunk images (sharing
 *              space with the chain images), and a ready flag per chunk.
 *              About 353 KiB per 64 steps of each head: 1.4 GB at B = 1,
 *              Hv = 32, T = 8192.
 * The outputs are summed with atomics (dq, dk over the Hv/Hk v-heads of each
 * k-head); dv, dg, dbeta and dstate_in are written once. */
GDN_API size_t gdn_prefill_backward_chunked_workspace_size(const gdn_dims *dims);
GDN_API gdn_status gdn_prefill_backward_chunked(const gdn_dims *dims, const uint16_t *q, const uint16_t *k,
                                                const uint16_t *v, const float *g, const float *beta,
                                                const float *state_in, const uint8_t *mask, const uint16_t *dy,
                                                const float *dstate_out, float *dq, float *dk, float *dv,
                                                float *dg, float *dbeta, float *dstate_in, void *workspace,
                                                size_t ws_bytes, gdn_stream stream);

/* Bytes of the optional gdn_prefill workspace for these sizes and this chunk
 * mode (0 or 64): about 8 bytes per batch row, rounded up to 256.  Returns 0
 * for invalid or unsupported arguments. */
GDN_API size_t gdn_prefill_workspace_size(const gdn_dims *dims, int chunk);

/* Human-readable name of a status code (static storage). */
GDN_API const char *gdn_status_string(gdn_status status);

/* Synchronises `stream`, then reads and clears the current device's error
 * word, which a kernel sets when one of its bounded waits (on an mbarrier or
 * a tensor-core commit) gives up.  Returns GDN_OK, GDN_ERR_TIMEOUT, or
 * GDN_ERR_CUDA if the synchronisation itself failed. */
GDN_API gdn_status gdn_device_status(gdn_stream stream);

/* Self-test of the failure path: launches a kernel whose bounded wait (on an
 * mbarrier nothing arrives on) runs out after a few thousand probes, and
 * checks that the error word reports it (GDN_ERR_TIMEOUT) and is cleared
 * again.  Returns GDN_OK when the timeout was reported, GDN_ERR_CUDA when it
 * was not (or the device failed).  No fault or unbounded wait is involved;
 * the context stays usable. */
GDN_API gdn_status gdn_selftest_timeout(gdn_stream stream);

/* ABI version of this header (incremented on any signature change). */
GDN_API int gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */

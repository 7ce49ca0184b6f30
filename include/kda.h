/*
 * kda.h -- C ABI of libkda, Kimi Delta Attention (KDA) on NVIDIA GB300 (sm_103a).
 *
 * KDA is the gated delta rule with a per-channel decay.  For one sequence and
 * one head the state S is a K x V fp32 matrix (K = d_k rows, V = d_v columns)
 * and each token t updates it and produces an output:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T (scale * q_t)
 *
 * with the gate g = -exp(A_log) * softplus(f + dt_bias) and beta = sigmoid(b).
 * The Kimi-K3 code audit (data/code-audit.json, finding
 * "dual-kda-execution-regimes") names the two regimes this library serves: a
 * chunked form for prefill and a fused recurrent form for one-token cached
 * decoding.  K3_ARTIFACT_AUDIT.md section 7.1 lists the interface facts of the
 * FlashKDA kernel library that this ABI also follows: K = V = 128, bf16 q/k/v,
 * fp32 A_log/dt_bias, fixed and variable length, initial and final recurrent
 * state.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a DEVICE pointer to row-major contiguous memory
 *   owned by the caller.  libkda allocates nothing except where an entry
 *   point says otherwise; scratch memory is passed in as `workspace`.
 * - Token tensors are laid out [N, H, D] (token, head, channel); states are
 *   [B, H, K, V] with the d_k row index first; beta is [N, H].
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Calls are asynchronous on it: the returned status covers host
 *   argument checks and launch errors only.
 * - Errors found on the device (an out-of-range cu_seqlens entry, a bounded
 *   wait that ran out) are recorded in a device error word and returned by
 *   kda_get_last_device_error().  No kernel traps or asserts.
 * - Pointers must be 16-byte aligned (KDA_ERR_MISALIGNED otherwise).
 * - No C++ exception crosses this ABI.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_VERSION 10200 /* 1.2.0 */

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum, bad cu_seqlens */
    KDA_ERR_UNSUPPORTED_SHAPE = 2,  /* e.g. K or V != 128 for prefill/decode */
    KDA_ERR_UNSUPPORTED_DTYPE = 3,
    KDA_ERR_MISALIGNED = 4,         /* a pointer is not 16-byte aligned */
    KDA_ERR_WORKSPACE_TOO_SMALL = 5,
    KDA_ERR_CUDA = 6,               /* a CUDA runtime call or launch failed */
    KDA_ERR_DEVICE_TIMEOUT = 7,     /* a bounded device-side wait ran out */
    KDA_ERR_NONFINITE = 8,          /* reserved for debug checks */
    KDA_ERR_NOT_IMPLEMENTED = 9,
    KDA_ERR_NO_DEVICE = 10,         /* no usable sm_103 device / driver */
    KDA_ERR_DECAY_RANGE = 11        /* kda_chunk_backward: a (sequence, head) whose chunk
                                       decay exceeds one chunk's range (device-side) */
} kda_status;

typedef enum kda_dtype {
    KDA_BF16 = 0,
    KDA_FP32 = 1
} kda_dtype;

/*
 * Shape of A_log.  K3_ARTIFACT_AUDIT.md section 5.2 records that the public
 * configuration, the HF code and FlashKDA's check expect A_log of shape [H]
 * while the checkpoint header holds [128]; all three readings are accepted.
 */
typedef enum kda_alog_mode {
    KDA_ALOG_PER_HEAD = 0,          /* A_log [H] */
    KDA_ALOG_PER_CHANNEL = 1,       /* A_log [K] */
    KDA_ALOG_PER_HEAD_CHANNEL = 2   /* A_log [H, K] */
} kda_alog_mode;

/*
 * kda_gate_fused -- the KDA gate in one pass (parameters: K3_ARTIFACT_AUDIT.md
 * section 4.1 tensor table and section 5.1 statistics; beta as an fp32 sigmoid
 * of the raw gate: finding 1 of the "[OMNIML-6079] [20/21] Add the Kimi-K3
 * expert-parallel adapter" review).
 *
 *   g[n,h,c]  = -(exp(A_log[.]) * softplus(f[n,h,c] + dt_bias[h,c]))
 *   beta[n,h] = 1 / (1 + exp(-b[n,h]))
 *
 * with softplus(x) = max(x, 0) + log1p(exp(-|x|)).  The result is bit-exact
 * with respect to a fixed binary32 specification (libkda's own exp and log1p,
 * every operation rounded to nearest, no contraction).
 *
 *   f        [N, H, K] of f_dtype (bf16 or fp32)
 *   b        [N, H] of b_dtype (bf16 or fp32) beta logits; may be NULL, in
 *            which case beta_out must be NULL and no beta is written
 *   A_log    fp32, shape selected by alog_mode
 *   dt_bias  fp32 [H, K]
 *   g_out    fp32 [N, H, K] (written)
 *   beta_out fp32 [N, H] (written) or NULL
 *
 * Shape-generic in K.  N == 0 is a no-op.
 */
kda_status kda_gate_fused(const void *f, kda_dtype f_dtype,
                          const void *b, kda_dtype b_dtype,
                          const float *A_log, kda_alog_mode alog_mode,
                          const float *dt_bias,
                          float *g_out, float *beta_out,
                          int64_t N, int H, int K, void *stream);

/*
 * Bytes of device workspace kda_chunk_prefill needs for these sizes.
 * The value never exceeds a few kilobytes; it is 0 only when nothing runs.
 */
size_t kda_chunk_prefill_workspace_size(int64_t N, int B, int H, int K, int V);

/*
 * kda_chunk_prefill -- the chunked KDA regime for prefill (code-audit.json,
 * finding "dual-kda-execution-regimes"; varlen and initial/final state as in
 * K3_ARTIFACT_AUDIT.md section 7.1).  Computes o and the final state exactly
 * as the token recurrence above would, chunk by chunk.
 *
 *   q, k, v       bf16 [N, H, 128]; q and k are used as given (no normalisation)
 *   g             fp32 [N, H, 128] log-decay, g <= 0.  A positive or NaN entry
 *                 sets INVALID_ARG in the device error word (that sequence's
 *                 results are then unspecified).  Chunks whose decay in some
 *                 channel exceeds what one chunk represents (160) are split on
 *                 the device, and a token whose own g is below -160 is taken
 *                 as -160 (e^-160 underflows fp32 as any stronger decay does),
 *                 so every decay is computed.
 *   beta          fp32 [N, H], already passed through the sigmoid
 *   cu_seqlens    int32 [B+1] device offsets of B packed sequences
 *                 (cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] = N); NULL
 *                 means one sequence of N tokens (B must be 1).  Entries that
 *                 break these rules are caught on the device: the sequence is
 *                 skipped and the device error word is set to INVALID_ARG.
 *                 Zero-length sequences are allowed (final = initial).
 *   scale         multiplies q
 *   initial_state fp32 [B, H, 128, 128] or NULL (zero state)
 *   final_state   fp32 [B, H, 128, 128] (written) or NULL; may alias
 *                 initial_state (each state is read before it is written)
 *   o             [N, H, 128] of o_dtype (bf16 or fp32), written
 *   workspace     device scratch of at least
 *                 kda_chunk_prefill_workspace_size(N, B, H, 128, 128) bytes,
 *                 16-byte aligned; its contents need not be initialised and
 *                 it must not be used by another call running concurrently.
 *
 * K and V must be 128 (KDA_ERR_UNSUPPORTED_SHAPE otherwise).
 */
kda_status kda_chunk_prefill(const void *q, const void *k, const void *v,
                             const float *g, const float *beta,
                             const int32_t *cu_seqlens, int B,
                             int64_t N, int H, int K, int V, float scale,
                             const float *initial_state, float *final_state,
                             void *o, kda_dtype o_dtype,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_chunk_prefill_gated -- kda_chunk_prefill with the gate computed inside
 * the chunked kernel, the interface K3_ARTIFACT_AUDIT.md section 7.1 records for
 * FlashKDA (gate pre-activation in bf16, A_log/dt_bias in fp32, beta logits):
 *
 *   g[n,h,c]  = -exp(A_log[.]) * softplus(f[n,h,c] + dt_bias[h,c])
 *   beta[n,h] = sigmoid(b[n,h])
 *
 * evaluated with the special-function unit (relative error ~1e-6; it is not
 * the bit-exact specification of kda_gate_fused).  The fp32 g and beta never
 * reach global memory.
 *
 *   f        bf16 [N, H, 128] gate pre-activation (f_dtype must be KDA_BF16)
 *   b        [N, H] beta logits, bf16 or fp32 (b_dtype); the sigmoid is applied
 *            here, once (the EP-adapter review's finding 1: never pass raw
 *            logits where post-sigmoid beta is expected, or vice versa)
 *   A_log    fp32, shape by alog_mode;  dt_bias fp32 [H, 128]
 * All other arguments, layouts and results are those of kda_chunk_prefill
 * (same workspace size).
 */
kda_status kda_chunk_prefill_gated(const void *q, const void *k, const void *v,
                                   const void *f, kda_dtype f_dtype,
                                   const void *b, kda_dtype b_dtype,
                                   const float *A_log, kda_alog_mode alog_mode,
                                   const float *dt_bias,
                                   const int32_t *cu_seqlens, int B,
                                   int64_t N, int H, int K, int V, float scale,
                                   const float *initial_state, float *final_state,
                                   void *o, kda_dtype o_dtype,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_chunk_prefill_noalloc -- kda_chunk_prefill without a workspace argument,
 * for callers that cannot allocate device memory: a host plugin interface that
 * hands the library only its input and output buffers and offers no way to ask
 * for scratch, or a serving process that reserved all device memory at start-up
 * and must not call cudaMalloc afterwards (it can fail, and it can synchronise
 * the device).  The pages this library follows have no counterpart to it.
 *
 * Arguments, layouts and results are those of kda_chunk_prefill.  The scratch
 * comes from a device array built into the library (4096 bytes; every GPU that
 * loads the library holds it until the process exits).  Sizes whose
 * kda_chunk_prefill_workspace_size() exceeds it are rejected with
 * KDA_ERR_WORKSPACE_TOO_SMALL.  The call allocates nothing: it never calls
 * cudaMalloc, cudaFree or any allocating library routine.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current, so make that first call before any stream capture.  All
 * calls on a device share the array: calls whose kernels overlap on the GPU
 * (on different streams) race on it; calls in stream order do not.
 */
kda_status kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v,
                                     const float *g, const float *beta,
                                     const int32_t *cu_seqlens, int B,
                                     int64_t N, int H, int K, int V, float scale,
                                     const float *initial_state, float *final_state,
                                     void *o, kda_dtype o_dtype, void *stream);

/*
 * kda_recurrent_decode -- the fused recurrent KDA regime for one-token cached
 * decoding (code-audit.json, finding "dual-kda-execution-regimes"): one new
 * token for each of B sequences, the state updated in place.
 *
 *   q, k, v   bf16 [B, H, 128]
 *   g         fp32 [B, H, 128];  beta fp32 [B, H] (post-sigmoid)
 *   state     fp32 [B, H, 128, 128], read and overwritten with S_t
 *   o         [B, H, 128] of o_dtype, written
 *
 * K and V must be 128.  B == 0 is a no-op.
 */
kda_status kda_recurrent_decode(const void *q, const void *k, const void *v,
                                const float *g, const float *beta,
                                float *state, int B, int H, int K, int V, float scale,
                                void *o, kda_dtype o_dtype, void *stream);

/*
 * kda_recurrent_decode_indexed -- kda_recurrent_decode over a pool of cached
 * states addressed by slot, with fp32 or bf16 state storage: the decode side
 * of continuous batching, where sequences come and go and their states live in
 * preallocated slots that are updated in place (indexed writes rather than
 * concatenation: the Kimi-K3 code audit's "repeated-mla-cache-concatenation"
 * recommendation; FlashKDA's bf16 / fp32 state modes, K3_ARTIFACT_AUDIT.md
 * section 7.4).
 *
 *   q, k, v        bf16 [B, H, 128];  g fp32 [B, H, 128];  beta fp32 [B, H]
 *   state_pool     [num_slots, H, 128, 128] of state_dtype (fp32 or bf16),
 *                  read and written in place; a bf16 state is computed in fp32
 *                  and rounded to nearest on the way back
 *   state_indices  int32 [B] device: the slot of each sequence.  A negative
 *                  index marks an inactive sequence (its state is untouched and
 *                  its output row is zero); an index >= num_slots is skipped the
 *                  same way and sets the device error word to INVALID_ARG.  Two
 *                  sequences must not share a slot.
 *   o              [B, H, 128] of o_dtype
 */
kda_status kda_recurrent_decode_indexed(const void *q, const void *k, const void *v,
                                        const float *g, const float *beta,
                                        void *state_pool, kda_dtype state_dtype,
                                        const int32_t *state_indices, int num_slots,
                                        int B, int H, int K, int V, float scale,
                                        void *o, kda_dtype o_dtype, void *stream);

/*
 * kda_recurrent_decode_gated -- the fused recurrent decode with the gate
 * computed in the same kernel, from the gate's own inputs (the interface
 * K3_ARTIFACT_AUDIT.md section 7.1 records for FlashKDA's prefill, applied to
 * the one-token regime of code-audit.json, finding "dual-kda-execution-
 * regimes").  g and beta are formed with exactly the binary32 operations of
 * kda_gate_fused, so the result equals kda_gate_fused followed by
 * kda_recurrent_decode_indexed bit for bit, with one launch and no fp32 g
 * buffer.  (Measured at B = 256, H = 96 on GB300 it is about 3 % slower than
 * the two launches: the exact gate arithmetic adds latency to every CTA of the
 * HBM-bound step.)
 *
 *   q, k, v        bf16 [B, H, 128]
 *   f              [B, H, 128] gate pre-activation, bf16 or fp32 (f_dtype)
 *   b              [B, H] beta logits, bf16 or fp32 (b_dtype); the sigmoid is
 *                  applied here, once
 *   A_log          fp32, shape by alog_mode;  dt_bias fp32 [H, 128]
 *   state_pool, state_dtype, state_indices, num_slots
 *                  as in kda_recurrent_decode_indexed; state_indices may be
 *                  NULL, meaning slot b for sequence b (then num_slots >= B)
 *   o              [B, H, 128] of o_dtype
 */
kda_status kda_recurrent_decode_gated(const void *q, const void *k, const void *v,
                                      const void *f, kda_dtype f_dtype,
                                      const void *b, kda_dtype b_dtype,
                                      const float *A_log, kda_alog_mode alog_mode,
                                      const float *dt_bias,
                                      void *state_pool, kda_dtype state_dtype,
                                      const int32_t *state_indices, int num_slots,
                                      int B, int H, int K, int V, float scale,
                                      void *o, kda_dtype o_dtype, void *stream);

/*
 * kda_recurrent_backward -- gradients of the KDA recurrence for training
 * ("chunked KDA for training", code-audit.json, finding
 * "dual-kda-execution-regimes"): given dL/do and dL/dS_final for the forward
 * pass that kda_chunk_prefill computes on the same inputs, the gradients with
 * respect to q, k, v, g, beta and the initial state.  With
 * S' = Diag(exp g_t) S_{t-1}, w = S'^T k_t, u = beta_t (v_t - w),
 * S_t = S' + k_t u^T, o_t = S_t^T (scale q_t), each reverse step from
 * G = dL/dS_t is
 *   G += (scale q_t) do_t^T;  du = G^T k_t;  dv_t = beta_t du;
 *   dbeta_t = du . (v_t - w);  dw = -beta_t du;  dk_t = G u + S' dw;
 *   dq_t = scale S_t do_t;  dg_t = rowsum((G + k_t dw^T) (.) S');
 *   G = Diag(exp g_t) (G + k_t dw^T)
 * (dL/dS_0 = G at the end).  Computed token by token in fp32 on CUDA cores:
 * a forward pass keeps the state every 16 tokens in the workspace, and each
 * 16-token segment is rerun from it in reverse order.
 *
 *   q, k, v        bf16 [N, H, 128];  g fp32 [N, H, 128];  beta fp32 [N, H]
 *   cu_seqlens, B, initial_state, scale   as in kda_chunk_prefill
 *   dO             [N, H, 128] of dO_dtype (bf16 or fp32)
 *   dS_final       fp32 [B, H, 128, 128] or NULL (zero)
 *   dq, dk, dv, dg fp32 [N, H, 128];  dbeta fp32 [N, H]   (all written)
 *   dS0            fp32 [B, H, 128, 128] or NULL (not computed)
 *   workspace      device, >= kda_recurrent_backward_workspace_size() bytes
 *                  (states every 16 tokens plus 1 MB per CTA; 1.7 GB for
 *                  N = 4096, H = 96); its contents are scratch
 *
 * The gate's own gradients (to f, A_log, dt_bias and the beta logits) are
 * the caller's: g and beta enter here as given tensors.  A bad cu_seqlens
 * entry sets the device error word to INVALID_ARG.
 */
size_t kda_recurrent_backward_workspace_size(int64_t N, int B, int H, int K, int V);

kda_status kda_recurrent_backward(const void *q, const void *k, const void *v,
                                  const float *g, const float *beta,
                                  const int32_t *cu_seqlens, int B,
                                  int64_t N, int H, int K, int V, float scale,
                                  const float *initial_state,
                                  const void *dO, kda_dtype dO_dtype, const float *dS_final,
                                  float *dq, float *dk, float *dv, float *dg, float *dbeta,
                                  float *dS0, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * kda_chunk_backward -- the same gradients as kda_recurrent_backward (same
 * arguments, layouts and results), in the chunked form the pages name for
 * training ("chunked KDA for training", code-audit.json, finding
 * "dual-kda-execution-regimes"), on the tensor cores.  A forward pass of the
 * chunked prefill keeps the state at the start of every 64-token chunk in the
 * workspace; then each (sequence, head) walks its chunks last to first, with
 * the state gradient in tensor memory, and per chunk forms the reverse mode
 * of the chunk-level (WY/UT) forward: dU = A_qk^T dO + Khat dS',
 * dS = Diag(e^{Gam_L}) dS' + Qbar^T dO - W^T dU, and the gradients of
 * A_qk, A_kk (through T = (I + A_kk)^-1), W, U-tilde and the decay factors,
 * down to dq, dk, dv, dg, dbeta.  Every product runs as tcgen05 bf16 MMAs on
 * operands split in a high and a low bf16 part (three products per pair,
 * a 16-bit significand) with fp32 accumulation; the chunk-start states come
 * from the tf32 forward, so the gradients agree with the exact reverse mode
 * to about 1e-3 relative L2 (the forward's state precision), not to fp32
 * rounding as kda_recurrent_backward does.  Every sum is added in a fixed
 * order, so two calls on the same inputs write the same bits.
 *
 * A (sequence, head) whose forward pass had to shorten a chunk (a chunk's
 * decay -sum(g) in some channel above 160) has no 64-token-aligned states:
 * its gradients are written as zeros and the device error word is set to
 * KDA_ERR_DECAY_RANGE; kda_recurrent_backward computes those.
 *
 *   workspace  device, >= kda_chunk_backward_workspace_size() bytes, 16-byte
 *              aligned: the chunk-start states ((N / 64 + B) H 64 KB, 400 MB
 *              for N = 4096, H = 96) plus 528 KB of operand scratch for each
 *              of up to min(B H, 160) CTAs; its contents are scratch.
 * The bounded waits use the product limit of kda_debug_set_wait_limit.
 */
size_t kda_chunk_backward_workspace_size(int64_t N, int B, int H, int K, int V);

kda_status kda_chunk_backward(const void *q, const void *k, const void *v,
                              const float *g, const float *beta,
                              const int32_t *cu_seqlens, int B,
                              int64_t N, int H, int K, int V, float scale,
                              const float *initial_state,
                              const void *dO, kda_dtype dO_dtype, const float *dS_final,
                              float *dq, float *dk, float *dv, float *dg, float *dbeta,
                              float *dS0, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * kda_chunk_prefill_checkpointed / kda_chunk_backward_checkpointed -- the
 * training pair of the chunked form: the forward pass that a training step
 * runs anyway also keeps the chunk-start states, and the backward reads them
 * instead of running the forward a second time (kda_chunk_backward does both
 * in one call, about 0.5 ms of its time for N = 4096, H = 96).
 *
 * kda_chunk_prefill_checkpointed takes the arguments of kda_chunk_prefill and
 * writes the same o and final_state (the same kernel, bit for bit), and in
 * addition:
 *   checkpoints  device, >= kda_chunk_checkpoints_size() bytes, 16-byte
 *                aligned, written (caller-owned; nothing else is kept): first
 *                one int32 per (sequence, head), b H + h, set to 1 where a
 *                chunk had to be shortened (decay -sum(g) in some channel
 *                above 160 within 64 tokens), padded to 256 bytes; then the
 *                fp32 state S [K, V] at the start of every 64-token chunk,
 *                chunk c of sequence b (c = 0, 1, ..) in slot
 *                cu_seqlens[b] / 64 + b + c, [slot, H, K, V] row-major
 *                ((N / 64 + B) H 64 KB: 400 MB for N = 4096, H = 96).
 *   workspace    >= kda_chunk_prefill_workspace_size() bytes, as for
 *                kda_chunk_prefill.
 *
 * kda_chunk_backward_checkpointed takes the arguments of kda_chunk_backward
 * with the checkpoints of a kda_chunk_prefill_checkpointed call on the same
 * q, k, v, g, beta, cu_seqlens, scale and initial state in place of
 * initial_state, and writes the same gradients, bit for bit, with the same
 * KDA_ERR_DECAY_RANGE rule for a marked (sequence, head).  It only reads the
 * checkpoints (they may serve several backward calls).
 *   workspace    device, >= kda_chunk_backward_checkpointed_workspace_size()
 *                bytes (512 bytes plus 528 KB for each of up to
 *                min(B H, 160) CTAs), 16-byte aligned; scratch.
 * Both return KDA_ERR_WORKSPACE_TOO_SMALL when checkpoints_bytes is below the
 * size above, and otherwise fail as the calls they extend.  The sizes return
 * 0 for arguments those calls reject.
 */
size_t kda_chunk_checkpoints_size(int64_t N, int B, int H, int K, int V);

kda_status kda_chunk_prefill_checkpointed(const void *q, const void *k, const void *v,
                                          const float *g, const float *beta,
                                          const int32_t *cu_seqlens, int B,
                                          int64_t N, int H, int K, int V, float scale,
                                          const float *initial_state, float *final_state,
                                          void *o, kda_dtype o_dtype,
                                          void *checkpoints, size_t checkpoints_bytes,
                                          void *workspace, size_t workspace_bytes,
                                          void *stream);

size_t kda_chunk_backward_checkpointed_workspace_size(int64_t N, int B, int H, int K, int V);

kda_status kda_chunk_backward_checkpointed(const void *q, const void *k, const void *v,
                                           const float *g, const float *beta,
                                           const int32_t *cu_seqlens, int B,
                                           int64_t N, int H, int K, int V, float scale,
                                           const void *checkpoints, size_t checkpoints_bytes,
                                           const void *dO, kda_dtype dO_dtype,
                                           const float *dS_final,
                                           float *dq, float *dk, float *dv, float *dg,
                                           float *dbeta, float *dS0,
                                           void *workspace, size_t workspace_bytes,
                                           void *stream);

/*
 * kda_gate_backward -- gradients of the gate (the training regime, after
 * kda_recurrent_backward): from dL/dg and dL/dbeta to the gate's inputs.
 * With x = f + dt_bias, a = exp(A_log), g = -a softplus(x), beta = sigmoid(b)
 * (K3_ARTIFACT_AUDIT.md sections 4.1 and 5.1):
 *   df = dg (-a sigmoid(x));   d dt_bias = sum over tokens of df;
 *   d A_log = sum of dg g over the axes A_log is broadcast along;
 *   db = dbeta beta (1 - beta)
 * x, a, g and beta are formed with kda_gate_fused's binary32 specification.
 * The sums are added in a fixed order (the result does not depend on timing).
 *
 *   f            [N, H, K] of f_dtype (bf16 or fp32);  dg fp32 [N, H, K]
 *   b, dbeta     [N, H] (b_dtype) and fp32 [N, H], with db fp32 [N, H]
 *                written; all three NULL to skip beta
 *   A_log        fp32 by alog_mode;  dt_bias fp32 [H, K]
 *   df           fp32 [N, H, K] written
 *   dA_log       fp32, shape of A_log, written (or NULL)
 *   ddt_bias     fp32 [H, K] written (or NULL)
 *   workspace    >= kda_gate_backward_workspace_size(N, H, K) bytes (about
 *                (2 min(N, 256) + 1) H K 4 bytes), 16-byte aligned
 * K must be a multiple of 8; f, dg, df 16-byte aligned.
 */
size_t kda_gate_backward_workspace_size(int64_t N, int H, int K);

kda_status kda_gate_backward(const void *f, kda_dtype f_dtype,
                             const void *b, kda_dtype b_dtype,
                             const float *A_log, kda_alog_mode alog_mode,
                             const float *dt_bias,
                             const float *dg, const float *dbeta,
                             float *df, float *db, float *dA_log, float *ddt_bias,
                             int64_t N, int H, int K,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_short_conv_qkv -- the KDA input pre-step over a packed batch, on the three
 * projection streams at once: a depthwise causal convolution of kernel size 4
 * per channel (the checkpoint's q/k/v_conv1d.weight, fp32 [H*128, 1, 4];
 * K3_ARTIFACT_AUDIT.md section 4.1, KDA tensor table), then SiLU, then for q
 * and k an L2 norm over each head's 128 channels:
 *
 *   a[p, c] = sum_{j=0..3} w[c, j] x[p - 3 + j, c]     (tap 3 on the current token)
 *   y = a * sigmoid(a);   q, k: y / sqrt(sum_head y^2 + 1e-6);   v: y
 *
 * Positions before a sequence's first token read that sequence's carried
 * state (the last three raw inputs of its previous segment, oldest first), or
 * zeros when conv_state_in is NULL.  Sequences never see each other.
 *
 *   x_q, x_k, x_v     bf16 [N, C] each, C = H * 128 (the projection outputs)
 *   w_q, w_k, w_v     fp32 [C, 4] each
 *   cu_seqlens, B     as in kda_chunk_prefill (NULL: one sequence, B = 1)
 *   conv_state_in     bf16 [B, 3 (q, k, v), 3 (oldest first), C] or NULL
 *   conv_state_out    bf16 [B, 3, 3, C] or NULL: each sequence's last three
 *                     inputs (state rows fill in for sequences shorter than 3;
 *                     an empty sequence passes its state through).  Must not
 *                     overlap conv_state_in.
 *   q, k, v           bf16 [N, C] outputs, ready for kda_chunk_prefill as
 *                     [N, H, 128]; must not overlap any input
 *
 * C must be a positive multiple of 128 (KDA_ERR_UNSUPPORTED_SHAPE).  A bad
 * cu_seqlens array sets the device error word to INVALID_ARG.  N == 0 with
 * conv_state_out copies the states through.
 */
kda_status kda_short_conv_qkv(const void *x_q, const void *x_k, const void *x_v,
                              const float *w_q, const float *w_k, const float *w_v,
                              const int32_t *cu_seqlens, int B, int64_t N, int C,
                              const void *conv_state_in, void *conv_state_out,
                              void *q, void *k, void *v, void *stream);

/*
 * kda_short_conv_qkv_step -- the same pre-step for one new token per sequence,
 * the carried conv states kept in a pool addressed by slot and updated in
 * place (the decode side of kda_short_conv_qkv).
 *
 *   x_q, x_k, x_v     bf16 [B, C];  w_q, w_k, w_v fp32 [C, 4]
 *   conv_state_pool   bf16 [num_slots, 3, 3, C], read and shifted in place
 *   state_indices     int32 [B] device, or NULL for slot b = sequence b
 *                     (then num_slots >= B).  Negative: inactive sequence
 *                     (outputs zero, state untouched); >= num_slots: skipped
 *                     the same way and the device error word set to
 *                     INVALID_ARG.  Two sequences must not share a slot.
 *   q, k, v           bf16 [B, C] outputs (may be the inputs themselves)
 *
 * C must be a positive multiple of 128; B <= 65535.
 */
kda_status kda_short_conv_qkv_step(const void *x_q, const void *x_k, const void *x_v,
                                   const float *w_q, const float *w_k, const float *w_v,
                                   void *conv_state_pool, const int32_t *state_indices,
                                   int num_slots, int B, int C,
                                   void *q, void *k, void *v, void *stream);

/*
 * kda_debug_check_gate_division -- test hook: the gate kernel's common path
 * (|f + dt_bias| < 87) divides with an fma-based correctly rounded division
 * (Markstein's method) instead of IEEE division; this call runs it against
 * IEEE division on the device for every operand pair that path can form
 * (about 1.07e9) and writes the number of differing results to *mismatches
 * (host pointer; 0 is the gate's bit-exactness).  Synchronises `stream`.
 */
kda_status kda_debug_check_gate_division(uint64_t *mismatches, void *stream);

/*
 * kda_debug_set_wait_limit -- test hook for the bounded device waits.  Every
 * wait of the chunked prefill kernels on a copy (TMA) or a tensor-core product
 * gives up after a bounded number of polls and records KDA_ERR_DEVICE_TIMEOUT
 * in the device error word instead of hanging (a failure is reported, never
 * turned into silent wrong numbers: the EP-adapter review, finding IMPORTANT
 * 1, asks for loud failure).  This call sets the bound of the main-loop waits
 * of later kda_chunk_prefill* launches in this process: copy_polls for copies,
 * product_polls for products; 0 gives up at the first poll, a negative value
 * restores the default.  A kernel that gives up stops issuing work and, before
 * it exits, waits for everything it had in flight with the default bound (this
 * drain is never shortened).  For tests only: the outputs of an aborted launch
 * are incomplete.  Always returns KDA_OK.
 */
kda_status kda_debug_set_wait_limit(int64_t copy_polls, int64_t product_polls);

/*
 * Synchronises `stream`, then returns and clears the device error word of the
 * current device (KDA_OK when no kernel recorded an error).  Returns
 * KDA_ERR_CUDA if the synchronisation itself fails.
 */
kda_status kda_get_last_device_error(void *stream);

/* A static, human-readable name for a status code. */
const char *kda_status_string(kda_status status);

/* KDA_VERSION of the built library. */
int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */

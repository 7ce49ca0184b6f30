// kda_internal.cuh -- declarations shared by libkda's CUDA translation units.
// Not part of the public ABI (include/kda.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Device error codes written to the device error word (first error wins).
// Values match kda_status so the host can return them directly.
enum : unsigned int {
    kDevOk = 0,
    kDevInvalidArg = 1,      // KDA_ERR_INVALID_ARG: a bad cu_seqlens entry
    kDevTimeout = 7,         // KDA_ERR_DEVICE_TIMEOUT: a bounded wait ran out
    kDevDecayRange = 11,     // KDA_ERR_DECAY_RANGE: chunked backward, a chain it cannot take
};

__device__ __forceinline__ void record_device_error(unsigned int *err, unsigned int code) {
    if (err != nullptr) atomicCAS(err, 0u, code);
}

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Raises `func`'s dynamic shared-memory limit to `bytes` on the current device.
// The attribute belongs to the device, so a process that drives several GPUs
// needs it on each: the call is made once per (device, kernel) under a lock
// (kda_api.cu) and later calls return at once.
cudaError_t ensure_dynamic_smem(const void *func, int bytes);

// Launchers (defined next to their kernels).  All are asynchronous on `s`.
cudaError_t launch_gate(const void *f, bool f_bf16, const void *b, bool b_bf16,
                        const float *A_log, int alog_mode, const float *dt_bias, float *g,
                        float *beta, int64_t N, int H, int K, int num_sms, cudaStream_t s);

// Test hook: the gate's fast division against IEEE division over every operand
// pair its common path forms; the count of differing results to *mismatches
// (host), the stream synchronised.
cudaError_t check_gate_division(unsigned long long *mismatches, int num_sms, cudaStream_t s);

cudaError_t launch_decode(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                          const __nv_bfloat16 *v, const float *g, const float *beta,
                          float *state, int B, int H, float scale, void *o, bool o_bf16,
                          cudaStream_t s);

cudaError_t launch_decode_indexed(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                  const __nv_bfloat16 *v, const float *g, const float *beta,
                                  void *state_pool, bool state_bf16, const int32_t *slots,
                                  int num_slots, int B, int H, float scale, void *o, bool o_bf16,
                                  unsigned int *err, cudaStream_t s);

cudaError_t launch_short_conv(const __nv_bfloat16 *const x[3], const float *const w[3],
                              __nv_bfloat16 *const y[3], const int32_t *cu_seqlens, int B,
                              int64_t N, int C, const __nv_bfloat16 *state_in,
                              __nv_bfloat16 *state_out, unsigned int *err, cudaStream_t s);

cudaError_t launch_short_conv_step(const __nv_bfloat16 *const x[3], const float *const w[3],
                                   __nv_bfloat16 *const y[3], __nv_bfloat16 *pool,
                                   const int32_t *slots, int num_slots, int B, int C,
                                   unsigned int *err, cudaStream_t s);

// Backward (kda_backward.cu): workspace for `ctas` CTAs, and the launch.
constexpr int kBackwardMaxCtas = 256;
size_t backward_workspace_bytes(int64_t N, int B, int H, int ctas);
int backward_ctas(int B, int H, int max_ctas);

cudaError_t launch_backward(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                            const __nv_bfloat16 *v, const float *g, const float *beta,
                            const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
                            const float *S0, const void *dO, bool dO_bf16, const float *dSf,
                            float *dq, float *dk, float *dv, float *dg, float *dbeta, float *dS0,
                            void *workspace, int ctas, unsigned int *err, cudaStream_t s);

cudaError_t launch_decode_gated(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                const __nv_bfloat16 *v, const void *f, bool f_bf16, const void *b,
                                bool b_bf16, const float *A_log, int alog_mode,
                                const float *dt_bias, void *state_pool, bool state_bf16,
                                const int32_t *slots, int num_slots, int B, int H, float scale,
                                void *o, bool o_bf16, unsigned int *err, cudaStream_t s);

// Gate backward (kda_gate_bwd.cu).
size_t gate_bwd_workspace_bytes(int64_t N, int H, int K);
cudaError_t launch_gate_backward(const void *f, bool f_bf16, const void *b, bool b_bf16,
                                 const float *A_log, int alog_mode, const float *dt_bias,
                                 const float *dg, const float *dbeta, float *df, float *db,
                                 float *dA_log, float *ddt_bias, int64_t N, int H, int K,
                                 void *workspace, cudaStream_t s);

// Prefill workspace layout is private to kda_chunk.cu.
size_t prefill_workspace_bytes(int64_t N, int B, int H);

cudaError_t launch_prefill(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, const float *g, const float *beta,
                           const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
                           const float *initial_state, float *final_state, void *o, bool o_bf16,
                           void *workspace, unsigned int *err, int num_sms, cudaStream_t s);

cudaError_t launch_prefill_gated(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                 const __nv_bfloat16 *v, const __nv_bfloat16 *f, const void *b,
                                 bool b_bf16, const float *A_log, int alog_mode,
                                 const float *dt_bias, const int32_t *cu_seqlens, int B, int64_t N,
                                 int H, float scale, const float *initial_state,
                                 float *final_state, void *o, bool o_bf16, void *workspace,
                                 unsigned int *err, int num_sms, cudaStream_t s);

// Bounds of the chunked prefill's main-loop waits for later launches (copies,
// products; a negative value restores the default).  Test use only.
void set_prefill_wait_polls(int64_t copy_polls, int64_t product_polls);

// Bound of the product waits set by set_prefill_wait_polls (the chunked
// backward uses it for all its waits).
uint32_t prefill_wait_polls();

// The chunked prefill as the forward pass of the chunked backward: no output,
// no final state; the state at the start of every 64-token chunk of chain
// (b, h) goes to ckpt[((cu[b] / 64 + b + c) * H + h) * 128 * 128 ..], and
// split[b * H + h] is set if a chunk had to be shortened.  counter: one zeroed
// unsigned int.
cudaError_t launch_prefill_checkpoints(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                       const __nv_bfloat16 *v, const float *g, const float *beta,
                                       const int32_t *cu_seqlens, int B, int64_t N, int H,
                                       float scale, const float *initial_state, float *ckpt,
                                       int *split, unsigned int *counter, unsigned int *err,
                                       int num_sms, cudaStream_t s);

// The chunked prefill that also stores, for a later backward pass, the state
// at every chunk start to ckpt and marks chains with a shortened chunk in split
// (both laid out as for launch_prefill_checkpoints; split is zeroed here).
cudaError_t launch_prefill_checkpointed(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                        const __nv_bfloat16 *v, const float *g, const float *beta,
                                        const int32_t *cu_seqlens, int B, int64_t N, int H,
                                        float scale, const float *initial_state, float *final_state,
                                        void *o, bool o_bf16, float *ckpt, int *split,
                                        void *workspace, unsigned int *err, int num_sms,
                                        cudaStream_t s);

// Chunked backward (kda_chunk_bwd.cu).
constexpr int kChunkBwdMaxCtas = 160;
size_t chunk_bwd_workspace_bytes(int64_t N, int B, int H, int ctas);
// Checkpoint buffer (split flags, then the chunk-start states) and the
// workspace of the backward that reads one.
size_t chunk_checkpoints_bytes(int64_t N, int B, int H);
size_t chunk_checkpoint_flags_bytes(int B, int H);  // the flags' part, at its start
size_t chunk_bwd_from_checkpoints_workspace_bytes(int ctas);
cudaError_t launch_chunk_backward_from_checkpoints(
    const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *g,
    const float *beta, const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
    const void *checkpoints, const void *dO, bool dO_bf16, const float *dSf, float *dq, float *dk,
    float *dv, float *dg, float *dbeta, float *dS0, void *workspace, int ctas, unsigned int *err,
    cudaStream_t s);
cudaError_t launch_chunk_backward(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                  const __nv_bfloat16 *v, const float *g, const float *beta,
                                  const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
                                  const float *S0, const void *dO, bool dO_bf16, const float *dSf,
                                  float *dq, float *dk, float *dv, float *dg, float *dbeta,
                                  float *dS0, void *workspace, int ctas, unsigned int *err,
                                  int num_sms, cudaStream_t s);

// Device address and size of the built-in prefill scratch on the current device
// (looked up once per device; see kda_chunk.cu).
cudaError_t builtin_prefill_scratch(void **ptr, size_t *bytes);

}  // namespace kda

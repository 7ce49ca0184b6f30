// kda_prefill.cu -- KDA prefill over packed variable-length sequences.
//
// Computes, for every (sequence, head), o_t = S_t^T (scale q_t) with
//   S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
// starting from the initial state (or zero) and writing the final state
// (code-audit.json, finding "dual-kda-execution-regimes"; varlen and
// initial/final state as in K3_ARTIFACT_AUDIT.md section 7.1).
//
// This version walks the tokens in order on CUDA cores: grid (4 d_v slices,
// H, B), the 128 x 32 fp32 state slice held in registers (warp w owns rows
// w + 8i, lane l owns column l of the slice).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kD = 128;
constexpr int kSlice = 32;
constexpr int kThreads = 256;
constexpr int kRows = kD / (kThreads / 32);  // 16 rows per thread

template <bool kOutBf16>
__global__ void __launch_bounds__(kThreads) prefill_recurrent_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const float *__restrict__ g,
    const float *__restrict__ beta, const int32_t *__restrict__ cu_seqlens, int64_t N, int H,
    float scale, const float *__restrict__ S0, float *__restrict__ Sf, void *__restrict__ o,
    unsigned int *err) {
    __shared__ float s_k[kD], s_q[kD], s_d[kD], s_v[kSlice], s_u[kSlice];
    __shared__ float s_red[2][kThreads / 32][kSlice];
    __shared__ float s_beta;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col = blockIdx.x * kSlice + lane;
    const int h = blockIdx.y, b = blockIdx.z;
    int64_t t0 = 0, t1 = N;
    if (cu_seqlens != nullptr) {
        t0 = cu_seqlens[b];
        t1 = cu_seqlens[b + 1];
        if (t0 < 0 || t1 < t0 || t1 > N) {
            if (tid == 0) record_device_error(err, kDevInvalidArg);
            return;
        }
    }
    const int64_t state_base = (static_cast<int64_t>(b) * H + h) * kD * kD;
    float S[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i)
        S[i] = (S0 != nullptr) ? S0[state_base + (warp + 8 * i) * kD + col] : 0.f;

    for (int64_t t = t0; t < t1; ++t) {
        const int64_t tok = t * H + h;
        if (tid < kD) {
            s_k[tid] = __bfloat162float(k[tok * kD + tid]);
            s_q[tid] = scale * __bfloat162float(q[tok * kD + tid]);
            s_d[tid] = expf(g[tok * kD + tid]);
        } else if (tid < kD + kSlice) {
            s_v[tid - kD] = __bfloat162float(v[tok * kD + blockIdx.x * kSlice + tid - kD]);
        } else if (tid == kD + kSlice) {
            s_beta = beta[tok];
        }
        __syncthreads();
        float w = 0.f, z = 0.f;
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const int r = warp + 8 * i;
            S[i] *= s_d[r];
            w += S[i] * s_k[r];
            z += S[i] * s_q[r];
        }
        s_red[0][warp][lane] = w;
        s_red[1][warp][lane] = z;
        __syncthreads();
        if (warp == 0) {
            float kq = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) kq += s_k[lane + 32 * j] * s_q[lane + 32 * j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
            float ws = 0.f, zs = 0.f;
#pragma unroll
            for (int j = 0; j < kThreads / 32; ++j) {
                ws += s_red[0][j][lane];
                zs += s_red[1][j][lane];
            }
            const float u = s_beta * (s_v[lane] - ws);
            s_u[lane] = u;
            const float out = zs + kq * u;
            if (kOutBf16)
                static_cast<__nv_bfloat16 *>(o)[tok * kD + col] = __float2bfloat16_rn(out);
            else
                static_cast<float *>(o)[tok * kD + col] = out;
        }
        __syncthreads();
        const float u = s_u[lane];
#pragma unroll
        for (int i = 0; i < kRows; ++i) S[i] += s_k[warp + 8 * i] * u;
        __syncthreads();
    }
    if (Sf != nullptr) {
#pragma unroll
        for (int i = 0; i < kRows; ++i) Sf[state_base + (warp + 8 * i) * kD + col] = S[i];
    }
}

}  // namespace

size_t prefill_workspace_bytes(int64_t N, int B, int H) {
    (void)N;
    return (B > 0 && H > 0) ? 256 : 0;
}

cudaError_t launch_prefill(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, const float *g, const float *beta,
                           const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
                           const float *initial_state, float *final_state, void *o, bool o_bf16,
                           void *workspace, unsigned int *err, int num_sms, cudaStream_t s) {
    (void)workspace;
    (void)num_sms;
    if (B == 0 || H == 0) return cudaSuccess;
    dim3 grid(kD / kSlice, H, B);
    if (o_bf16)
        prefill_recurrent_kernel<true><<<grid, kThreads, 0, s>>>(
            q, k, v, g, beta, cu_seqlens, N, H, scale, initial_state, final_state, o, err);
    else
        prefill_recurrent_kernel<false><<<grid, kThreads, 0, s>>>(
            q, k, v, g, beta, cu_seqlens, N, H, scale, initial_state, final_state, o, err);
    return cudaGetLastError();
}

}  // namespace kda

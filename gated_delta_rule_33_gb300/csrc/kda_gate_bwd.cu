// kda_gate_bwd.cu -- gradients of the KDA gate (the training regime's last
// step: from dL/dg and dL/dbeta of kda_recurrent_backward to the gate's own
// inputs).  With x = f + dt_bias, a = exp(A_log), g = -a softplus(x) and
// beta = sigmoid(b) (K3_ARTIFACT_AUDIT.md sections 4.1 and 5.1):
//
//   df            = dg * (-a sigmoid(x))          (softplus' = sigmoid)
//   d dt_bias     = sum over tokens of df
//   d A_log       = sum of dg * g over the axes A_log is broadcast along
//   db            = dbeta * beta (1 - beta)
//
// x, a, g and beta are formed with the forward gate's binary32 specification
// (kda_gate_spec.cuh), so they are the values the forward pass produced.
//
// Data path: HBM-bound, like the gate.  One thread owns 8 consecutive channels
// of one head and walks token rows with a fixed stride, so its parameters are
// loaded once and its partial sums for d dt_bias and d A_log stay in
// registers; the partials go to a workspace and two small kernels add them in
// a fixed order (deterministic results).
#include "kda_gate_spec.cuh"

namespace kda {
namespace {

using namespace gate_spec;

constexpr int kMaxRowGroups = 256;

__device__ __forceinline__ float sigmoid_f32(float x) { return 1.f / (1.f + expf(-x)); }

// grid: HK8 * R threads; thread t owns octet t % HK8 and rows t / HK8 + R j.
__global__ void __launch_bounds__(256) gate_bwd_kernel(
    const void *__restrict__ f, bool f_bf16, const void *__restrict__ b, bool b_bf16,
    const float *__restrict__ A_log, int alog_mode, const float *__restrict__ dt_bias,
    const float *__restrict__ dg, const float *__restrict__ dbeta, float *__restrict__ df,
    float *__restrict__ db, float *__restrict__ part_dt, float *__restrict__ part_da, int64_t N,
    int H, int K, int R) {
    const int64_t HK8 = static_cast<int64_t>(H) * K / 8;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (tid >= HK8 * R) return;
    const int64_t oct = tid % HK8;
    const int row0 = static_cast<int>(tid / HK8);
    const int h = static_cast<int>((oct * 8) / K);
    const int c0 = static_cast<int>((oct * 8) % K);
    float a[8], dt[8], sdt[8], sda[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a[j] = gate_exp(alog_at(A_log, alog_mode, h, c0 + j, K));
        dt[j] = dt_bias[oct * 8 + j];
        sdt[j] = 0.f;
        sda[j] = 0.f;
    }
    const bool do_beta = (b != nullptr) && (c0 == 0);
    for (int64_t r = row0; r < N; r += R) {
        const int64_t base = r * (HK8 * 8) + oct * 8;
        float fv[8], gv[8];
        if (f_bf16) {
            const uint4 raw = __ldcs(reinterpret_cast<const uint4 *>(
                static_cast<const __nv_bfloat16 *>(f) + base));
            const __nv_bfloat162 *pairs = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 p = __bfloat1622float2(pairs[j]);
                fv[2 * j] = p.x;
                fv[2 * j + 1] = p.y;
            }
        } else {
            const float4 lo = __ldcs(reinterpret_cast<const float4 *>(static_cast<const float *>(f) + base));
            const float4 hi = __ldcs(reinterpret_cast<const float4 *>(static_cast<const float *>(f) + base + 4));
            fv[0] = lo.x; fv[1] = lo.y; fv[2] = lo.z; fv[3] = lo.w;
            fv[4] = hi.x; fv[5] = hi.y; fv[6] = hi.z; fv[7] = hi.w;
        }
        const float4 g_lo = __ldcs(reinterpret_cast<const float4 *>(dg + base));
        const float4 g_hi = __ldcs(reinterpret_cast<const float4 *>(dg + base + 4));
        gv[0] = g_lo.x; gv[1] = g_lo.y; gv[2] = g_lo.z; gv[3] = g_lo.w;
        gv[4] = g_hi.x; gv[5] = g_hi.y; gv[6] = g_hi.z; gv[7] = g_hi.w;
        float out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float x = __fadd_rn(fv[j], dt[j]);
            out[j] = gv[j] * (-a[j] * sigmoid_f32(x));
            sdt[j] += out[j];
            sda[j] += gv[j] * gate_g(fv[j], dt[j], a[j]);
        }
        __stcs(reinterpret_cast<float4 *>(df + base), make_float4(out[0], out[1], out[2], out[3]));
        __stcs(reinterpret_cast<float4 *>(df + base + 4), make_float4(out[4], out[5], out[6], out[7]));
        if (do_beta) {
            const int64_t bi = r * H + h;
            const float bl = b_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(b)[bi])
                                    : static_cast<const float *>(b)[bi];
            const float bt = gate_sigmoid(bl);
            db[bi] = dbeta[bi] * bt * (1.f - bt);
        }
    }
    float *pdt = part_dt + static_cast<int64_t>(row0) * H * K + oct * 8;
    float *pda = part_da + static_cast<int64_t>(row0) * H * K + oct * 8;
    *reinterpret_cast<float4 *>(pdt) = make_float4(sdt[0], sdt[1], sdt[2], sdt[3]);
    *reinterpret_cast<float4 *>(pdt + 4) = make_float4(sdt[4], sdt[5], sdt[6], sdt[7]);
    *reinterpret_cast<float4 *>(pda) = make_float4(sda[0], sda[1], sda[2], sda[3]);
    *reinterpret_cast<float4 *>(pda + 4) = make_float4(sda[4], sda[5], sda[6], sda[7]);
}

// One thread per (h, c): the row-group partials in order.
__global__ void gate_bwd_reduce_rows(const float *__restrict__ part_dt,
                                     const float *__restrict__ part_da, float *__restrict__ ddt,
                                     float *__restrict__ s_hc, int HK, int R) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= HK) return;
    float a = 0.f, c = 0.f;
    for (int r = 0; r < R; ++r) {
        a += part_dt[static_cast<int64_t>(r) * HK + i];
        c += part_da[static_cast<int64_t>(r) * HK + i];
    }
    if (ddt != nullptr) ddt[i] = a;
    s_hc[i] = c;
}

// d A_log by mode from the per-(h, c) sums, in order.
__global__ void gate_bwd_reduce_alog(const float *__restrict__ s_hc, float *__restrict__ dA,
                                     int mode, int H, int K) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (mode == 0) {          // [H]: over channels
        if (i >= H) return;
        float acc = 0.f;
        for (int c = 0; c < K; ++c) acc += s_hc[i * K + c];
        dA[i] = acc;
    } else if (mode == 1) {   // [K]: over heads
        if (i >= K) return;
        float acc = 0.f;
        for (int h = 0; h < H; ++h) acc += s_hc[h * K + i];
        dA[i] = acc;
    } else {                  // [H, K]
        if (i >= H * K) return;
        dA[i] = s_hc[i];
    }
}

}  // namespace

int gate_bwd_row_groups(int64_t N) {
    return static_cast<int>(N < kMaxRowGroups ? (N > 0 ? N : 1) : kMaxRowGroups);
}

size_t gate_bwd_workspace_bytes(int64_t N, int H, int K) {
    if (N < 0 || H < 1 || K < 1) return 0;
    const size_t hk = static_cast<size_t>(H) * K;
    return (2 * static_cast<size_t>(gate_bwd_row_groups(N)) + 1) * hk * sizeof(float);
}

cudaError_t launch_gate_backward(const void *f, bool f_bf16, const void *b, bool b_bf16,
                                 const float *A_log, int alog_mode, const float *dt_bias,
                                 const float *dg, const float *dbeta, float *df, float *db,
                                 float *dA_log, float *ddt_bias, int64_t N, int H, int K,
                                 void *workspace, cudaStream_t s) {
    const int R = gate_bwd_row_groups(N);
    const int64_t hk = static_cast<int64_t>(H) * K;
    float *part_dt = static_cast<float *>(workspace);
    float *part_da = part_dt + R * hk;
    float *s_hc = part_da + R * hk;
    const int64_t threads = hk / 8 * R;
    gate_bwd_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(
        f, f_bf16, b, b_bf16, A_log, alog_mode, dt_bias, dg, dbeta, df, db, part_dt, part_da, N,
        H, K, R);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    gate_bwd_reduce_rows<<<static_cast<unsigned>((hk + 255) / 256), 256, 0, s>>>(
        part_dt, part_da, ddt_bias, s_hc, static_cast<int>(hk), R);
    e = cudaGetLastError();
    if (e != cudaSuccess || dA_log == nullptr) return e;
    gate_bwd_reduce_alog<<<static_cast<unsigned>((hk + 255) / 256), 256, 0, s>>>(
        s_hc, dA_log, alog_mode, H, K);
    return cudaGetLastError();
}

}  // namespace kda

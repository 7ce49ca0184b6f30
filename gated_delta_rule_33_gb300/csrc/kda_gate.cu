// kda_gate.cu -- the KDA gate in one coalesced, vectorised pass.
//
//   g[n,h,c]  = -(exp(A_log[.]) * softplus(f[n,h,c] + dt_bias[h,c]))
//   beta[n,h] = 1 / (1 + exp(-b[n,h]))
//
// Parameters as in K3_ARTIFACT_AUDIT.md section 4.1 (A_log, dt_bias [96 x 128],
// b_proj per head, low-rank f) and section 5.1 (their statistics); beta is an
// fp32 sigmoid of the raw logits, the requirement behind finding 1 of the
// "[OMNIML-6079] [20/21] Add the Kimi-K3 expert-parallel adapter" review.
//
// The result is bit-exact with respect to a fixed binary32 specification
// (kda_gate_spec.cuh: explicitly rounded intrinsics and this library's own
// Cody-Waite exp and atanh-series log1p).
//
// Data path: HBM-bound.  One thread owns 8 consecutive channels of one head
// (a 16-byte bf16 load of f, two 16-byte stores of g) and walks token rows with
// a stride chosen so that its (head, channel) set never changes: exp(A_log) and
// dt_bias are computed/loaded once per thread.
#include "kda_gate_spec_x2.cuh"

namespace kda {
namespace {

using namespace gate_spec;

__device__ __forceinline__ float load_as_f32(const void *p, int64_t i, bool is_bf16) {
    return is_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i])
                   : static_cast<const float *>(p)[i];
}


// Vector path: H*K % 8 == 0, K % 8 == 0, pointers 16-byte aligned.
// Thread t owns channel octet (t % HK8) and rows t / HK8, + row_stride, ...
template <bool kFBf16>
__global__ void __launch_bounds__(256) gate_vec_kernel(
    const void *__restrict__ f, const void *__restrict__ b, bool b_bf16,
    const float *__restrict__ A_log, int alog_mode, const float *__restrict__ dt_bias,
    float *__restrict__ g, float *__restrict__ beta, int64_t N, int H, int K,
    int64_t row_stride) {
    const int64_t HK8 = static_cast<int64_t>(H) * K / 8;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (tid >= HK8 * row_stride) return;
    const int64_t oct = tid % HK8;
    const int64_t row0 = tid / HK8;
    const int h = static_cast<int>((oct * 8) / K);
    const int c0 = static_cast<int>((oct * 8) % K);

    float dt[8], a[8];
    const float4 dt_lo = *reinterpret_cast<const float4 *>(dt_bias + oct * 8);
    const float4 dt_hi = *reinterpret_cast<const float4 *>(dt_bias + oct * 8 + 4);
    dt[0] = dt_lo.x; dt[1] = dt_lo.y; dt[2] = dt_lo.z; dt[3] = dt_lo.w;
    dt[4] = dt_hi.x; dt[5] = dt_hi.y; dt[6] = dt_hi.z; dt[7] = dt_hi.w;
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = gate_exp(alog_at(A_log, alog_mode, h, c0 + j, K));
    const bool do_beta = (b != nullptr) && (c0 == 0);

    for (int64_t r = row0; r < N; r += row_stride) {
        const int64_t base = r * (HK8 * 8) + oct * 8;
        float fv[8];
        if (kFBf16) {
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
        float out[8];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {  // packed pairs, the same bits as gate_g
            const float2 gp = gate_g_x2(fv[j], fv[j + 1], dt[j], dt[j + 1], a[j], a[j + 1]);
            out[j] = gp.x;
            out[j + 1] = gp.y;
        }
        __stcs(reinterpret_cast<float4 *>(g + base), make_float4(out[0], out[1], out[2], out[3]));
        __stcs(reinterpret_cast<float4 *>(g + base + 4), make_float4(out[4], out[5], out[6], out[7]));
        if (do_beta) {
            const int64_t bi = r * H + h;
            beta[bi] = gate_sigmoid(load_as_f32(b, bi, b_bf16));
        }
    }
}

// Generic path: any K; one element per thread iteration.
__global__ void __launch_bounds__(256) gate_scalar_kernel(
    const void *__restrict__ f, bool f_bf16, const void *__restrict__ b, bool b_bf16,
    const float *__restrict__ A_log, int alog_mode, const float *__restrict__ dt_bias,
    float *__restrict__ g, float *__restrict__ beta, int64_t N, int H, int K) {
    const int64_t total = N * H * K;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += stride) {
        const int c = static_cast<int>(i % K);
        const int64_t nh = i / K;
        const int h = static_cast<int>(nh % H);
        const float a = gate_exp(alog_at(A_log, alog_mode, h, c, K));
        g[i] = gate_g(load_as_f32(f, i, f_bf16), dt_bias[static_cast<int64_t>(h) * K + c], a);
        if (b != nullptr && c == 0) beta[nh] = gate_sigmoid(load_as_f32(b, nh, b_bf16));
    }
}

}  // namespace

cudaError_t launch_gate(const void *f, bool f_bf16, const void *b, bool b_bf16,
                        const float *A_log, int alog_mode, const float *dt_bias, float *g,
                        float *beta, int64_t N, int H, int K, int num_sms, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int64_t HK = static_cast<int64_t>(H) * K;
    const int threads = 256;
    if (K % 8 == 0) {
        const int64_t HK8 = HK / 8;
        const int64_t target = static_cast<int64_t>(num_sms) * 2048;  // resident threads
        int64_t rows = (target + HK8 - 1) / HK8;
        if (rows > N) rows = N;
        if (rows < 1) rows = 1;
        const int64_t blocks = (HK8 * rows + threads - 1) / threads;
        if (f_bf16)
            gate_vec_kernel<true><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
                f, b, b_bf16, A_log, alog_mode, dt_bias, g, beta, N, H, K, rows);
        else
            gate_vec_kernel<false><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
                f, b, b_bf16, A_log, alog_mode, dt_bias, g, beta, N, H, K, rows);
    } else {
        int64_t blocks = (N * HK + threads - 1) / threads;
        const int64_t cap = static_cast<int64_t>(num_sms) * 8;
        if (blocks > cap) blocks = cap;
        gate_scalar_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
            f, f_bf16, b, b_bf16, A_log, alog_mode, dt_bias, g, beta, N, H, K);
    }
    return cudaGetLastError();
}

namespace {

__device__ unsigned long long g_division_mismatches;

// Every operand pair of the two divisions in the gate's common path, through
// div2_common, against IEEE division: index i < kY runs y over every normal
// binary32 value in [2^-126, 1] (a = y - (u - 1), b = u = 1 + y, as formed
// there); the rest runs u over every binary32 value in [1, 2] (a = f, b = 2 + f
// with f = u - 1, or u / 2 - 1 above sqrt 2).  Consecutive indices make the
// pairs of the packed division.
constexpr uint32_t kYLo = 0x00800000u, kYHi = 0x3f800000u;   // 2^-126 .. 1
constexpr uint32_t kULo = 0x3f800000u, kUHi = 0x40000000u;   // [1, 2]
constexpr int64_t kY = kYHi - kYLo + 1, kU = kUHi - kULo + 1;

__device__ __forceinline__ void division_operands(int64_t i, float &a, float &b) {
    if (i < kY) {
        const float y = __uint_as_float(kYLo + static_cast<uint32_t>(i));
        const float u = __fadd_rn(1.0f, y);
        a = __fsub_rn(y, __fsub_rn(u, 1.0f));
        b = u;
    } else {
        const float u = __uint_as_float(kULo + static_cast<uint32_t>(i - kY));
        const float f = __fsub_rn(__fmul_rn(u, u > 0x1.6a09e6p+0f ? 0.5f : 1.0f), 1.0f);
        a = f;
        b = __fadd_rn(2.0f, f);
    }
}

__global__ void __launch_bounds__(256) gate_division_check_kernel() {
    unsigned long long bad = 0;
    const int64_t n = kY + kU;
    for (int64_t i = 2 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x); i < n;
         i += 2 * static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float a0, b0, a1 = 1.0f, b1 = 1.0f;
        division_operands(i, a0, b0);
        if (i + 1 < n) division_operands(i + 1, a1, b1);
        const float2 q = f2_split(div2_common(f2(a0, a1), f2(b0, b1)));
        if (__float_as_uint(q.x) != __float_as_uint(__fdiv_rn(a0, b0))) ++bad;
        if (i + 1 < n && __float_as_uint(q.y) != __float_as_uint(__fdiv_rn(a1, b1))) ++bad;
    }
    if (bad != 0) atomicAdd(&g_division_mismatches, bad);
}

}  // namespace

cudaError_t check_gate_division(unsigned long long *mismatches, int num_sms, cudaStream_t s) {
    const unsigned long long zero = 0;
    cudaError_t e = cudaMemcpyToSymbolAsync(g_division_mismatches, &zero, sizeof(zero), 0,
                                            cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    gate_division_check_kernel<<<static_cast<unsigned>(num_sms) * 8, 256, 0, s>>>();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbolAsync(mismatches, g_division_mismatches, sizeof(*mismatches), 0,
                                  cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

}  // namespace kda

// kda_decode.cu -- fused recurrent KDA for one-token cached decoding.
//
// The Kimi-K3 code audit (data/code-audit.json, finding
// "dual-kda-execution-regimes") names this regime: one new token per sequence
// against a cached state.  For each (sequence, head), with the 128 x 128 fp32
// state S (d_k rows, d_v columns):
//
//   S' = Diag(exp(g)) S
//   w  = S'^T k,   z = S'^T (scale q)
//   u  = beta (v - w)
//   S  = S' + k u^T                   (written back in place)
//   o  = S^T (scale q) = z + (scale k.q) u
//
// Data path: the step is HBM-bound (0.9 flop/byte); every state is read once
// and written once.  One 256-thread CTA per (sequence, head): warp w owns rows
// w, w+8, ..., w+120 and lane l owns columns 4l..4l+3, so each warp-wide 16-byte
// load or store moves one contiguous 512-byte state row.  The 64 KB state stays
// in registers (16 float4 per thread) between the column reductions and the
// write, so HBM sees exactly one read and one write of it.  A bf16 state (32 KB)
// is staged in shared memory instead, by 16-byte cp.async: it holds no
// registers, so six CTAs share an SM and their loads keep more bytes in flight
// than register-held states could.
#include "kda_gate_spec.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr int kRowsPerThread = kD / (kThreads / 32);  // 16

// The thread's 16 x 4 state elements between the two passes of a step: fp32
// values in registers, or a bf16 state read from its copy in shared memory
// (widened where used).
template <bool kStateBf16>
struct StateRegs;

template <>
struct StateRegs<false> {
    float4 v[kRowsPerThread];
    __device__ __forceinline__ void load(int i, const void *S, int64_t idx) {
        v[i] = __ldcs(reinterpret_cast<const float4 *>(static_cast<const float *>(S) + idx));
    }
    __device__ __forceinline__ float4 get(int i) const { return v[i]; }
    __device__ __forceinline__ void store(void *S, int64_t idx, float4 x) const {
        __stcs(reinterpret_cast<float4 *>(static_cast<float *>(S) + idx), x);
    }
};

template <>
struct StateRegs<true> {
    const uint2 *sp;  // this thread's columns of row `warp` of the staged state
    __device__ __forceinline__ float4 get(int i) const {
        const uint2 raw = sp[i * 8 * (kD / 4)];  // row warp + 8 i
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    __device__ __forceinline__ void store(void *S, int64_t idx, float4 x) const {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y);
        const __nv_bfloat162 b = __floats2bfloat162_rn(x.z, x.w);
        uint2 raw;
        raw.x = *reinterpret_cast<const uint32_t *>(&a);
        raw.y = *reinterpret_cast<const uint32_t *>(&b);
        __stcs(reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(S) + idx), raw);
    }
};

// The gate inputs of the gated decode (kGate): g and beta are computed here
// from them with the same binary32 operations as the gate kernel.
struct DecodeGate {
    const void *f;          // [B, H, 128] pre-activation, bf16 or fp32
    int f_bf16;
    const void *b;          // [B, H] beta logits, bf16 or fp32
    int b_bf16;
    const float *A_log;
    int alog_mode;
    const float *dt_bias;   // [H, 128]
};

// One CTA per (sequence, head).  With `slots` the state of sequence b lives in
// pool slot slots[b] (negative: inactive sequence, nothing read or written,
// o = 0; >= num_slots: a device error, skipped); without it, slot b.
template <bool kOutBf16, bool kStateBf16, bool kGate>
__global__ void __launch_bounds__(kThreads, kStateBf16 ? 6 : 2) decode_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const float *__restrict__ g,
    const float *__restrict__ beta, const DecodeGate gt, void *__restrict__ state,
    const int32_t *__restrict__ slots, int num_slots, int H, float scale,
    void *__restrict__ o, unsigned int *err) {
    __shared__ float s_k[kD], s_q[kD], s_decay[kD];
    __shared__ __align__(16) float s_u[kD];                   // read as float4
    __shared__ __align__(16) float s_red[2][kThreads / 32][kD];   // written as float4
    __shared__ float s_kq, s_beta;
    __shared__ __align__(16) uint8_t s_state[kStateBf16 ? kD * kD * 2 : 16];

    const int64_t bh = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t slot = bh / H;
    if (slots != nullptr) {
        const int sl = slots[bh / H];
        if (sl < 0 || sl >= num_slots) {
            if (sl >= num_slots && tid == 0) record_device_error(err, kDevInvalidArg);
            if (tid < kD) {
                if (kOutBf16)
                    static_cast<__nv_bfloat16 *>(o)[bh * kD + tid] = __float2bfloat16_rn(0.f);
                else
                    static_cast<float *>(o)[bh * kD + tid] = 0.f;
            }
            return;
        }
        slot = sl;
    }
    const int64_t sbase = (slot * H + bh % H) * (kD * kD);

    // Issue the whole state read first: the full state in flight per CTA.
    StateRegs<kStateBf16> s;
    if constexpr (kStateBf16) {
        const uint8_t *src = static_cast<const uint8_t *>(state) + sbase * 2;
#pragma unroll
        for (int j = 0; j < kD * kD * 2 / 16 / kThreads; ++j)
            sm100::cp_async_16(s_state + (tid + kThreads * j) * 16, src + (tid + kThreads * j) * 16, true);
        s.sp = reinterpret_cast<const uint2 *>(s_state) + warp * (kD / 4) + lane;
    } else {
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) s.load(i, state, sbase + (warp + 8 * i) * kD + 4 * lane);
    }

    if (tid < kD) {
        const int64_t idx = bh * kD + tid;
        s_k[tid] = __bfloat162float(k[idx]);
        s_q[tid] = scale * __bfloat162float(q[idx]);
        if (!kGate) {
            s_decay[tid] = expf(g[idx]);
            if (tid == 0) s_beta = beta[bh];
        }
    } else if (kGate) {
        // the gate on the other four warps, alongside the loads above
        using namespace gate_spec;
        const int c = tid - kD;
        const int64_t idx = bh * kD + c;
        const int h = static_cast<int>(bh % H);
        const float fv = gt.f_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(gt.f)[idx])
                                   : static_cast<const float *>(gt.f)[idx];
        const float a = gate_exp(alog_at(gt.A_log, gt.alog_mode, h, c, kD));
        s_decay[c] = expf(gate_g(fv, gt.dt_bias[h * kD + c], a));
        if (c == 0) {
            const float bl = gt.b_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(gt.b)[bh])
                                       : static_cast<const float *>(gt.b)[bh];
            s_beta = gate_sigmoid(bl);
        }
    }
    if constexpr (kStateBf16) sm100::cp_async_wait_all();
    __syncthreads();

    if (warp == 0) {  // scale * k.q
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc += s_k[lane + 32 * j] * s_q[lane + 32 * j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) s_kq = acc;
    }

    float4 w = make_float4(0.f, 0.f, 0.f, 0.f), z = w;
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        const int r = warp + 8 * i;
        const float d = s_decay[r], kr = s_k[r], qr = s_q[r];
        float4 x = s.get(i);
        x.x *= d; x.y *= d; x.z *= d; x.w *= d;
        if constexpr (!kStateBf16) s.v[i] = x;   // fp32: keep S'; bf16: formed again below
        w.x += x.x * kr; w.y += x.y * kr; w.z += x.z * kr; w.w += x.w * kr;
        z.x += x.x * qr; z.y += x.y * qr; z.z += x.z * qr; z.w += x.w * qr;
    }
    reinterpret_cast<float4 *>(s_red[0][warp])[lane] = w;
    reinterpret_cast<float4 *>(s_red[1][warp])[lane] = z;
    __syncthreads();

    if (tid < kD) {
        float ws = 0.f, zs = 0.f;
#pragma unroll
        for (int j = 0; j < kThreads / 32; ++j) {
            ws += s_red[0][j][tid];
            zs += s_red[1][j][tid];
        }
        const float u = s_beta * (__bfloat162float(v[bh * kD + tid]) - ws);
        s_u[tid] = u;
        const float out = zs + s_kq * u;
        if (kOutBf16)
            static_cast<__nv_bfloat16 *>(o)[bh * kD + tid] = __float2bfloat16_rn(out);
        else
            static_cast<float *>(o)[bh * kD + tid] = out;
    }
    __syncthreads();

    const float4 u4 = reinterpret_cast<const float4 *>(s_u)[lane];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        const int r = warp + 8 * i;
        const float kr = s_k[r];
        float4 x = s.get(i);
        if constexpr (kStateBf16) {
            const float d = s_decay[r];
            x.x *= d; x.y *= d; x.z *= d; x.w *= d;
        }
        x.x += kr * u4.x; x.y += kr * u4.y; x.z += kr * u4.z; x.w += kr * u4.w;
        s.store(state, sbase + r * kD + 4 * lane, x);
    }
}

}  // namespace

template <bool kOutBf16, bool kGate>
static cudaError_t launch_decode_t(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                   const __nv_bfloat16 *v, const float *g, const float *beta,
                                   const DecodeGate &gt, void *state, bool state_bf16,
                                   const int32_t *slots, int num_slots, int64_t units, int H,
                                   float scale, void *o, unsigned int *err, cudaStream_t s) {
    if (state_bf16)
        decode_kernel<kOutBf16, true, kGate><<<static_cast<unsigned>(units), kThreads, 0, s>>>(
            q, k, v, g, beta, gt, state, slots, num_slots, H, scale, o, err);
    else
        decode_kernel<kOutBf16, false, kGate><<<static_cast<unsigned>(units), kThreads, 0, s>>>(
            q, k, v, g, beta, gt, state, slots, num_slots, H, scale, o, err);
    return cudaGetLastError();
}

cudaError_t launch_decode(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                          const __nv_bfloat16 *v, const float *g, const float *beta,
                          float *state, int B, int H, float scale, void *o, bool o_bf16,
                          cudaStream_t s) {
    const int64_t units = static_cast<int64_t>(B) * H;
    if (units == 0) return cudaSuccess;
    const DecodeGate none{};
    return o_bf16 ? launch_decode_t<true, false>(q, k, v, g, beta, none, state, false, nullptr, B,
                                                 units, H, scale, o, nullptr, s)
                  : launch_decode_t<false, false>(q, k, v, g, beta, none, state, false, nullptr, B,
                                                  units, H, scale, o, nullptr, s);
}

cudaError_t launch_decode_indexed(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                  const __nv_bfloat16 *v, const float *g, const float *beta,
                                  void *state_pool, bool state_bf16, const int32_t *slots,
                                  int num_slots, int B, int H, float scale, void *o, bool o_bf16,
                                  unsigned int *err, cudaStream_t s) {
    const int64_t units = static_cast<int64_t>(B) * H;
    if (units == 0) return cudaSuccess;
    const DecodeGate none{};
    return o_bf16 ? launch_decode_t<true, false>(q, k, v, g, beta, none, state_pool, state_bf16,
                                                 slots, num_slots, units, H, scale, o, err, s)
                  : launch_decode_t<false, false>(q, k, v, g, beta, none, state_pool, state_bf16,
                                                  slots, num_slots, units, H, scale, o, err, s);
}

cudaError_t launch_decode_gated(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                const __nv_bfloat16 *v, const void *f, bool f_bf16, const void *b,
                                bool b_bf16, const float *A_log, int alog_mode,
                                const float *dt_bias, void *state_pool, bool state_bf16,
                                const int32_t *slots, int num_slots, int B, int H, float scale,
                                void *o, bool o_bf16, unsigned int *err, cudaStream_t s) {
    const int64_t units = static_cast<int64_t>(B) * H;
    if (units == 0) return cudaSuccess;
    const DecodeGate gt{f, f_bf16 ? 1 : 0, b, b_bf16 ? 1 : 0, A_log, alog_mode, dt_bias};
    return o_bf16 ? launch_decode_t<true, true>(q, k, v, nullptr, nullptr, gt, state_pool,
                                                state_bf16, slots, num_slots, units, H, scale, o,
                                                err, s)
                  : launch_decode_t<false, true>(q, k, v, nullptr, nullptr, gt, state_pool,
                                                 state_bf16, slots, num_slots, units, H, scale, o,
                                                 err, s);
}

}  // namespace kda

// kda_backward.cu -- gradients of the KDA recurrence (the training regime:
// "chunked KDA for training", data/code-audit.json, finding
// "dual-kda-execution-regimes"), token by token on CUDA cores.
//
// Forward step (per sequence and head, 128 x 128 fp32 state, d_k rows):
//   S' = Diag(exp g_t) S_{t-1};  w = S'^T k_t;  u = beta_t (v_t - w)
//   S_t = S' + k_t u^T;          o_t = S_t^T (scale q_t)
// Reverse step, from G = dL/dS_t (dL/dS_T given, or zero):
//   G    += (scale q_t) do_t^T
//   du    = G^T k_t;   dv_t = beta_t du;   dbeta_t = du . (v_t - w);   dw = -beta_t du
//   dk_t  = G u + S' dw
//   dq_t  = scale S_t do_t = scale (S' do_t + k_t (u . do_t))
//   dg_t  = rowsum((G + k_t dw^T) (.) S') = rowsum(G (.) S') + k_t (S' dw)
//   G     = Diag(exp g_t) (G + k_t dw^T)                       (= dL/dS_{t-1})
// and dL/dS_0 = G at the end.
//
// The reverse step needs S_{t-1}.  One CTA runs a whole (sequence, head)
// chain: a forward pass stores a checkpoint of the state every kCk tokens;
// then, segment by segment from the last, the forward steps of the segment are
// rerun from its checkpoint writing each S_{t-1} to a per-CTA scratch, and the
// reverse steps read them back (each step's token vectors and S_{t-1} are
// requested one step ahead, so no step waits a full memory latency).  Every thread reads back only the elements it
// wrote, so checkpoints and scratch are kept in a thread-interleaved order
// (for a fixed row slot, the 256 threads' float4 are contiguous).
//
// Element ownership: 16 warps, warp w owns rows w, w+16, ..., w+112 and lane l
// owns columns 4l..4l+3 (8 rows x 4 columns per thread).  Column sums (w, du)
// reduce over a thread's 8 rows, then over the 16 warps in shared memory; row
// sums (for dk, dq, dg) reduce over the 32 lanes with a halving exchange that
// leaves lane l holding one of the 32 (row, quantity) sums of the step.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = kD / kWarps;   // rows per thread (8)
constexpr int kCk = 16;          // tokens per checkpoint segment
constexpr int kStateF4 = kD * kD / 4;   // float4 per state

struct BwdParams {
    const __nv_bfloat16 *q, *k, *v;
    const float *g, *beta;
    const int32_t *cu_seqlens;
    int B;
    int64_t N;
    int H;
    float scale;
    const float *S0;       // [B, H, 128, 128] or null
    const void *dO;        // [N, H, 128] bf16 or fp32
    int dO_bf16;
    const float *dSf;      // [B, H, 128, 128] or null
    float *dq, *dk, *dv, *dg, *dbeta, *dS0;
    float4 *ckpt;          // checkpoint slots x H states (thread-interleaved)
    float4 *scratch;       // per CTA: kCk states (thread-interleaved)
    unsigned int *counter;
    unsigned int *err;
};

// 16-byte aligned (and so padded to a multiple of 16 bytes): the reverse
// step reads dO as float4.
struct __align__(16) TokenVecs {
    float q[kD], k[kD], v[kD], d[kD], dO[kD];
    float beta;
};
static_assert(sizeof(TokenVecs) % 16 == 0, "TokenVecs must keep float4 alignment in arrays");

__device__ __forceinline__ float4 f4_scale(float4 a, float s) {
    return make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
}
__device__ __forceinline__ float4 f4_fma(float s, float4 b, float4 c) {   // s b + c
    return make_float4(fmaf(s, b.x, c.x), fmaf(s, b.y, c.y), fmaf(s, b.z, c.z), fmaf(s, b.w, c.w));
}
__device__ __forceinline__ float f4_dot(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// Halving exchange over the 32 lanes: on entry every lane holds 32 values
// (one per (row, quantity) slot); on exit lane l holds, in v[0], the sum over
// all lanes of slot l.  31 shuffles instead of 32 x 5.
__device__ __forceinline__ void lane_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int o = 16, half = 16; o > 0; o >>= 1, half >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float give = up ? v[j] : v[j + half];
            const float keep = up ? v[j + half] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, give, o);
        }
    }
}

// A token's vectors as loaded by threads 0..127 (raw, so that nothing waits
// on the loads until commit_token), one step before they are used.
struct TokenRegs {
    __nv_bfloat16 q, k, v;
    float g, beta;
    uint32_t dO;     // bf16 or fp32 bits
};

template <bool kDoBf16>
__device__ __forceinline__ void fetch_token(const BwdParams &p, int64_t t, int h, int tid,
                                            TokenRegs &r) {
    if (tid < kD) {
        const int64_t idx = (t * p.H + h) * kD + tid;
        r.q = p.q[idx];
        r.k = p.k[idx];
        r.v = p.v[idx];
        r.g = p.g[idx];
        if (kDoBf16)
            r.dO = static_cast<const unsigned short *>(p.dO)[idx];
        else
            r.dO = static_cast<const uint32_t *>(p.dO)[idx];
        if (tid == 0) r.beta = p.beta[t * p.H + h];
    }
}

template <bool kDoBf16>
__device__ __forceinline__ void commit_token(const BwdParams &p, const TokenRegs &r,
                                             TokenVecs &tv, int tid) {
    if (tid < kD) {
        tv.q[tid] = p.scale * __bfloat162float(r.q);
        tv.k[tid] = __bfloat162float(r.k);
        tv.v[tid] = __bfloat162float(r.v);
        tv.d[tid] = expf(r.g);
        tv.dO[tid] = kDoBf16 ? __uint_as_float(r.dO << 16) : __uint_as_float(r.dO);
        if (tid == 0) tv.beta = r.beta;
    }
}

// 16-byte asynchronous global -> shared copy (own data: only the issuing
// thread reads it back, after cp_async_wait<N>).
__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool kDoBf16>
__global__ void __launch_bounds__(kThreads, 1) backward_kernel(const BwdParams p) {
    // float4 accesses below: every array 16-byte aligned
    extern __shared__ float4 s_prev[];   // [2][kStateF4]: S_{t-1} of the next two steps
    __shared__ TokenVecs s_tok[2];
    __shared__ __align__(16) float s_red[2][kThreads / 32][kD];
    __shared__ __align__(16) float s_u[kD];
    __shared__ __align__(16) float s_dw[kD];
    __shared__ float s_sc[2][4];
    __shared__ int s_chain;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = 4 * lane;
    const int H = p.H;
    const int num_chains = p.B * H;
    float4 *scratch = p.scratch + static_cast<int64_t>(blockIdx.x) * kCk * kStateF4;

    while (true) {
        __syncthreads();
        if (tid == 0) s_chain = static_cast<int>(atomicAdd(p.counter, 1u));
        __syncthreads();
        const int chain = s_chain;
        if (chain >= num_chains) break;
        const int b = chain / H, h = chain % H;
        int64_t t0 = 0, t1 = p.N;
        if (p.cu_seqlens != nullptr) {
            t0 = p.cu_seqlens[b];
            t1 = p.cu_seqlens[b + 1];
            if (t0 < 0 || t1 < t0 || t1 > p.N) {
                if (tid == 0) record_device_error(p.err, kDevInvalidArg);
                continue;
            }
        }
        const int64_t state_off = (static_cast<int64_t>(b) * H + h) * kD * kD;
        const int nseg = static_cast<int>((t1 - t0 + kCk - 1) / kCk);
        // checkpoint slot of segment j: floor(t0 / kCk) + b + j (disjoint across sequences)
        const int64_t slot0 = t0 / kCk + b;
        auto ckpt_at = [&](int j, int i) -> float4 * {
            return p.ckpt + ((slot0 + j) * H + h) * kStateF4 + i * kThreads + tid;
        };

        float4 s[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            s[i] = (p.S0 != nullptr)
                       ? *reinterpret_cast<const float4 *>(p.S0 + state_off + (warp + kWarps * i) * kD + c0)
                       : make_float4(0.f, 0.f, 0.f, 0.f);

        // One forward step on s (token vectors in tv, visible to all threads).
        auto forward_step = [&](const TokenVecs &tv) {
            float4 wp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                const int r = warp + kWarps * i;
                s[i] = f4_scale(s[i], tv.d[r]);
                wp = f4_fma(tv.k[r], s[i], wp);
            }
            *reinterpret_cast<float4 *>(&s_red[0][warp][c0]) = wp;
            __syncthreads();
            if (tid < kD) {
                float w = 0.f;
#pragma unroll
                for (int j = 0; j < kThreads / 32; ++j) w += s_red[0][j][tid];
                s_u[tid] = tv.beta * (tv.v[tid] - w);
            }
            __syncthreads();
            const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[c0]);
#pragma unroll
            for (int i = 0; i < kRows; ++i) s[i] = f4_fma(tv.k[warp + kWarps * i], u4, s[i]);
        };

        // ---- forward pass: checkpoints at the start of every segment ----
        for (int j = 0; j < nseg; ++j) {
#pragma unroll
            for (int i = 0; i < kRows; ++i) *ckpt_at(j, i) = s[i];
            if (j == nseg - 1) break;   // the last segment's steps are not needed here
            const int64_t ts = t0 + static_cast<int64_t>(j) * kCk;
            TokenRegs tr;
            fetch_token<kDoBf16>(p, ts, h, tid, tr);
            for (int64_t t = ts; t < ts + kCk; ++t) {
                TokenVecs &tv = s_tok[t & 1];
                commit_token<kDoBf16>(p, tr, tv, tid);
                if (t + 1 < ts + kCk) fetch_token<kDoBf16>(p, t + 1, h, tid, tr);
                __syncthreads();
                forward_step(tv);
            }
        }
        __syncthreads();   // the token buffers change hands between phases

        // ---- reverse pass ----
        float4 G[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            G[i] = (p.dSf != nullptr)
                       ? *reinterpret_cast<const float4 *>(p.dSf + state_off + (warp + kWarps * i) * kD + c0)
                       : make_float4(0.f, 0.f, 0.f, 0.f);

        for (int j = nseg - 1; j >= 0; --j) {
            const int64_t ts = t0 + static_cast<int64_t>(j) * kCk;
            const int64_t te = (ts + kCk < t1) ? ts + kCk : t1;
            // rerun the segment from its checkpoint, keeping S_{t-1} of every step
            __syncthreads();
#pragma unroll
            for (int i = 0; i < kRows; ++i) s[i] = *ckpt_at(j, i);
            TokenRegs tr;
            if (ts + 1 < te) fetch_token<kDoBf16>(p, ts, h, tid, tr);
            for (int64_t t = ts; t < te; ++t) {
                float4 *sc = scratch + (t - ts) * kStateF4 + tid;
#pragma unroll
                for (int i = 0; i < kRows; ++i) sc[i * kThreads] = s[i];
                if (t + 1 < te) {   // the last step's S_t is not needed
                    TokenVecs &tv = s_tok[t & 1];
                    commit_token<kDoBf16>(p, tr, tv, tid);
                    if (t + 2 < te) fetch_token<kDoBf16>(p, t + 1, h, tid, tr);
                    __syncthreads();
                    forward_step(tv);
                }
            }
            __syncthreads();
            // reverse steps; the next step's token and S_{t-1} are requested
            // one step ahead (registers; cp.async into s_prev)
            auto prefetch_prev = [&](int64_t t) {
                const float4 *src = scratch + (t - ts) * kStateF4 + tid;
                float4 *dst = s_prev + (t & 1) * kStateF4 + tid;
#pragma unroll
                for (int i = 0; i < kRows; ++i) cp_async_16(dst + i * kThreads, src + i * kThreads);
                cp_async_commit();
            };
            fetch_token<kDoBf16>(p, te - 1, h, tid, tr);
            prefetch_prev(te - 1);
            for (int64_t t = te - 1; t >= ts; --t) {
                TokenVecs &tv = s_tok[t & 1];
                commit_token<kDoBf16>(p, tr, tv, tid);
                if (t - 1 >= ts) {
                    fetch_token<kDoBf16>(p, t - 1, h, tid, tr);
                    prefetch_prev(t - 1);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                const float4 *sp = s_prev + (t & 1) * kStateF4 + tid;
#pragma unroll
                for (int i = 0; i < kRows; ++i) s[i] = sp[i * kThreads];   // S_{t-1}
                __syncthreads();
                const float4 do4 = *reinterpret_cast<const float4 *>(&tv.dO[c0]);
                float4 wp = make_float4(0.f, 0.f, 0.f, 0.f), dup = wp;
#pragma unroll
                for (int i = 0; i < kRows; ++i) {
                    const int r = warp + kWarps * i;
                    s[i] = f4_scale(s[i], tv.d[r]);          // S'
                    G[i] = f4_fma(tv.q[r], do4, G[i]);        // G += (scale q) do^T
                    wp = f4_fma(tv.k[r], s[i], wp);
                    dup = f4_fma(tv.k[r], G[i], dup);
                }
                *reinterpret_cast<float4 *>(&s_red[0][warp][c0]) = wp;
                *reinterpret_cast<float4 *>(&s_red[1][warp][c0]) = dup;
                __syncthreads();
                if (tid < kD) {
                    float w = 0.f, du = 0.f;
#pragma unroll
                    for (int jj = 0; jj < kThreads / 32; ++jj) {
                        w += s_red[0][jj][tid];
                        du += s_red[1][jj][tid];
                    }
                    const float vw = tv.v[tid] - w;
                    const float u = tv.beta * vw;
                    s_u[tid] = u;
                    s_dw[tid] = -tv.beta * du;
                    p.dv[(t * H + h) * kD + tid] = tv.beta * du;
                    float pb = du * vw, pu = u * tv.dO[tid];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        pb += __shfl_xor_sync(0xffffffffu, pb, off);
                        pu += __shfl_xor_sync(0xffffffffu, pu, off);
                    }
                    if (lane == 0) {
                        s_sc[0][warp] = pb;
                        s_sc[1][warp] = pu;
                    }
                }
                __syncthreads();
                const float udo = s_sc[1][0] + s_sc[1][1] + s_sc[1][2] + s_sc[1][3];
                if (tid == 0) p.dbeta[t * H + h] = s_sc[0][0] + s_sc[0][1] + s_sc[0][2] + s_sc[0][3];
                const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[c0]);
                const float4 dw4 = *reinterpret_cast<const float4 *>(&s_dw[c0]);
                // per-row partial sums: 8 rows x 4 quantities = 32 slots
#pragma unroll
                for (int half = 0; half < kRows / 8; ++half) {
                    float v32[32];
#pragma unroll
                    for (int ii = 0; ii < 8; ++ii) {
                        const int i = 8 * half + ii;
                        v32[4 * ii + 0] = f4_dot(G[i], u4);     // (G u)_r
                        v32[4 * ii + 1] = f4_dot(s[i], dw4);    // (S' dw)_r
                        v32[4 * ii + 2] = f4_dot(s[i], do4);    // (S' do)_r
                        v32[4 * ii + 3] = f4_dot(G[i], s[i]);   // rowsum(G (.) S')_r
                    }
                    lane_transpose_sum32(v32, lane);
                    // lane l: row slot ii = l / 4, quantity l % 4
                    const float x = v32[0];
                    const float sdw = __shfl_sync(0xffffffffu, x, (lane & ~3) | 1);
                    const int r = warp + kWarps * (8 * half + (lane >> 2));
                    const int64_t oi = (t * H + h) * kD + r;
                    const int qn = lane & 3;
                    if (qn == 0) p.dk[oi] = x + sdw;
                    else if (qn == 2) p.dq[oi] = p.scale * (x + tv.k[r] * udo);
                    else if (qn == 3) p.dg[oi] = x + tv.k[r] * sdw;
                }
#pragma unroll
                for (int i = 0; i < kRows; ++i) {
                    const int r = warp + kWarps * i;
                    G[i] = f4_scale(f4_fma(tv.k[r], dw4, G[i]), tv.d[r]);
                }
            }
        }
        if (p.dS0 != nullptr) {
#pragma unroll
            for (int i = 0; i < kRows; ++i)
                *reinterpret_cast<float4 *>(p.dS0 + state_off + (warp + kWarps * i) * kD + c0) = G[i];
        }
    }
}

}  // namespace

// Workspace: [counter 256 B][checkpoints][scratch], each 256-byte aligned.
size_t backward_workspace_bytes(int64_t N, int B, int H, int ctas) {
    if (N < 0 || B < 1 || H < 1 || ctas < 1) return 0;
    const size_t state = static_cast<size_t>(kD) * kD * sizeof(float);
    const size_t slots = static_cast<size_t>(N / kCk) + static_cast<size_t>(B);
    return 256 + slots * H * state + static_cast<size_t>(ctas) * kCk * state;
}

int backward_ctas(int B, int H, int max_ctas) {
    const int64_t chains = static_cast<int64_t>(B) * H;
    return static_cast<int>(chains < max_ctas ? chains : max_ctas);
}

cudaError_t launch_backward(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                            const __nv_bfloat16 *v, const float *g, const float *beta,
                            const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
                            const float *S0, const void *dO, bool dO_bf16, const float *dSf,
                            float *dq, float *dk, float *dv, float *dg, float *dbeta, float *dS0,
                            void *workspace, int ctas, unsigned int *err, cudaStream_t s) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t state = static_cast<size_t>(kD) * kD * sizeof(float);
    const size_t slots = static_cast<size_t>(N / kCk) + static_cast<size_t>(B);
    BwdParams p;
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.cu_seqlens = cu_seqlens; p.B = B; p.N = N; p.H = H; p.scale = scale;
    p.S0 = S0; p.dO = dO; p.dO_bf16 = dO_bf16 ? 1 : 0; p.dSf = dSf;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dg = dg; p.dbeta = dbeta; p.dS0 = dS0;
    p.counter = reinterpret_cast<unsigned int *>(ws);
    p.ckpt = reinterpret_cast<float4 *>(ws + 256);
    p.scratch = reinterpret_cast<float4 *>(ws + 256 + slots * H * state);
    p.err = err;
    constexpr size_t kDynSmem = 2 * kStateF4 * sizeof(float4);   // 128 KB
    {
        cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(backward_kernel<true>),
                                            static_cast<int>(kDynSmem));
        if (e == cudaSuccess)
            e = ensure_dynamic_smem(reinterpret_cast<const void *>(backward_kernel<false>),
                                    static_cast<int>(kDynSmem));
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaMemsetAsync(ws, 0, 256, s);
    if (e != cudaSuccess) return e;
    if (dO_bf16)
        backward_kernel<true><<<ctas, kThreads, kDynSmem, s>>>(p);
    else
        backward_kernel<false><<<ctas, kThreads, kDynSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda

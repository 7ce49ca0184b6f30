// kda_shortconv.cu -- the KDA input pre-step: depthwise causal convolution of
// kernel size 4 on each of the q, k, v projection streams, SiLU, and an L2
// norm per (token, head) on q and k.
//
// The Kimi-K3 checkpoint holds q/k/v_conv1d.weight as fp32 [12288, 1, 4]
// (96 heads x 128 dims, kernel size 4; K3_ARTIFACT_AUDIT.md section 4.1, KDA
// tensor table).  For channel c and a token at position p of its sequence:
//
//   a[p, c] = sum_{j=0..3} w[c, j] * x[p - 3 + j, c]    (tap 3 = current token)
//   y = SiLU(a) = a * sigmoid(a)
//   q, k:  y / sqrt(sum over the head's 128 channels of y^2 + 1e-6);  v: y
//
// Positions before a sequence's first token read its carried conv state (the
// last three inputs of the previous segment, oldest first), zero without one.
//
// Data path: HBM-bound (12 bytes moved per channel-token over the three
// streams, ~12 instructions of arithmetic).  Lane l of a warp owns 8
// consecutive channels (one 16-byte load or store of bf16), so a warp covers
// two heads of 128 channels and the per-head norm is a reduction over 16 lanes
// by shuffles.  A warp walks 128 consecutive tokens in segments that stay
// inside one sequence, requesting 4 rows at a time; the rows two batches
// ahead are brought into L2 by bulk prefetches, so each load waits on L2
// rather than HBM (the taps and the three-token halo before the first row are
// loaded once per segment).  The arithmetic runs on packed pairs of channels
// (f32x2 instructions, each the IEEE operation on both halves).
#include "kda_f32x2.cuh"
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kTaps = 4;
constexpr int kHalo = kTaps - 1;
constexpr int kHeadDim = 128;
constexpr int kLaneCh = 8;                 // channels per lane
constexpr int kWarpCh = 32 * kLaneCh;      // 256 channels per warp
constexpr int kWarps = 8;
constexpr int kTT = 128;                   // tokens per warp
constexpr int kBatch = 4;                  // rows requested together
constexpr float kNormEps = 1e-6f;

static_assert(kWarpCh == 2 * kHeadDim, "a warp covers two heads; the norm reduces 16 lanes");

struct ConvStreams {
    const __nv_bfloat16 *x[3];   // [N, C] (prefill) or [B, C] (decode)
    const float *w[3];           // [C, 4]
    __nv_bfloat16 *y[3];         // like x
};

// Stream z's pointers, selected without indexing the parameter arrays by a
// runtime value (which would copy them to local memory).
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[3], int z) {
    return z == 0 ? a[0] : (z == 1 ? a[1] : a[2]);
}

constexpr int kLanePairs = kLaneCh / 2;   // channel pairs per lane
using Pair = uint64_t;                     // two fp32 values: channels 2i, 2i + 1

// The 8 bf16 channels of a 16-byte row piece as 4 packed pairs.
__device__ __forceinline__ void unpack_row(uint4 raw, Pair (&r)[kLanePairs]) {
    const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < kLanePairs; ++i)
        r[i] = f2(__uint_as_float(u[i] << 16), __uint_as_float(u[i] & 0xffff0000u));
}

__device__ __forceinline__ void load_row(const __nv_bfloat16 *p, Pair (&r)[kLanePairs]) {
    unpack_row(__ldcs(reinterpret_cast<const uint4 *>(p)), r);
}

__device__ __forceinline__ void store_row(__nv_bfloat16 *p, const Pair (&r)[kLanePairs]) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < kLanePairs; ++i) {
        const float2 v = f2_split(r[i]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
        u[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    __stcs(reinterpret_cast<uint4 *>(p), make_uint4(u[0], u[1], u[2], u[3]));
}

__device__ __forceinline__ void zero_row(Pair (&r)[kLanePairs]) {
#pragma unroll
    for (int i = 0; i < kLanePairs; ++i) r[i] = 0ull;
}

// w[i][j]: tap j of channels 2i and 2i + 1.
__device__ __forceinline__ void load_taps(const float *wz, int c, bool active,
                                          Pair (&w)[kLanePairs][kTaps]) {
    if (active) {
        const float4 *w4 = reinterpret_cast<const float4 *>(wz + static_cast<int64_t>(c) * kTaps);
#pragma unroll
        for (int i = 0; i < kLanePairs; ++i) {
            const float4 a = __ldg(w4 + 2 * i), b = __ldg(w4 + 2 * i + 1);
            w[i][0] = f2(a.x, b.x);
            w[i][1] = f2(a.y, b.y);
            w[i][2] = f2(a.z, b.z);
            w[i][3] = f2(a.w, b.w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < kLanePairs; ++i) w[i][0] = w[i][1] = w[i][2] = w[i][3] = 0ull;
    }
}

// 2^x and 1/x on the special-function unit.
__device__ __forceinline__ float sfu_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sfu_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One output row: the 4-tap convolution, SiLU (a / (1 + e^-a), with e^-a as
// 2^(-a log2 e)) and, for q and k, the head norm.  All 32 lanes must call it
// together (the norm shuffles within 16-lane halves).
__device__ __forceinline__ void conv_row(const Pair (&w)[kLanePairs][kTaps],
                                         const Pair (&win)[kHalo][kLanePairs],
                                         const Pair (&xt)[kLanePairs], bool norm,
                                         Pair (&out)[kLanePairs]) {
    const Pair nl2e = f2(-1.4426950408889634f, -1.4426950408889634f), one = f2(1.f, 1.f);
    Pair ss2 = 0ull;
#pragma unroll
    for (int i = 0; i < kLanePairs; ++i) {
        Pair a = f2_mul(w[i][0], win[0][i]);
        a = f2_fma(w[i][1], win[1][i], a);
        a = f2_fma(w[i][2], win[2][i], a);
        a = f2_fma(w[i][3], xt[i], a);
        const float2 t = f2_split(f2_mul(a, nl2e));
        const float2 d = f2_split(f2_add(one, f2(sfu_exp2(t.x), sfu_exp2(t.y))));
        const Pair y = f2_mul(a, f2(sfu_rcp(d.x), sfu_rcp(d.y)));
        out[i] = y;
        ss2 = f2_fma(y, y, ss2);
    }
    if (norm) {
        const float2 sp = f2_split(ss2);
        float ss = sp.x + sp.y;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss + kNormEps);
        const Pair inv2 = f2(inv, inv);
#pragma unroll
        for (int i = 0; i < kLanePairs; ++i) out[i] = f2_mul(out[i], inv2);
    }
}

// Carried state row `r` (0 = oldest) of sequence s for stream z: [B, 3, 3, C].
__device__ __forceinline__ int64_t state_index(int64_t s, int z, int r, int C, int c) {
    return ((s * 3 + z) * kHalo + r) * static_cast<int64_t>(C) + c;
}

// Prefill over a packed batch.  grid = (token tiles of kWarps * kTT tokens,
// channel groups of kWarpCh channels, 3 streams); warp w of a block takes
// tokens [tile * kWarps * kTT + w * kTT, + kTT) of the group's channels.
__global__ void __launch_bounds__(kWarps * 32, 2) short_conv_kernel(
    ConvStreams io, const int32_t *__restrict__ cu, int B, int64_t N, int C,
    const __nv_bfloat16 *__restrict__ state_in, __nv_bfloat16 *__restrict__ state_out,
    unsigned int *err) {
    const int z = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = blockIdx.y * kWarpCh + lane * kLaneCh;
    const bool active = c < C;
    const bool norm = z < 2;
    const __nv_bfloat16 *__restrict__ x = pick(io.x, z);
    __nv_bfloat16 *__restrict__ y = pick(io.y, z);

    if (cu != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && z == 0 && threadIdx.x == 0) {
        bool ok = cu[0] == 0 && cu[B] == N;
        for (int s = 0; s < B && ok; ++s) ok = cu[s] <= cu[s + 1];
        if (!ok) record_device_error(err, kDevInvalidArg);
    }

    const int64_t t_begin = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * kTT;
    const int64_t t_end = min(t_begin + kTT, N);
    auto seq_end = [&](int s) -> int64_t { return cu == nullptr ? N : cu[s + 1]; };
    auto seq_start = [&](int s) -> int64_t { return cu == nullptr ? 0 : cu[s]; };

    // State of sequence s passes through unchanged (an empty sequence).
    auto pass_state = [&](int s) {
        if (state_out == nullptr || !active) return;
#pragma unroll
        for (int r = 0; r < kHalo; ++r) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (state_in != nullptr)
                v = *reinterpret_cast<const uint4 *>(state_in + state_index(s, z, r, C, c));
            *reinterpret_cast<uint4 *>(state_out + state_index(s, z, r, C, c)) = v;
        }
    };
    // Empty sequences in front of the first token belong to the first warp.
    if (t_begin == 0)
        for (int s = 0; s < B && seq_end(s) <= 0; ++s) pass_state(s);
    if (t_begin >= t_end) return;

    Pair w[kLanePairs][kTaps];
    load_taps(pick(io.w, z), c, active, w);

    // The sequence holding t_begin: the first s with cu[s + 1] > t_begin.
    int s = 0;
    if (cu != nullptr) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (cu[mid + 1] > t_begin) hi = mid; else lo = mid + 1;
        }
        s = lo;
    }

    // Window rows 0..2 hold positions t-3, t-2, t-1 of the current sequence.
    Pair win[kHalo][kLanePairs];
    auto load_window = [&](int64_t t, int seq) {
        const int64_t start = seq_start(seq);
#pragma unroll
        for (int r = 0; r < kHalo; ++r) {
            const int64_t pos = t - kHalo + r;
            if (!active) {
                zero_row(win[r]);
            } else if (pos >= start && pos >= 0) {
                load_row(x + pos * C + c, win[r]);
            } else {
                const int64_t sr = pos - start + kHalo;   // 0..2 for pos in [start-3, start)
                if (state_in != nullptr && sr >= 0 && sr < kHalo)
                    load_row(state_in + state_index(seq, z, static_cast<int>(sr), C, c), win[r]);
                else
                    zero_row(win[r]);
            }
        }
    };
    // The warp's rows of this channel group (512 bytes at most) are brought
    // into L2 ahead of their loads by bulk prefetches, one row per lane.
    const int gc0 = blockIdx.y * kWarpCh;
    const uint32_t row_bytes = static_cast<uint32_t>(min(kWarpCh, C - gc0)) * 2u;
    auto prefetch_row = [&](int64_t t) {
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(x + t * C + gc0), "r"(row_bytes)
                     : "memory");
    };

    // The warp's tokens in segments that lie inside one sequence: each segment
    // loads its window once, then runs batches of kBatch rows with every row of
    // a batch requested before the first is used and no per-row test beyond
    // the segment bound; rows two batches ahead are prefetched into L2.
    for (int64_t a = t_begin; a < t_end;) {
        while (s < B - 1 && seq_end(s) <= a) ++s;
        const int64_t send = seq_end(s);
        const int64_t b = min(t_end, send);
        if (lane < 2 * kBatch && a + lane < b) prefetch_row(a + lane);  // the first two batches
        load_window(a, s);
        for (int64_t tb = a; tb < b; tb += kBatch) {
            if (lane < kBatch && tb + 2 * kBatch + lane < b) prefetch_row(tb + 2 * kBatch + lane);
            uint4 raw[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                raw[j] = (active && tb + j < b)
                             ? __ldcs(reinterpret_cast<const uint4 *>(x + (tb + j) * C + c))
                             : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                Pair xt[kLanePairs], out[kLanePairs];
                unpack_row(raw[j], xt);
                conv_row(w, win, xt, norm, out);
                if (active && tb + j < b) store_row(y + (tb + j) * C + c, out);
                // (rows past the segment only shift the window, which the
                // next segment reloads)
#pragma unroll
                for (int i = 0; i < kLanePairs; ++i) {
                    win[0][i] = win[1][i];
                    win[1][i] = win[2][i];
                    win[2][i] = xt[i];
                }
            }
        }
        if (b == send) {  // the last token of sequence s: its carried state
            if (state_out != nullptr && active) {
                load_window(b, s);
#pragma unroll
                for (int r = 0; r < kHalo; ++r) store_row(state_out + state_index(s, z, r, C, c), win[r]);
            }
            for (int s2 = s + 1; s2 < B && seq_end(s2) <= send; ++s2) pass_state(s2);
        }
        a = b;
    }
}

// One token per sequence, state updated in place in a pool addressed by slot.
// grid = (channel groups of kWarps * kWarpCh, B, 3 streams).
__global__ void __launch_bounds__(kWarps * 32) short_conv_step_kernel(
    ConvStreams io, __nv_bfloat16 *__restrict__ pool, const int32_t *__restrict__ slots,
    int num_slots, int C, unsigned int *err) {
    const int z = blockIdx.z;
    const int64_t b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = (blockIdx.x * kWarps + warp) * kWarpCh + lane * kLaneCh;
    const bool active = c < C;
    const int sl = slots != nullptr ? slots[b] : static_cast<int>(b);
    __nv_bfloat16 *__restrict__ y = pick(io.y, z) + b * C + c;
    if (sl < 0 || sl >= num_slots) {
        if (sl >= num_slots && threadIdx.x == 0 && blockIdx.x == 0 && z == 0)
            record_device_error(err, kDevInvalidArg);
        Pair zero[kLanePairs];
        zero_row(zero);
        if (active) store_row(y, zero);
        return;
    }
    Pair w[kLanePairs][kTaps], win[kHalo][kLanePairs], xt[kLanePairs], out[kLanePairs];
    load_taps(pick(io.w, z), c, active, w);
    if (active) {
#pragma unroll
        for (int r = 0; r < kHalo; ++r) load_row(pool + state_index(sl, z, r, C, c), win[r]);
        load_row(pick(io.x, z) + b * C + c, xt);
    } else {
#pragma unroll
        for (int r = 0; r < kHalo; ++r) zero_row(win[r]);
        zero_row(xt);
    }
    conv_row(w, win, xt, z < 2, out);
    if (active) {
        store_row(y, out);
        store_row(pool + state_index(sl, z, 0, C, c), win[1]);
        store_row(pool + state_index(sl, z, 1, C, c), win[2]);
        store_row(pool + state_index(sl, z, 2, C, c), xt);
    }
}

}  // namespace

cudaError_t launch_short_conv(const __nv_bfloat16 *const x[3], const float *const w[3],
                              __nv_bfloat16 *const y[3], const int32_t *cu_seqlens, int B,
                              int64_t N, int C, const __nv_bfloat16 *state_in,
                              __nv_bfloat16 *state_out, unsigned int *err, cudaStream_t s) {
    ConvStreams io;
    for (int i = 0; i < 3; ++i) {
        io.x[i] = x[i];
        io.w[i] = w[i];
        io.y[i] = y[i];
    }
    const int64_t tiles = (N + kWarps * kTT - 1) / (kWarps * kTT);
    const dim3 grid(static_cast<unsigned>(tiles > 0 ? tiles : 1),
                    static_cast<unsigned>((C + kWarpCh - 1) / kWarpCh), 3);
    short_conv_kernel<<<grid, kWarps * 32, 0, s>>>(io, cu_seqlens, B, N, C, state_in, state_out,
                                                   err);
    return cudaGetLastError();
}

cudaError_t launch_short_conv_step(const __nv_bfloat16 *const x[3], const float *const w[3],
                                   __nv_bfloat16 *const y[3], __nv_bfloat16 *pool,
                                   const int32_t *slots, int num_slots, int B, int C,
                                   unsigned int *err, cudaStream_t s) {
    ConvStreams io;
    for (int i = 0; i < 3; ++i) {
        io.x[i] = x[i];
        io.w[i] = w[i];
        io.y[i] = y[i];
    }
    const int per_block = kWarps * kWarpCh;
    const dim3 grid(static_cast<unsigned>((C + per_block - 1) / per_block),
                    static_cast<unsigned>(B), 3);
    short_conv_step_kernel<<<grid, kWarps * 32, 0, s>>>(io, pool, slots, num_slots, C, err);
    return cudaGetLastError();
}

}  // namespace kda

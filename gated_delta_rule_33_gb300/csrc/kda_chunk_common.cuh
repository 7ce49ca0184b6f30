// kda_chunk_common.cuh -- device and host helpers of the chunked prefill
// kernel (kda_chunk.cu): chunk constants, the UT-inverse building blocks, the
// T beta operand stores, bounded CTA waits and TMA tensor maps.  Not part of
// the public ABI.
#pragma once

#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_f32x2.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace chunk {

using namespace sm100;

constexpr int kC = 64;              // chunk length
constexpr int kD = 128;             // d_k = d_v
// Largest per-channel decay -sum(g) of one chunk that the midpoint-referenced
// factors represent (every factor within e^{+-80}); a chunk that would exceed
// it in some channel is shortened.  A single token whose own decay exceeds it
// forms a chunk of one token with its decay taken as this value: e^{-160}
// underflows fp32 exactly as any larger decay does.
constexpr float kMaxChunkDecay = 160.f;
// Bound of every mbarrier wait (polls of try_wait, each itself a bounded wait).
constexpr uint32_t kMaxPolls = 1u << 20;
// The tf32 T beta tile lives in rows 128..191 of a 192-row K-major tile (the
// chunk kernel's [Khat^T ; T beta -> A_qk] B operand), so its rows are
// addressed with this offset and row count.
constexpr uint32_t kTbRow0 = 128;
constexpr uint32_t kTbRows = 192;

// The 1024-byte-aligned base of the dynamic shared memory (the launch asks for
// 1024 bytes more than it uses).  It is formed by indexing the shared array,
// not through an integer round trip, so that accesses derived from it stay
// shared-memory accesses instead of generic ones.
__device__ __forceinline__ uint8_t *smem_base() {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    return smem_raw + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ float bf(const uint8_t *base, uint32_t off) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(base + off));
}

__device__ __forceinline__ void st_f32(uint8_t *base, uint32_t off, float x) {
    *reinterpret_cast<float *>(base + off) = x;
}

// log2(1 + e) of both halves of a packed pair, e in [0, 1], as e P(e) with P
// the degree-7 Chebyshev interpolant of log2(1 + e) / e on [0, 1] in monomial
// form (coefficients from gen_log2p1_poly.py; relative error of this fp32
// evaluation below 4e-7).  It runs on the FMA pipe, which the operand build
// leaves less loaded than the special-function unit.
__device__ __forceinline__ uint64_t log2_1p_unit2(uint64_t e) {
    uint64_t p = f2(-0.0120770205f, -0.0120770205f);
    p = f2_fma(p, e, f2(0.0627484322f, 0.0627484322f));
    p = f2_fma(p, e, f2(-0.154152006f, -0.154152006f));
    p = f2_fma(p, e, f2(0.255176336f, 0.255176336f));
    p = f2_fma(p, e, f2(-0.353096366f, -0.353096366f));
    p = f2_fma(p, e, f2(0.480012447f, 0.480012447f));
    p = f2_fma(p, e, f2(-0.721306741f, -0.721306741f));
    p = f2_fma(p, e, f2(1.44269478f, 1.44269478f));
    return f2_mul(p, e);
}

// Barrier of the 128 threads (warps 0-3) that compute the UT inverse while
// the other warps run the state pass.
__device__ __forceinline__ void inverse_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Named barriers between the inverse warps (which arrive) and the warp that
// issues the W' and U-tilde products (which waits); n counts every thread of
// both sides.
__device__ __forceinline__ void named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
constexpr int kBarDiag = 2, kBarLevel1 = 3, kBarLevel2 = 4;
// Between the inverse warps (which arrive) and the forward's T beta writers
// (which wait): T of the diagonal blocks, then of level 1, is in place.
constexpr int kBarDiagT = 5, kBarLevel1T = 6;
// Between the forward's level-2 warps 0 (arrives) and 1 (waits): Y rows 0-15.
constexpr int kBarLevel2Y = 7;

// 2^x with the special-function unit (inputs here lie within +-116).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Thread 0 waits (bounded, `polls` polls) on an mbarrier phase, then the
// whole CTA meets at a barrier; a time-out raises the CTA abort flag and
// records the error.  Returns false (in every thread, through the barrier's
// AND reduction) when this wait ran out.  Only one thread polls, so the other warps do not
// compete with the tensor core for shared-memory bandwidth while they wait.
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity, int *abort_flag,
                                         unsigned int *err, int tid, uint32_t polls) {
    bool ok = true;
    if (tid == 0 && !mbar_wait_bounded(bar, parity, polls)) {
        *abort_flag = 1;
        record_device_error(err, kDevTimeout);
        ok = false;
    }
    ok = __syncthreads_and(ok);
    tc_fence_after();
    return ok;
}

// T beta[r][s] = T[r][s] beta_s as a tf32 operand tile and as bf16 high + low
// tiles (all K-major [r][s], 128-byte swizzle), four adjacent s at a time.
__device__ __forceinline__ void store_tbeta4(uint8_t *tb, uint8_t *tb16, int r, int s4, float4 t,
                                             const float *beta) {
    const float x0 = t.x * beta[s4], x1 = t.y * beta[s4 + 1];
    const float x2 = t.z * beta[s4 + 2], x3 = t.w * beta[s4 + 3];
    *reinterpret_cast<float4 *>(tb + sw128_offset(kTbRow0 + r, s4, kTbRows, 4)) =
        make_float4(to_tf32(x0), to_tf32(x1), to_tf32(x2), to_tf32(x3));
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(x0, x1), h23 = __floats2bfloat162_rn(x2, x3);
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(x0 - f01.x, x1 - f01.y);
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(x2 - f23.x, x3 - f23.y);
    uint2 hv, lv;
    hv.x = *reinterpret_cast<const uint32_t *>(&h01); hv.y = *reinterpret_cast<const uint32_t *>(&h23);
    lv.x = *reinterpret_cast<const uint32_t *>(&l01); lv.y = *reinterpret_cast<const uint32_t *>(&l23);
    *reinterpret_cast<uint2 *>(tb16 + sw128_offset(r, s4, 64, 2)) = hv;
    *reinterpret_cast<uint2 *>(tb16 + 8192 + sw128_offset(r, s4, 64, 2)) = lv;
}

// Where the UT inverse writes its result, as each block of T is final: the
// forward kernel's T beta operand tiles in shared memory.  (The chunked
// backward supplies its own policy with the same two members.)
struct TbetaTiles {
    uint8_t *tb, *tb16;
    const float *beta;
    // one element T[r][s]
    __device__ __forceinline__ void one(int r, int s, float t) const {
        const float xb = t * beta[s];
        st_f32(tb, sw128_offset(kTbRow0 + r, s, kTbRows, 4), to_tf32(xb));
        const __nv_bfloat16 hi = __float2bfloat16_rn(xb);
        const __nv_bfloat16 lo = __float2bfloat16_rn(xb - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat16 *>(tb16 + sw128_offset(r, s, 64, 2)) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(tb16 + 8192 + sw128_offset(r, s, 64, 2)) = lo;
    }
    // T[r][s4 .. s4 + 3]
    __device__ __forceinline__ void four(int r, int s4, float4 t) const {
        store_tbeta4(tb, tb16, r, s4, t, beta);
    }
    // column j of a diagonal block: T[r0 + i][j] = x[i], i < 16
    __device__ __forceinline__ void col(int r0, int j, const float (&x)[16]) const {
        const float bj = beta[j];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float xb = x[i] * bj;
            st_f32(tb, sw128_offset(kTbRow0 + r0 + i, j, kTbRows, 4), to_tf32(xb));
            const __nv_bfloat16 hi = __float2bfloat16_rn(xb);
            const __nv_bfloat16 lo = __float2bfloat16_rn(xb - __bfloat162float(hi));
            *reinterpret_cast<__nv_bfloat16 *>(tb16 + sw128_offset(r0 + i, j, 64, 2)) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(tb16 + 8192 + sw128_offset(r0 + i, j, 64, 2)) = lo;
        }
    }
};

// An output policy that keeps every block of T in the row-major T itself: the
// diagonal solve already writes its columns there, and four() stores the
// blocks of the two levels (T_32 and the lower-left 32 x 32 block too), so
// that T is complete (fp32, row-major, zero above the diagonal) wherever a
// level ends.
struct TRowMajor {
    float *t;
    __device__ __forceinline__ void col(int, int, const float (&)[16]) const {}  // already in T
    __device__ __forceinline__ void four(int r, int s4, float4 x) const {
        *reinterpret_cast<float4 *>(t + r * 64 + s4) = x;
    }
};

// ---- T = (I + A)^{-1} for the strictly lower-triangular 64 x 64 A_kk ----
// Layouts (fp32, shared memory):
//   At     A column-major, At[s * 64 + r] = A[r][s] (zero for s >= r)
//   T      row-major [64][64]; the blocks T_00, T_11, T_22 and T_10 are written
//   Tdiag  the diagonal blocks column-major, Tdiag[b * 256 + s * 16 + r] = T_bb[r][s]
//   T32c   T_32 column-major, T32c[s * 16 + r]
//   P      scratch: level 1 two 16 x 16 row-major products; level 2 Y (32 x 32,
//          row-major with the float4 group index XOR-ed by row % 8)
// Products are register-blocked 2 rows x 4 columns per thread: per step one
// 8-byte load of two rows of a column-major factor and one 16-byte load of a
// row of the other feed eight FMAs.

// acc{0,1} += sum over s < n of (Ac[s * ac_stride], Ac[s * ac_stride + 1]) x
// B[s * b_stride .. + 3]: rows r0, r0 + 1 of a column-major left factor times
// four columns of a row-major right factor.
// Accumulators as packed pairs: {acc0.xy, acc0.zw, acc1.xy, acc1.zw}.
struct Acc2x4 {
    uint64_t v[4];
    __device__ __forceinline__ Acc2x4() {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = 0ull;  // +0.0f in both halves
    }
    // rows (a.x, a.y) times the four columns b
    __device__ __forceinline__ void step(float2 a, float4 b) {
        const uint64_t ax = f2(a.x, a.x), ay = f2(a.y, a.y);
        const uint64_t b01 = f2(b.x, b.y), b23 = f2(b.z, b.w);
        v[0] = f2_fma(ax, b01, v[0]);
        v[1] = f2_fma(ax, b23, v[1]);
        v[2] = f2_fma(ay, b01, v[2]);
        v[3] = f2_fma(ay, b23, v[3]);
    }
    // row 0 or 1, negated, as a float4
    __device__ __forceinline__ float4 neg_row(int i) const {
        const float2 lo = f2_split(v[2 * i]), hi = f2_split(v[2 * i + 1]);
        return make_float4(-lo.x, -lo.y, -hi.x, -hi.y);
    }
    __device__ __forceinline__ float4 row(int i) const {
        const float2 lo = f2_split(v[2 * i]), hi = f2_split(v[2 * i + 1]);
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
};

// kU: unroll factor (a kernel short of instruction cache unrolls less)
template <int kN, int kU = kN>
__device__ __forceinline__ void gemm_2x4(Acc2x4 &acc, const float *Ac, int ac_stride,
                                         const float *B, int b_stride) {
#pragma unroll kU
    for (int s = 0; s < kN; ++s)
        acc.step(*reinterpret_cast<const float2 *>(Ac + s * ac_stride),
                 *reinterpret_cast<const float4 *>(B + s * b_stride));
}

// Y index of (row r, columns c .. c + 3), c a multiple of 4
__device__ __forceinline__ int y_idx(int r, int c) { return r * 32 + (((c >> 2) ^ (r & 7)) << 2); }

// The four 16x16 diagonal blocks (warps 0-1: block tid / 16, column j = tid % 16)
// by forward substitution in its right-looking form (once x_s is final,
// subtract A[r][s] x_s from every later row): 15 steps of independent FMAs,
// each reading one block column of At as four 16-byte loads, the next column
// loaded while the current one is applied.  Writes T (row-major), Tdiag and
// the T beta operand tiles.
template <class Out>
__device__ __forceinline__ void ut_diag_solve(const float *At, float *T, float *Tdiag, const Out &out,
                                              int tid) {
    const int bb = tid >> 4, j = tid & 15, base = bb * 16;
    const float *Ab = At + base * 64 + base;   // Ab[s * 64 + r] = A_bb[r][s]
    // x as packed row pairs; a step updates whole pairs from the one holding
    // row s + 1 on (when that is row s's pair, row s gets A_bb[s][s] x_s = 0)
    uint64_t xp[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) xp[q] = f2((2 * q == j) ? 1.f : 0.f, (2 * q + 1 == j) ? 1.f : 0.f);
    float4 c[4], n[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = *reinterpret_cast<const float4 *>(Ab + 4 * q);
#pragma unroll
    for (int s = 0; s < 15; ++s) {
        if (s < 14) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                n[q] = *reinterpret_cast<const float4 *>(Ab + (s + 1) * 64 + 4 * q);
        }
        const uint64_t colp[8] = {f2(c[0].x, c[0].y), f2(c[0].z, c[0].w), f2(c[1].x, c[1].y),
                                  f2(c[1].z, c[1].w), f2(c[2].x, c[2].y), f2(c[2].z, c[2].w),
                                  f2(c[3].x, c[3].y), f2(c[3].z, c[3].w)};
        const float2 ps = f2_split(xp[s >> 1]);
        const float nxs = -((s & 1) ? ps.y : ps.x);
        const uint64_t nx2 = f2(nxs, nxs);
#pragma unroll
        for (int q = (s + 1) >> 1; q < 8; ++q) xp[q] = f2_fma(colp[q], nx2, xp[q]);
        if (s < 14) {
#pragma unroll
            for (int q = 0; q < 4; ++q) c[q] = n[q];
        }
    }
    float x[16];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float2 v = f2_split(xp[q]);
        x[2 * q] = v.x;
        x[2 * q + 1] = v.y;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) T[(base + r) * 64 + base + j] = x[r];
    float *Td = Tdiag + bb * 256 + j * 16;  // column j of T_bb
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        *reinterpret_cast<float4 *>(Td + 4 * q4) =
            make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
    // T (beta) of the diagonal block, column j (16 rows)
    out.col(base, base + j, x);
}

// Level 1 (warps 0-1, warp t / 2 for target t = 0, 2; it solved T_tt and
// T_{t+1,t+1} itself): T_{t+1,t} = -T_{t+1,t+1} (A_{t+1,t} T_tt).  Lane l owns
// rows r0 = 2 (l / 4), r0 + 1 and columns c0 = 4 (l % 4) .. + 3 of the block.
// T_10 goes to T (row-major, part of T_top in level 2), T_32 to T32c.
template <class Out, int kU = 32>
__device__ __forceinline__ void ut_level1(const float *At, const float *T, const float *Tdiag,
                                          float *P, float *Tw, float *T32c, const Out &out,
                                          int tid) {
    const int t = 2 * (tid >> 5), l = tid & 31, r0 = 2 * (l >> 2), c0 = 4 * (l & 3);
    float *Pt = P + (t >> 1) * 256;
    Acc2x4 a;
    // P_t = A_{t+1,t} T_tt (T_tt is zero above its diagonal)
    gemm_2x4<16, kU>(a, At + (16 * t) * 64 + 16 * (t + 1) + r0, 64, T + (16 * t) * 64 + 16 * t + c0, 64);
    *reinterpret_cast<float4 *>(Pt + r0 * 16 + c0) = a.row(0);
    *reinterpret_cast<float4 *>(Pt + (r0 + 1) * 16 + c0) = a.row(1);
    __syncwarp();
    Acc2x4 b;
    gemm_2x4<16, kU>(b, Tdiag + (t + 1) * 256 + r0, 16, Pt + c0, 16);
    const float4 x0 = b.neg_row(0), x1 = b.neg_row(1);
    if (t == 0) {
        *reinterpret_cast<float4 *>(Tw + (16 + r0) * 64 + c0) = x0;
        *reinterpret_cast<float4 *>(Tw + (17 + r0) * 64 + c0) = x1;
    } else {
        *reinterpret_cast<float2 *>(T32c + (c0 + 0) * 16 + r0) = make_float2(x0.x, x1.x);
        *reinterpret_cast<float2 *>(T32c + (c0 + 1) * 16 + r0) = make_float2(x0.y, x1.y);
        *reinterpret_cast<float2 *>(T32c + (c0 + 2) * 16 + r0) = make_float2(x0.z, x1.z);
        *reinterpret_cast<float2 *>(T32c + (c0 + 3) * 16 + r0) = make_float2(x0.w, x1.w);
    }
    out.four(16 * (t + 1) + r0, 16 * t + c0, x0);
    out.four(16 * (t + 1) + r0 + 1, 16 * t + c0, x1);
}

// Level 2 (warps 0-3): the lower-left 32x32 block X = T[32:64, 0:32] =
// -T_bot (A_bl T_top), T_top = T[0:32, 0:32] and T_bot = T[32:64, 32:64] block
// lower triangular (complete after level 1), A_bl = A[32:64, 0:32].  Warp w
// owns rows 16 (w % 2) .. + 15 and columns 16 (w / 2) .. + 15 of Y and X, so
// every triangular bound is warp-uniform; lane l owns rows r0 = 16 (w % 2) +
// 2 (l / 4), r0 + 1 and columns c0 = 16 (w / 2) + 4 (l % 4) .. + 3.
template <class Out, int kU = 32>
__device__ __forceinline__ void ut_level2(const float *At, const float *T, const float *Tdiag,
                                          const float *T32c, float *Y, const Out &out, int tid) {
    const int w = tid >> 5, l = tid & 31, rh = w & 1, cb = w >> 1;
    const int r0 = 16 * rh + 2 * (l >> 2), c0 = 16 * cb + 4 * (l & 3);
    Acc2x4 a;
    // Y = A_bl T_top: T_top[s][c] is zero for s < 16 * block(c)
    if (cb == 0)
        gemm_2x4<32, kU>(a, At + 32 + r0, 64, T + c0, 64);
    else
        gemm_2x4<16, kU>(a, At + 16 * 64 + 32 + r0, 64, T + 16 * 64 + c0, 64);
    *reinterpret_cast<float4 *>(Y + y_idx(r0, c0)) = a.row(0);
    *reinterpret_cast<float4 *>(Y + y_idx(r0 + 1, c0)) = a.row(1);
    inverse_sync();
    // X = -T_bot Y: T_bot[r][s] is zero for s >= 16 * (block(r) + 1)
    Acc2x4 b;
#pragma unroll kU
    for (int s = 0; s < 16; ++s)
        b.step(rh == 0 ? *reinterpret_cast<const float2 *>(Tdiag + 2 * 256 + s * 16 + r0)
                       : *reinterpret_cast<const float2 *>(T32c + s * 16 + r0 - 16),
               *reinterpret_cast<const float4 *>(Y + y_idx(s, c0)));
    if (rh == 1) {
#pragma unroll kU
        for (int s = 16; s < 32; ++s)
            b.step(*reinterpret_cast<const float2 *>(Tdiag + 3 * 256 + (s - 16) * 16 + r0 - 16),
                   *reinterpret_cast<const float4 *>(Y + y_idx(s, c0)));
    }
    out.four(32 + r0, c0, b.neg_row(0));
    out.four(33 + r0, c0, b.neg_row(1));
}

// ---- host: TMA tensor maps -------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// Tensor map of a [N, H, 128] tensor (bf16, or fp32 when `f32`) with a
// (box_x, 1, 64) box.
inline bool make_map(CUtensorMap *map, const void *base, int64_t N, int H, uint32_t box_x, bool swizzle,
              bool f32 = false) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(N)};
    const cuuint64_t esize = f32 ? 4 : 2;
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * esize,
                                   static_cast<cuuint64_t>(H) * kD * esize};
    const cuuint32_t box[3] = {box_x, 1, static_cast<cuuint32_t>(kC)};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void *>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace chunk
}  // namespace kda

// kda_chunk_common.cuh -- device and host helpers of the chunked prefill
// kernel (kda_chunk.cu): chunk constants, the UT-inverse building blocks, the
// T beta operand stores, bounded CTA waits and TMA tensor maps.  Not part of
// the public ABI.
#pragma once

#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace chunk {

using namespace sm100;

constexpr int kC = 64;              // chunk length
constexpr int kD = 128;             // d_k = d_v
constexpr float kMaxDecay = 160.f;  // largest per-channel chunk decay represented
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

// A_kk is stored row-major with its column index XOR-ed by (row % 32), so that
// one thread per row can write it without shared-memory bank conflicts.
__device__ __forceinline__ int akk_idx(int r, int s) { return r * 64 + (s ^ (r & 31)); }

// log2(1 + e) for e in [0, 1], as e P(e) with P the degree-7 Chebyshev
// interpolant of log2(1 + e) / e on [0, 1] in monomial form (coefficients from
// gen_log2p1_poly.py; relative error of this fp32 evaluation below 4e-7).  It
// runs on the FMA pipe, which the operand build leaves less loaded than the
// special-function unit.
__device__ __forceinline__ float log2_1p_unit(float e) {
    float p = -0.0120770205f;
    p = __fmaf_rn(p, e, 0.0627484322f);
    p = __fmaf_rn(p, e, -0.154152006f);
    p = __fmaf_rn(p, e, 0.255176336f);
    p = __fmaf_rn(p, e, -0.353096366f);
    p = __fmaf_rn(p, e, 0.480012447f);
    p = __fmaf_rn(p, e, -0.721306741f);
    p = __fmaf_rn(p, e, 1.44269478f);
    return p * e;
}

// Barrier of the 256 threads (warps 0-7) that compute the UT inverse while
// warps 8-15 run the state pass.
__device__ __forceinline__ void inverse_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// 2^x with the special-function unit (inputs here lie within +-116).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Thread 0 waits (bounded) on an mbarrier phase, then the whole CTA meets at a
// barrier; a time-out raises the CTA abort flag, which every thread reads
// after the barrier.  Only one thread polls, so the other warps do not compete
// with the tensor core for shared-memory bandwidth while they wait.
__device__ __forceinline__ void cta_wait(uint64_t *bar, uint32_t parity, int *abort_flag,
                                         unsigned int *err, int tid) {
    if (tid == 0 && !mbar_wait_bounded(bar, parity, kMaxPolls)) {
        *abort_flag = 1;
        record_device_error(err, kDevTimeout);
    }
    __syncthreads();
    tc_fence_after();
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

// Level 1 of the off-diagonal blocks: T_10 and T_32 (the block sub-diagonal
// inside each 32x32 half), T_{t+1,t} = -T_{t+1,t+1} A_{t+1,t} T_tt, t = 0, 2.
// 64 threads per target: 16 rows x 4 column quads.  T_10 goes to T (row-major,
// read by level 2 as part of T_top); T_32 goes column-major to T32c (read by
// level 2 as part of T_bot, a row per thread).
__device__ __forceinline__ void ut_level1(const float *A, const float *Tdiag, float *T, float *P,
                                          float *T32c, uint8_t *tb, uint8_t *tb16,
                                          const float *beta, int tid) {
    if (tid < 128) {
        const int t = 2 * (tid >> 6), r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
        const int arow = 16 * (t + 1) + r;
        const float *Ar = A + arow * 64;
        const int sw = arow & 31;
        const float *Tb = T + (16 * t) * 64 + 16 * t + c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const float a = Ar[(16 * t + s) ^ sw];
            const float4 tv = *reinterpret_cast<const float4 *>(Tb + s * 64);
            acc.x += a * tv.x; acc.y += a * tv.y; acc.z += a * tv.z; acc.w += a * tv.w;
        }
        *reinterpret_cast<float4 *>(&P[((tid >> 6) << 8) + (r << 4) + c4]) = acc;
    }
    inverse_sync();
    if (tid < 128) {
        const int t = 2 * (tid >> 6), r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
        const float *Ti = Tdiag + (t + 1) * 256 + r;   // T_{t+1,t+1}[r][s] at Ti[16 s]
        const float *Pb = P + ((tid >> 6) << 8) + c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const float4 pv = *reinterpret_cast<const float4 *>(Pb + s * 16);
            const float a = Ti[16 * s];   // zero above the diagonal
            acc.x += a * pv.x; acc.y += a * pv.y; acc.z += a * pv.z; acc.w += a * pv.w;
        }
        const float4 tij = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        if (t == 0) {
            *reinterpret_cast<float4 *>(&T[(16 + r) * 64 + c4]) = tij;
        } else {
            T32c[c4 * 16 + r] = tij.x;
            T32c[(c4 + 1) * 16 + r] = tij.y;
            T32c[(c4 + 2) * 16 + r] = tij.z;
            T32c[(c4 + 3) * 16 + r] = tij.w;
        }
        store_tbeta4(tb, tb16, 16 * (t + 1) + r, 16 * t + c4, tij, beta);
    }
    inverse_sync();
}

// Level 2: the lower-left 32x32 block X = T[32:64, 0:32] = -T_bot (A_bl T_top),
// with T_top = T[0:32, 0:32], T_bot = T[32:64, 32:64] (both block lower
// triangular, complete after level 1) and A_bl = A[32:64, 0:32].
// 256 threads, 32 rows x 8 column quads; every warp's rows and columns fall in
// one 16-block, so the triangular bounds are compile-time per branch.
// Y = A_bl T_top goes through P.  T_bot is read from its column-major blocks
// (T_22 and T_33 in Tdiag, T_32 in T32c): the eight rows a warp covers then
// fall in eight banks (a row-major read with stride 64 would hit one).
template <int S0>
__device__ __forceinline__ float4 level2_y(const float *Ar, int sw, const float *T, int c) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = S0; s < 32; ++s) {
        const float a = Ar[s ^ sw];
        const float4 tv = *reinterpret_cast<const float4 *>(&T[s * 64 + c]);
        acc.x += a * tv.x; acc.y += a * tv.y; acc.z += a * tv.z; acc.w += a * tv.w;
    }
    return acc;
}

// acc += sum over 16 s of Tc[16 s] * P[s0 + s][c .. c + 3] (Tc: one row of a
// column-major 16x16 block)
__device__ __forceinline__ void level2_x16(float4 &acc, const float *Tc, const float *P, int s0,
                                           int c) {
#pragma unroll
    for (int s = 0; s < 16; ++s) {
        const float a = Tc[16 * s];
        const float4 yv = *reinterpret_cast<const float4 *>(&P[(s0 + s) * 32 + c]);
        acc.x += a * yv.x; acc.y += a * yv.y; acc.z += a * yv.z; acc.w += a * yv.w;
    }
}

__device__ __forceinline__ void ut_level2(const float *A, const float *T, const float *Tdiag,
                                          const float *T32c, float *P, uint8_t *tb,
                                          uint8_t *tb16, const float *beta, int tid) {
    // task: column block cb = tid / 128, row r = (tid / 4) % 32, quad q = tid % 4
    const int cb = tid >> 7, r = (tid >> 2) & 31, c = 16 * cb + 4 * (tid & 3);
    if (tid < 256) {
        const int arow = 32 + r;
        // T_top[s][c] is zero for s < 16 * block(c)
        const float4 y = (cb == 0) ? level2_y<0>(A + arow * 64, arow & 31, T, c)
                                   : level2_y<16>(A + arow * 64, arow & 31, T, c);
        *reinterpret_cast<float4 *>(&P[r * 32 + c]) = y;
    }
    inverse_sync();
    if (tid < 256) {
        // T_bot[r][s] is zero for s >= 16 * (block(r) + 1)
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < 16) {
            level2_x16(acc, Tdiag + 2 * 256 + r, P, 0, c);
        } else {
            level2_x16(acc, T32c + (r - 16), P, 0, c);
            level2_x16(acc, Tdiag + 3 * 256 + (r - 16), P, 16, c);
        }
        const float4 x = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        store_tbeta4(tb, tb16, 32 + r, c, x, beta);
    }
    inverse_sync();
}

// The four 16x16 diagonal blocks of T = (I + A)^{-1} (threads 0..63: block
// tid / 16, column tid % 16) by forward substitution in its right-looking form
// (once x_s is final, subtract A[r][s] x_s from every later row): 15 steps of
// independent FMAs, each step reading one block column of `Adiag` (column-major
// 16x16 blocks) as four broadcast 16-byte loads.  Writes the blocks into T
// (row-major, stride 64), column-major into Tdiag, and T beta into the tf32 and
// bf16 high/low operand tiles.
__device__ __forceinline__ void ut_diag_solve(const float *Adiag, float *T, float *Tdiag,
                                              uint8_t *tb, uint8_t *tb16, const float *beta,
                                              int tid) {
        const int bb = tid >> 4, j = tid & 15, base = bb * 16;
        const float *Ab = Adiag + bb * 256;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
        for (int s = 0; s < 15; ++s) {
            float col[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 v = *reinterpret_cast<const float4 *>(Ab + s * 16 + 4 * q4);
                col[4 * q4] = v.x; col[4 * q4 + 1] = v.y; col[4 * q4 + 2] = v.z; col[4 * q4 + 3] = v.w;
            }
            const float xs = x[s];
#pragma unroll
            for (int r = s + 1; r < 16; ++r) x[r] -= col[r] * xs;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T[(base + r) * 64 + base + j] = x[r];
        float *Td = Tdiag + bb * 256 + j * 16;  // column j of T_bb
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
            *reinterpret_cast<float4 *>(Td + 4 * q4) =
                make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
        // T beta of the diagonal block, column j (16 rows)
        const float bj = beta[base + j];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float xb = x[r] * bj;
            st_f32(tb, sw128_offset(kTbRow0 + base + r, base + j, kTbRows, 4), to_tf32(xb));
            const __nv_bfloat16 hi = __float2bfloat16_rn(xb);
            const __nv_bfloat16 lo = __float2bfloat16_rn(xb - __bfloat162float(hi));
            *reinterpret_cast<__nv_bfloat16 *>(tb16 + sw128_offset(base + r, base + j, 64, 2)) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(tb16 + 8192 + sw128_offset(base + r, base + j, 64, 2)) = lo;
        }
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

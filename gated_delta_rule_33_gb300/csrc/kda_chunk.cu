// kda_chunk.cu -- chunked KDA prefill on tcgen05 tensor cores (sm_103a).
//
// The chunked regime of Kimi Delta Attention (data/code-audit.json, finding
// "dual-kda-execution-regimes"), over packed variable-length sequences with
// initial and final state (K3_ARTIFACT_AUDIT.md section 7.1).  For a chunk of
// L <= 64 tokens starting from state S (rows r, s are tokens of the chunk):
//
//   Gam_r     = sum_{i<=r} g_i                                 (per channel)
//   A_kk[r,s] = beta_r <k_r exp(Gam_r - Gam_s), k_s>   (s < r)
//   A_qk[r,s] = scale <q_r exp(Gam_r - Gam_s), k_s>    (s <= r)
//   T         = (I + A_kk)^{-1}
//   W         = T diag(beta) (k exp(Gam)),   Ut = T diag(beta) V
//   U         = Ut - W S
//   O         = scale (q exp(Gam)) S + A_qk U
//   S        <- Diag(exp(Gam_L)) S + (k exp(Gam_L - Gam))^T U
//
// Numerics.  Every per-channel exponential is split around a per-channel
// reference m = Gam_L / 2 so that each factor lies in [e^{-D/2}, e^{D/2}] with
// D = -Gam_L the chunk's total decay.  D <= 160 is represented: a chunk whose
// decay would exceed it in some channel is shortened to the rows before the
// first one past it (the rest of its tile starts the next chunk); a token
// whose own decay exceeds 160 forms a chunk of one with its decay taken as 160
// (e^{-160} underflows fp32 like any larger decay), so every decay is
// computed.  A_qk and A_kk come from one
// product [Qt; Kr] Ks^T with Qt = scale q e^{Gam-m}, Kr = k e^{Gam-m} and
// Ks = k e^{m-Gam}.  The same Qt and Kr serve the state products because the
// state operand is stored pre-scaled, S_op = Diag(e^m) S, and
// W' = T diag(beta) Kr = W Diag(e^{-m}).  All products run as tcgen05
// kind::tf32 MMAs (operands rounded to tf32, to nearest) with fp32
// accumulation in tensor memory; Ut = T beta V uses kind::f16 with the bf16 V
// tile as loaded and T beta split into a bf16 high and low part.  The state S
// stays in tensor memory in fp32 for the whole sequence.
//
// Work decomposition: one CTA of 512 threads per (sequence, head) chain at a
// time, chains taken from a counter in the workspace.  Warp w serves lane
// quarter w % 4 (channels / tensor-memory lanes 32 (w % 4) ... + 31) and group
// w / 4, which selects its 16 chunk rows when building operands and its slice
// of columns in every tensor-memory epilogue.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"
#include "kda_chunk_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace chunk;

constexpr int kThreads = 512;  // 16 warps: 4 lane quarters x 4 column/row groups

// Shared memory map (bytes from a 1024-aligned base).  Operand tiles are
// K-major with the 128-byte swizzle; "rows" is the M or N extent.
constexpr uint32_t OFF_Q = 0;            // raw q bf16 [64][128] (TMA, no swizzle)
constexpr uint32_t OFF_K = 16384;        // raw k bf16 [64][128] (TMA, no swizzle)
constexpr uint32_t OFF_V = 32768;        // raw v bf16 [64 s][128 v] (TMA, 2 swizzled boxes)
constexpr uint32_t OFF_QK = 49152;       // [Qt ; Kr] tf32, 128 rows (r) x 128 (channel)
constexpr uint32_t OFF_KS = 114688;      // g fp32 64 x 128 (TMA) -> Ks tf32 -> A_kk^T | T fp32
constexpr uint32_t OFF_KH = 147456;      // one tf32 tile, 192 rows x 64 (r), k-block stride 24576:
                                         // rows 0..127 Khat^T (channel), 128..191 T beta -> A_qk
constexpr uint32_t OFF_TB16 = 196608;    // T beta bf16 hi 64 x 64 | lo 64 x 64
constexpr uint32_t OFF_MISC = 212992;
constexpr uint32_t MISC_BETA = 0;        // float[64]
constexpr uint32_t MISC_EM = 256;        // float[128] e^{m}
constexpr uint32_t MISC_DEC = 768;       // float[128] e^{Gam_L}
constexpr uint32_t MISC_P = 1280;        // float[4][256] T-inverse partial products
constexpr uint32_t MISC_PART = 5376;     // float[4][128] partial decay sums per row group
constexpr uint32_t MISC_BNEXT = 7424;    // float[64] beta of the next chunk (cp.async)
constexpr uint32_t MISC_T32 = 7680;      // float[16][16] T_32 column-major (1 KB of 4 KB used)
constexpr uint32_t MISC_TDIAG = 11776;   // float[4][16][16] diagonal blocks of T, column-major
constexpr uint32_t MISC_BAR = 15872;     // 4 mbarriers
constexpr uint32_t MISC_CTRL = 15904;    // int[8]: tmem base, chain, abort, -, split row
constexpr uint32_t kSmemBytes = OFF_MISC + 15936;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

// Tensor memory columns (lane = M row).
//   S_acc: S^T fp32 (lane v, column k)      S_op: tf32(e^{m_k} S[k][v])
//   U: U^T (lane v, column r)               O: W'^T (lane k, column r), then O^T
//   A: [Qt; Kr] Ks^T (lane = row of [Qt; Kr], column s)   W: Kr^T (lane k, column s)
// O^T of a chunk is read out while the next chunk's first MMA runs.  O sits
// between S_acc and U so that one MMA updates [O | U] and one [S_acc | O].
constexpr uint32_t T_SACC = 0, T_O = 128, T_U = 192, T_SOP = 256, T_A = 384, T_W = 448;

struct Params {
    const float *g;              // fp32 log-decay [N, H, 128]   (unfused)
    const float *beta;           // fp32 beta [N, H]             (unfused)
    const void *f;               // bf16 gate pre-activation     (fused gate)
    const void *blog;            // beta logits, bf16 or fp32    (fused gate)
    int blog_bf16;
    const float *A_log;          // per alog_mode                (fused gate)
    int alog_mode;
    const float *dt_bias;        // [H, 128]                     (fused gate)
    const int32_t *cu_seqlens;
    int B;
    int64_t N;
    int H;
    float scale;
    const float *S0;
    float *Sf;
    void *o;
    unsigned int *err;
    unsigned int *counter;
    uint32_t polls_tma;          // bound of the main loop's waits on copies
    uint32_t polls_mma;          // and on products (the drain always uses kMaxPolls)
    float *ckpt;                 // chunk-start states for a backward pass, or NULL
    int *split;                  // per chain: set when a chunk was shortened (with ckpt)
};

// Y[r][c] of level 2 (32 x 32, fp32) in the unused upper-right quarter of T
// (rows 0-31, columns 32-63), the float4 group index XOR-ed by row % 8
__device__ __forceinline__ int ty_idx(int r, int c) { return r * 64 + 32 + (((c >> 2) ^ (r & 7)) << 2); }

// Accumulators of rows r0, r0 + 1 and columns c .. c + 3 of Y as stored.
__device__ __forceinline__ Acc2x4 load_y(const float *T, int r0, int c) {
    Acc2x4 a;
    const float4 y0 = *reinterpret_cast<const float4 *>(T + ty_idx(r0, c));
    const float4 y1 = *reinterpret_cast<const float4 *>(T + ty_idx(r0 + 1, c));
    a.v[0] = f2(y0.x, y0.y);
    a.v[1] = f2(y0.z, y0.w);
    a.v[2] = f2(y1.x, y1.y);
    a.v[3] = f2(y1.z, y1.w);
    return a;
}
__device__ __forceinline__ void store_y(float *T, int r0, int c, const Acc2x4 &a) {
    *reinterpret_cast<float4 *>(T + ty_idx(r0, c)) = a.row(0);
    *reinterpret_cast<float4 *>(T + ty_idx(r0 + 1, c)) = a.row(1);
}

// T = (I + A)^{-1} for the strictly lower-triangular 64 x 64 A_kk (column-major
// in the OFF_KS region), by 16 x 16 blocks, on warps 0-3 -- the 2 x 2-block
// inverse [[A, 0], [C, B]]^-1 = [[A^-1, 0], [-B^-1 C A^-1, B^-1]] applied at 16
// and then at 32 rows:
//   diagonal blocks T_bb by forward substitution (warps 0-1);
//   level 1, T_10 and T_32 (warps 0-1, each on the blocks it solved);
//   level 2, the lower-left 32 x 32 block X = -T_bot Y, Y = A_bl T_top
//   (T_top = T[0:32, 0:32], T_bot = T[32:64, 32:64], A_bl = A[32:64, 0:32]).
// Warp w owns rows 16 (w % 2) .. + 15 and columns 16 (w / 2) .. + 15 of Y and
// X.  What level 2 needs of the diagonal blocks alone is done by warps 2-3
// while warps 0-1 run level 1: their own Y blocks (T_11 only) and the first
// half (T_00) of the K range of warps 0-1's Y blocks.  After level 1, warps 0-1
// finish their Y blocks over the T_10 half, and every warp forms its X block.
// Every sum runs over k in the same order as in one pass.
// The first two levels write T only; warps 6-7 (tbeta_writer) turn their
// blocks into T beta as each level completes, so the conversion and its stores
// stay off the inverse's path; level 2 writes its T beta blocks itself.  (The
// strictly upper blocks of the T beta tiles hold zeros.)  The warp that issues
// the W' and U-tilde products is told when each column block of T beta is
// complete: block 3 after the diagonal solve, block 2 after level 1, blocks
// 0-1 after level 2.  The operands are found from the shared-memory base
// inside the function (a pointer argument would reach it as a generic
// address).
__device__ __forceinline__ void ut_inverse(int tid) {
    uint8_t *smem = smem_base();
    uint8_t *misc = smem + OFF_MISC;
    const float *At = reinterpret_cast<const float *>(smem + OFF_KS);
    float *T = reinterpret_cast<float *>(smem + OFF_KS) + 64 * 64;
    float *Tdiag = reinterpret_cast<float *>(misc + MISC_TDIAG);
    float *T32c = reinterpret_cast<float *>(misc + MISC_T32);
    float *P = reinterpret_cast<float *>(misc + MISC_P);
    const float *beta = reinterpret_cast<const float *>(misc + MISC_BETA);
    const TbetaTiles out{smem + OFF_KH, smem + OFF_TB16, beta};
    const int w = tid >> 5, l = tid & 31, rh = w & 1, cb = w >> 1;
    const int r0 = 16 * rh + 2 * (l >> 2), c0 = 16 * cb + 4 * (l & 3);
    if (tid < 64) {
        // the first two levels into T only (T_32 too, beside its column-major
        // copy); their T beta tiles are written by warps 6-7
        const TRowMajor t_only{T};
        ut_diag_solve(At, T, Tdiag, t_only, tid);
        named_arrive(kBarDiagT, 192);
        __syncwarp();
        ut_level1(At, T, Tdiag, P, T, T32c, t_only, tid);
        named_arrive(kBarLevel1T, 128);
    } else {
        named_sync(kBarDiagT, 192);
        // Y over T_11 (final) and Y over T_00 (the first half of column block 0)
        Acc2x4 y1, y0;
        gemm_2x4<16>(y1, At + 16 * 64 + 32 + r0, 64, T + 16 * 64 + c0, 64);
        gemm_2x4<16>(y0, At + 32 + r0, 64, T + c0 - 16, 64);
        store_y(T, r0, c0, y1);
        store_y(T, r0, c0 - 16, y0);
    }
    inverse_sync();
    if (w < 2) {
        // the T_10 half of column block 0 of Y
        Acc2x4 y = load_y(T, r0, c0);
        gemm_2x4<16>(y, At + 16 * 64 + 32 + r0, 64, T + 16 * 64 + c0, 64);
        store_y(T, r0, c0, y);
        if (w == 0) {
            __syncwarp();
            named_arrive(kBarLevel2Y, 64);
        } else {
            named_sync(kBarLevel2Y, 64);
        }
    }
    // X block of this warp: -T_bot[rows][k] Y[k][c0 .. + 3], k over the nonzero
    // blocks of T_bot (T_32 first, then T_33, for rows 16-31)
    Acc2x4 x;
#pragma unroll
    for (int s = 0; s < 16; ++s)
        x.step(rh == 0 ? *reinterpret_cast<const float2 *>(Tdiag + 2 * 256 + s * 16 + r0)
                       : *reinterpret_cast<const float2 *>(T32c + s * 16 + r0 - 16),
               *reinterpret_cast<const float4 *>(T + ty_idx(s, c0)));
    if (rh == 1) {
#pragma unroll
        for (int s = 16; s < 32; ++s)
            x.step(*reinterpret_cast<const float2 *>(Tdiag + 3 * 256 + (s - 16) * 16 + r0 - 16),
                   *reinterpret_cast<const float4 *>(T + ty_idx(s, c0)));
    }
    out.four(32 + r0, c0, x.neg_row(0));
    out.four(33 + r0, c0, x.neg_row(1));
    fence_proxy_async_smem();
    named_arrive(kBarLevel2, 160);
}

// Warps 6-7 (w = 0..63) during the inverse: T beta of the diagonal blocks once
// the diagonal solve is done (block 3 first, for the first W' / U-tilde k-steps),
// then of T_10 and T_32 once level 1 is done; one row quad T[r][s4 .. s4 + 3]
// read from T per store.
__device__ __forceinline__ void tbeta_writer(int w) {
    uint8_t *smem = smem_base();
    uint8_t *misc = smem + OFF_MISC;
    const float *T = reinterpret_cast<const float *>(smem + OFF_KS) + 64 * 64;
    const float *beta = reinterpret_cast<const float *>(misc + MISC_BETA);
    uint8_t *tb = smem + OFF_KH, *tb16 = smem + OFF_TB16;
    const int r = w >> 2, s4 = 4 * (w & 3);  // row and column quad within a 16 x 16 block
    auto quad = [&](int r0, int c0) {
        store_tbeta4(tb, tb16, r0 + r, c0 + s4,
                     *reinterpret_cast<const float4 *>(T + (r0 + r) * 64 + c0 + s4), beta);
    };
    named_sync(kBarDiagT, 192);
    quad(48, 48);
    fence_proxy_async_smem();
    named_arrive(kBarDiag, 96);
    quad(32, 32);
    quad(16, 16);
    quad(0, 0);
    named_sync(kBarLevel1T, 128);
    quad(48, 32);
    quad(16, 0);
    fence_proxy_async_smem();
    named_arrive(kBarLevel1, 96);
}

// The state pass of a chunk, S_op = tf32(e^{m_k} S[k][v]) and
// S_acc = e^{Gam_L,k} S[k][v] in tensor memory, on warps 8-15 while warps 0-3
// compute the UT inverse: warp w covers lane quarter w % 4 and the 16-column
// slices w / 4 - 2 + 2 n.  With `ckpt`, the chunk-start state S[k][v] is also
// stored there (fp32 [128][128]) for the chunked backward.
__device__ __forceinline__ void state_pass(uint32_t tmem_lane, int warp, const float *em,
                                           const float *dec, float *ckpt, int v) {
    float r16[16], o16[16];
#pragma unroll 1
    for (int cs = (warp >> 2) - 2; cs < 8; cs += 2) {
        const int c0 = 16 * cs;
        tmem_ld16(tmem_lane + T_SACC + c0, r16);
        tmem_wait_ld();
        if (ckpt != nullptr) {  // S[k][v] at the chunk start, k = c0 + j
#pragma unroll
            for (int j = 0; j < 16; ++j) ckpt[(c0 + j) * kD + v] = r16[j];
        }
#pragma unroll
        for (int j = 0; j < 16; j += 2) {  // packed pairs of columns
            const uint64_t rr = f2(r16[j], r16[j + 1]);
            const float2 o = f2_split(f2_mul(rr, *reinterpret_cast<const uint64_t *>(em + c0 + j)));
            const float2 d = f2_split(f2_mul(rr, *reinterpret_cast<const uint64_t *>(dec + c0 + j)));
            o16[j] = to_tf32(o.x);
            o16[j + 1] = to_tf32(o.y);
            r16[j] = d.x;
            r16[j + 1] = d.y;
        }
        tmem_st16(tmem_lane + T_SOP + c0, o16);
        tmem_st16(tmem_lane + T_SACC + c0, r16);
    }
    tmem_wait_st();
}

// kGate: the gate is computed in this kernel from the bf16 pre-activation f,
// A_log, dt_bias and the beta logits (g = -exp(A_log) softplus(f + dt_bias),
// beta = sigmoid(logit)) with the special-function unit, instead of reading a
// precomputed fp32 g and beta.  kCkpt: the forward pass of the chunked
// backward (chunk-start states to p.ckpt, shortened chunks to p.split).
template <bool kOutBf16, bool kGate, bool kCkpt>
__global__ void __launch_bounds__(kThreads, 1) chunk_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                            const __grid_constant__ CUtensorMap tm_k,
                                                            const __grid_constant__ CUtensorMap tm_v,
                                                            const __grid_constant__ CUtensorMap tm_g,
                                                            const Params p) {
    uint8_t *smem = smem_base();
    uint8_t *misc = smem + OFF_MISC;
    float *s_beta = reinterpret_cast<float *>(misc + MISC_BETA);
    float *s_em = reinterpret_cast<float *>(misc + MISC_EM);
    float *s_dec = reinterpret_cast<float *>(misc + MISC_DEC);
    uint64_t *bar_qk = reinterpret_cast<uint64_t *>(misc + MISC_BAR);
    uint64_t *bar_v = bar_qk + 1;
    uint64_t *bar_mma = bar_qk + 2;
    uint64_t *bar_g = bar_qk + 3;
    float *s_bnext = reinterpret_cast<float *>(misc + MISC_BNEXT);
    int *ctrl = reinterpret_cast<int *>(misc + MISC_CTRL);  // [0] tmem [1] chain [2] abort [4] split row

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, grp = warp >> 2;
    const int ch = quarter * 32 + (tid & 31);  // channel / tensor-memory lane
    const int H = p.H;
    const int num_chains = p.B * H;

    if (warp == 0) tmem_alloc(reinterpret_cast<uint32_t *>(&ctrl[0]), 512);
    if (tid == 0) {
        mbar_init(bar_qk, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_g, 1);
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
        ctrl[2] = 0;
        ctrl[4] = kC;
    }
    // The strictly upper blocks of the T beta tiles are zero for every chunk and
    // are never written again (A_qk, which reuses the tf32 rows, is zero there too).
    for (int e = tid; e < 49152 / 16; e += kThreads)
        reinterpret_cast<float4 *>(smem + OFF_KH)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int e = tid; e < 16384 / 16; e += kThreads)
        reinterpret_cast<float4 *>(smem + OFF_TB16)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(ctrl[0]);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float *s_part = reinterpret_cast<float *>(misc + MISC_PART);

    // Phases consumed so far (identical in every thread) and, in thread 0,
    // whether a TMA batch is in flight.  A batch or product whose wait ran out
    // stays marked in flight (its phase is not advanced), so the drain at the
    // end waits for it before the CTA releases tensor memory and exits.
    uint32_t ph_qk = 0, ph_v = 0, ph_mma = 0, ph_g = 0;
    bool pend_qk = false, pend_v = false, pend_g = false;
    // a product commit on bar_mma is not yet consumed (identical in every thread)
    bool pend_mma = false;

    const uint32_t a_qk = smem_addr(smem + OFF_QK);
    const uint32_t a_ks = smem_addr(smem + OFF_KS);
    const uint32_t a_kh = smem_addr(smem + OFF_KH);
    const uint32_t a_tb16 = smem_addr(smem + OFF_TB16);
    const uint32_t a_v = smem_addr(smem + OFF_V);
    // Shared-memory descriptors of every operand tile (128-byte swizzle), built
    // once; a k-step adds its constant byte offset / 16 to the start address.
    const uint64_t d_qk = smem_desc(a_qk, 16, 1024, kSwizzle128B);
    const uint64_t d_ks = smem_desc(a_ks, 16, 1024, kSwizzle128B);
    const uint64_t d_kh = smem_desc(a_kh, 16, 1024, kSwizzle128B);
    const uint64_t d_tb16 = smem_desc(a_tb16, 16, 1024, kSwizzle128B);
    const uint64_t d_v = smem_desc(a_v, 8192, 1024, kSwizzle128B);  // MN-major, 64-wide M blocks
    float *Akk = reinterpret_cast<float *>(smem + OFF_KS);
    // largest chunk decay represented, in log2 units
    const float kMaxChunkLog2 = kMaxChunkDecay * 1.4426950408889634f;

    while (ctrl[2] == 0) {
        __syncthreads();
        if (tid == 0) ctrl[1] = static_cast<int>(atomicAdd(p.counter, 1u));
        __syncthreads();
        const int chain = ctrl[1];
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
        // O^T of the chunk starting at token tcw (Lw valid rows) from tensor memory to o
        // (rows 16 gw .. + 15 of the warp's lane quarter)
        auto write_output = [&](int64_t tcw, int Lw, int gw) {
            if (p.o == nullptr) return;
            float o16[16];
            tmem_ld16(tmem + lane_base + T_O + 16 * gw, o16);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = 16 * gw + j;
                if (r < Lw) {
                    const int64_t idx = ((tcw + r) * H + h) * kD + ch;
                    if (kOutBf16)
                        static_cast<__nv_bfloat16 *>(p.o)[idx] = __float2bfloat16_rn(o16[j]);
                    else
                        static_cast<float *>(p.o)[idx] = o16[j];
                }
            }
        };

        // ---- initial state into S_acc (lane v, column k holds S[k][v]) ----
        {
            float r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                r[j] = (p.S0 != nullptr) ? p.S0[state_off + (32 * grp + j) * kD + ch] : 0.f;
            tmem_st32(tmem + lane_base + T_SACC + 32 * grp, r);
            tmem_wait_st();
        }

        auto issue_qk = [&](int64_t tc) {
            mbar_arrive_expect_tx(bar_qk, 2 * 16384);
            tma_load_3d(smem + OFF_Q, &tm_q, bar_qk, 0, h, static_cast<int32_t>(tc));
            tma_load_3d(smem + OFF_K, &tm_k, bar_qk, 0, h, static_cast<int32_t>(tc));
            pend_qk = true;
        };
        auto issue_v = [&](int64_t tc) {
            mbar_arrive_expect_tx(bar_v, 16384);
            tma_load_3d(smem + OFF_V, &tm_v, bar_v, 0, h, static_cast<int32_t>(tc));
            tma_load_3d(smem + OFF_V + 8192, &tm_v, bar_v, 64, h, static_cast<int32_t>(tc));
            pend_v = true;
        };
        // g of the chunk: one TMA tile into the OFF_KS region; beta: one
        // zero-filled 4-byte cp.async per row into s_bnext (threads 0..63).
        auto issue_g = [&](int64_t tc) {
            mbar_arrive_expect_tx(bar_g, kGate ? 16384 : 32768);
            tma_load_3d(smem + OFF_KS, &tm_g, bar_g, 0, h, static_cast<int32_t>(tc));
            pend_g = true;
        };
        // fused gate: per-channel exp(A_log) and dt_bias of this head
        float gate_a = 0.f, gate_dt = 0.f, blog_reg = 0.f;
        if (kGate) {
            const int ai = (p.alog_mode == 0) ? h : (p.alog_mode == 1 ? ch : h * kD + ch);
            gate_a = expf(p.A_log[ai]);
            gate_dt = p.dt_bias[h * kD + ch];
        }
        auto load_beta = [&](int64_t tc, int L) {
            if (kGate) {
                // the logit stays in a register until the chunk is processed;
                // rows past the sequence get -inf, whose sigmoid is 0
                if (tid < kC) {
                    if (tid < L) {
                        const int64_t bi = (tc + tid) * H + h;
                        blog_reg = p.blog_bf16
                                       ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p.blog)[bi])
                                       : static_cast<const float *>(p.blog)[bi];
                    } else {
                        blog_reg = -__int_as_float(0x7f800000);
                    }
                }
            } else if (tid < kC) {
                cp_async_4(&s_bnext[tid], p.beta + ((tid < L) ? (tc + tid) * H + h : 0), tid < L);
            }
        };
        if (t1 > t0) {
            if (tid == 0) {
                issue_g(t0);
                issue_qk(t0);
                issue_v(t0);
            }
            load_beta(t0, static_cast<int>((t1 - t0) < kC ? (t1 - t0) : kC));
        }

        // The chunk whose output is still in the O columns of tensor memory.
        int64_t prev_tc = t0;
        int prev_L = 0;
        // checkpoint slot of this sequence's first chunk (see kda_chunk_bwd.cu)
        bool ckpt_ok = kCkpt;
        const int64_t ckpt_slot0 = t0 / kC + b;
        for (int64_t tc = t0; tc < t1;) {
            // L tokens from tc; a chunk whose decay exceeds the represented
            // range in some channel is shortened below (and the rest of its
            // tile starts the next chunk)
            int L = static_cast<int>((t1 - tc) < kC ? (t1 - tc) : kC);

            // ---- S1: cumulative decay, references, operands ----
            cp_async_wait_all();
            // polled by warp 1: thread 0 may still be issuing the previous
            // chunk's last product
            bool copies_ok = true;
            if (tid == 32 && (!mbar_wait_bounded(bar_qk, ph_qk & 1, p.polls_tma) ||
                              !mbar_wait_bounded(bar_g, ph_g & 1, p.polls_tma))) {
                ctrl[2] = 1;
                record_device_error(p.err, kDevTimeout);
                copies_ok = false;
            }
            copies_ok = __syncthreads_and(copies_ok);
            tc_fence_after();
            if (!copies_ok) break;  // the batches stay pending for the drain
            ph_g++;
            ph_qk++;
            pend_g = false;
            pend_qk = false;
            // cumulative decay in log2 units: gam = log2(e) * sum g
            float gam[16];
            {
                const float kLog2e = 1.4426950408889634f;
                float acc = 0.f;
                if (kGate) {
                    // log2(e) g = -exp(A_log) (log2(e) max(x, 0) + log2(1 + 2^{-log2(e)|x|})),
                    // x = f + dt_bias
                    const __nv_bfloat16 *ft = reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_KS);
                    const uint64_t dt2 = f2(gate_dt, gate_dt), na2 = f2(-gate_a, -gate_a);
                    const uint64_t l2e2 = f2(kLog2e, kLog2e);
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {  // rows r, r + 1 as packed pairs
                        const int r = 16 * grp + i;
                        const float2 x = f2_split(f2_add(f2(__bfloat162float(ft[r * kD + ch]),
                                                            __bfloat162float(ft[(r + 1) * kD + ch])),
                                                         dt2));
                        const uint64_t e = f2(fast_exp2(-kLog2e * fabsf(x.x)), fast_exp2(-kLog2e * fabsf(x.y)));
                        const float2 g2 = f2_split(f2_mul(
                            na2, f2_fma(l2e2, f2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log2_1p_unit2(e))));
                        acc += (r < L) ? g2.x : 0.f;
                        gam[i] = acc;
                        acc += (r + 1 < L) ? g2.y : 0.f;
                        gam[i + 1] = acc;
                    }
                } else {
                    const float *gt = reinterpret_cast<const float *>(smem + OFF_KS);
                    // g must be a decay (g <= 0): a positive or NaN g in the
                    // chunk's rows is reported (rows past the sequence belong
                    // to the next one or are zero-filled)
                    float gmax = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int r = 16 * grp + i;
                        const float gv = kLog2e * gt[r * kD + ch];
                        gmax = fmaxf(gmax, gv);
                        acc += (r < L) ? gv : 0.f;
                        gam[i] = acc;
                    }
                    if (gmax > 0.f || acc != acc) record_device_error(p.err, kDevInvalidArg);
                }
            }
            float beta_r = 0.f;  // beta of row tid (threads 0..63)
            if (tid < kC) beta_r = kGate ? 1.f / (1.f + __expf(-blog_reg)) : s_bnext[tid];
            // Builds the operands of the chunk's first L rows from gam and finds
            // (wide) whether some channel's decay exceeds the represented range;
            // runs a second time for a chunk that is split.  Returns false when
            // the CTA is aborting.
            float prefix = 0.f;  // decay before this thread's rows, log2 units
            bool wide = false;
            auto build = [&]() -> bool {
                s_part[grp * kD + ch] = gam[15];
                if (tid < kC) s_beta[tid] = beta_r;
                __syncthreads();  // every g read is done before Ks overwrites the tile
                float gam_l = 0.f;
                prefix = 0.f;
#pragma unroll
                for (int g2 = 0; g2 < 4; ++g2) {
                    const float pg = s_part[g2 * kD + ch];
                    if (g2 < grp) prefix += pg;
                    gam_l += pg;
                }
                const bool over = -gam_l > kMaxChunkLog2;
                const float m = 0.5f * gam_l;
                if (grp == 0) {
                    s_em[ch] = fast_exp2(m);
                    s_dec[ch] = fast_exp2(gam_l);
                }
                const float ekh = fast_exp2(gam_l - m);
                const float qscale = p.scale;
                float krt[16], khv[16];
                const uint64_t m2 = f2(m, m), pre2 = f2(prefix, prefix), qs2 = f2(qscale, qscale);
                const uint64_t ekh2 = f2(ekh, ekh);
#pragma unroll
                for (int i = 0; i < 16; i += 2) {  // rows r, r + 1 as packed pairs
                    const int r = 16 * grp + i;
                    const bool v0 = r < L, v1 = r + 1 < L;  // rows past the chunk stay zero
                    const uint64_t gr = f2_add(pre2, f2(gam[i], gam[i + 1]));
                    const float2 du = f2_split(f2_sub(gr, m2)), dd = f2_split(f2_sub(m2, gr));
                    const uint64_t e_up = f2(fast_exp2(du.x), fast_exp2(du.y));  // e^{Gam_r - m}
                    const uint64_t e_dn = f2(fast_exp2(dd.x), fast_exp2(dd.y));  // e^{m - Gam_r}
                    const uint64_t qv = f2(v0 ? bf(smem + OFF_Q, (r * kD + ch) * 2) : 0.f,
                                           v1 ? bf(smem + OFF_Q, ((r + 1) * kD + ch) * 2) : 0.f);
                    const uint64_t kv = f2(v0 ? bf(smem + OFF_K, (r * kD + ch) * 2) : 0.f,
                                           v1 ? bf(smem + OFF_K, ((r + 1) * kD + ch) * 2) : 0.f);
                    const float2 qt = f2_split(f2_mul(f2_mul(qs2, qv), e_up));
                    const float2 kr = f2_split(f2_mul(kv, e_up));
                    const float2 ks = f2_split(f2_mul(kv, e_dn));
                    const float2 kh = f2_split(f2_mul(kv, f2_mul(e_dn, ekh2)));
                    st_f32(smem + OFF_QK, sw128_offset(r, ch, 128, 4), to_tf32(qt.x));
                    st_f32(smem + OFF_QK, sw128_offset(r + 1, ch, 128, 4), to_tf32(qt.y));
                    krt[i] = to_tf32(kr.x);
                    krt[i + 1] = to_tf32(kr.y);
                    st_f32(smem + OFF_QK, sw128_offset(r + 64, ch, 128, 4), krt[i]);
                    st_f32(smem + OFF_QK, sw128_offset(r + 65, ch, 128, 4), krt[i + 1]);
                    st_f32(smem + OFF_KS, sw128_offset(r, ch, 64, 4), to_tf32(ks.x));
                    st_f32(smem + OFF_KS, sw128_offset(r + 1, ch, 64, 4), to_tf32(ks.y));
                    khv[i] = to_tf32(kh.x);
                    khv[i + 1] = to_tf32(kh.y);
                }
                // The previous chunk's [S | O] product, which reads Khat^T, ran while
                // these operands were formed; it is complete before Khat^T is overwritten.
                if (pend_mma) {
                    if (!cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid, p.polls_mma)) return false;
                    ph_mma++;
                    pend_mma = false;
                }
                // Khat^T row ch, columns r = 16 grp .. +15: four 16-byte stores
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<float4 *>(smem + OFF_KH + sw128_offset(ch, 16 * grp + 4 * q4, 192, 4)) =
                        make_float4(khv[4 * q4], khv[4 * q4 + 1], khv[4 * q4 + 2], khv[4 * q4 + 3]);
                tmem_st16(tmem + lane_base + T_W + 16 * grp, krt);
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                wide = __syncthreads_or(over) != 0;
                tc_fence_after();
                return true;
            };
            if (!build()) break;
            if (wide) {
                // A chunk split (rare: some channel's decay exceeds the range).
                // The rows from the first one beyond the range in any channel
                // start the next chunk; gam keeps its values up to the new last
                // row and repeats the last one after it (those rows add no
                // decay), and the operands are formed again.  A first token
                // whose own decay exceeds the range makes a chunk of one token
                // with its decay taken as the range: e^-160 vanishes in fp32
                // like any larger decay.
                int first = kC;
#pragma unroll
                for (int i = 15; i >= 0; --i) {
                    const int r = 16 * grp + i;
                    if (r < L && -(prefix + gam[i]) > kMaxChunkLog2) first = r;
                }
                if (first < kC) atomicMin(&ctrl[4], first);
                __syncthreads();
                int Ls = ctrl[4];
                __syncthreads();  // every thread has read the split row
                if (tid == 0) ctrl[4] = kC;
                if (Ls == 0) {
                    Ls = 1;
                    if (grp == 0) gam[0] = fmaxf(gam[0], -kMaxChunkLog2);
                }
                if (Ls < L) {
                    L = Ls;
                    if (tid >= L) beta_r = 0.f;
                }
                float last = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (16 * grp + i < L)
                        last = gam[i];
                    else
                        gam[i] = last;
                }
                if (!build()) break;
            }
            // a shortened chunk: later chunk starts are no longer 64-token aligned,
            // so this chain's checkpoints stop here and the chain is marked
            if (kCkpt && L < kC && tc + L < t1) {
                if (tid == 0) p.split[chain] = 1;
                ckpt_ok = false;
            }
            const int64_t tn = tc + L;
            const int Ln = static_cast<int>(tn >= t1 ? 0 : ((t1 - tn) < kC ? (t1 - tn) : kC));

            // ---- S2: D_A = [Qt; Kr] Ks^T ; next q/k loads ; previous chunk's output ----
            if (warp == 0) {
                // a converged warp issues faster than one lane of a divergent one
                __syncwarp();
                const uint32_t id = instr_desc(128, 64, kFmtTF32, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint64_t ad = (d_qk + static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4));
                    const uint64_t bd = (d_ks + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4));
                    mma_tf32_ss_w(tmem + T_A, ad, bd, id, kk > 0);
                }
                mma_commit_w(bar_mma);
                if (tid == 0 && Ln > 0) issue_qk(tn);
            }
            pend_mma = true;
            // warp 0 issues the products; warp 4 (same lane quarter) takes its rows
            // (a full chunk's rows are stored without a per-row test)
            if (prev_L == kC && warp != 0) {
                write_output(prev_tc, kC, grp);
                if (warp == 4) write_output(prev_tc, kC, 0);
            } else if (prev_L > 0 && warp != 0) {
                write_output(prev_tc, prev_L, grp);
                if (warp == 4) write_output(prev_tc, prev_L, 0);
            }

            // ---- S3: A_kk from the k-side rows of D_A ----
            if (!cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid, p.polls_mma)) break;
            ph_mma++;
            pend_mma = false;
            if (quarter >= 2) {
                const int r = ch - 64;
                const float br = s_beta[r];
                float d16[16];
                tmem_ld16(tmem + lane_base + T_A + 16 * grp, d16);
                tmem_wait_ld();
                // Ks is dead once D_A is complete; A_kk (column-major) overwrites it
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int s = 16 * grp + j;
                    Akk[s * 64 + r] = (s < r) ? br * d16[j] : 0.f;
                }
            }
            __syncthreads();

            // ---- S4: UT inverse (warps 0-3) with its T beta tiles (warps 6-7
            // for the first two levels); W'^T = Kr^T (T beta)^T and
            // Ut^T = V^T (T beta)^T issued by warp 4 one column block of T beta
            // (one K range of the products) at a time as the inverse completes
            // it; the state pass (warps 8-15) ----
            if (warp < 4) {
                ut_inverse(tid);
            } else if (warp == 4) {
                const uint32_t idw = instr_desc(128, 64, kFmtTF32, 0, 0);
                const uint32_t idu = instr_desc(128, 64, kFmtBF16, 1, 0);
                bool v_ok = true;
                // W' over tf32 k-steps kk (8 columns of T beta each), U-tilde over
                // bf16 k-steps ku (16 columns) for the high and low halves
                auto issue_w = [&](int kk, bool first) {
                    const uint64_t bd = (d_kh + static_cast<uint64_t>(((kk >> 2) * 24576 + 16384 + (kk & 3) * 32) >> 4));
                    mma_tf32_ts_w(tmem + T_O, tmem + T_W + kk * 8, bd, idw, first ? 0u : 1u);
                };
                auto issue_u = [&](int ku, bool first) {
                    const uint64_t ad = (d_v + static_cast<uint64_t>((ku * 2048) >> 4));
                    mma_f16_ss_w(tmem + T_U, ad, d_tb16 + static_cast<uint64_t>((ku * 32) >> 4), idu,
                                 first ? 0u : 1u);
                    mma_f16_ss_w(tmem + T_U, ad, d_tb16 + static_cast<uint64_t>((8192 + ku * 32) >> 4),
                                 idu, 1u);
                };
                named_sync(kBarDiag, 96);
                tc_fence_after();
                issue_w(6, true);
                issue_w(7, false);
                int ok = 1;
                if (lane == 0 && !mbar_wait_bounded(bar_v, ph_v & 1, p.polls_tma)) {
                    ok = 0;
                    ctrl[2] = 1;
                    record_device_error(p.err, kDevTimeout);
                }
                // no product reads V unless its copy is known to be complete
                v_ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
                if (v_ok) issue_u(3, true);
                named_sync(kBarLevel1, 96);
                tc_fence_after();
                issue_w(4, false);
                issue_w(5, false);
                if (v_ok) issue_u(2, false);
                named_sync(kBarLevel2, 160);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) issue_w(kk, false);
                if (v_ok) {
                    issue_u(0, false);
                    issue_u(1, false);
                }
                mma_commit_w(bar_mma);
            } else if (warp == 6 || warp == 7) {
                tbeta_writer(tid - 192);
            } else if (warp >= 8) {
                float *ck = nullptr;
                if (kCkpt && ckpt_ok && ((tc - t0) % kC) == 0)
                    ck = p.ckpt + ((ckpt_slot0 + (tc - t0) / kC) * H + h) * (kD * kD);
                state_pass(tmem + lane_base, warp, s_em, s_dec, ck, ch);
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            pend_mma = true;
            // a V copy that did not arrive stays pending for the drain
            if (ctrl[2] != 0) break;
            ph_v++;
            pend_v = false;

            // ---- S5: the W' and U-tilde products complete ----
            // A_kk and T are consumed: the next chunk's g and beta are staged now.
            if (Ln > 0) load_beta(tn, Ln);
            if (tid == 0 && Ln > 0) issue_g(tn);
            if (!cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid, p.polls_mma)) break;
            ph_mma++;
            pend_mma = false;
            if (tid == 0 && Ln > 0) issue_v(tn);

            // ---- S6: -W' into rows 64..127 of the [Qt ; Kr] tile (Kr is dead
            // since D_A); the O columns are cleared for the accumulating MMA ----
            {
                float w16[16];
                tmem_ld16(tmem + lane_base + T_O + 16 * grp, w16);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    st_f32(smem + OFF_QK, sw128_offset(64 + 16 * grp + j, ch, 128, 4), -to_tf32(w16[j]));
                    w16[j] = 0.f;
                }
                tmem_st16(tmem + lane_base + T_O + 16 * grp, w16);
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

            // ---- S7: [O^T | U^T] += S_op [Qt ; -W']^T (O columns start at zero) ----
            if (warp == 0) {
                __syncwarp();
                const uint32_t id = instr_desc(128, 128, kFmtTF32, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint64_t bq = (d_qk + static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4));
                    mma_tf32_ts_w(tmem + T_O, tmem + T_SOP + kk * 8, bq, id, 1);
                }
                mma_commit_w(bar_mma);
            }
            pend_mma = true;
            // A_qk (K-major [r][s], zero above the diagonal) while MMA1/MMA2 run;
            // the T beta tile it overwrites was consumed by the W' product.
            // (warp 0 issues the products; warp 4, same lane quarter, takes its columns)
            auto store_aqk = [&](int gw) {
                const int r = ch;
                float a16[16];
                tmem_ld16(tmem + lane_base + T_A + 16 * gw, a16);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int s = 16 * gw + j;
                    st_f32(smem + OFF_KH, sw128_offset(kTbRow0 + r, s, kTbRows, 4),
                           (s <= r) ? to_tf32(a16[j]) : 0.f);
                }
            };
            if (quarter < 2 && warp != 0) {
                store_aqk(grp);
                if (warp == 4) store_aqk(0);
            }
            fence_proxy_async_smem();
            if (!cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid, p.polls_mma)) break;
            ph_mma++;
            pend_mma = false;

            // ---- S8: U rounded to tf32 in place (A operand of the next MMAs) ----
            {
                float u16[16];
                tmem_ld16(tmem + lane_base + T_U + 16 * grp, u16);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) u16[j] = to_tf32(u16[j]);
                tmem_st16(tmem + lane_base + T_U + 16 * grp, u16);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

            // ---- S9: [S_acc^T | O^T] += U^T [Khat^T ; A_qk]^T ----
            if (warp == 0) {
                __syncwarp();
                const uint32_t id = instr_desc(128, 192, kFmtTF32, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t bk = (d_kh + static_cast<uint64_t>(((kk >> 2) * 24576 + (kk & 3) * 32) >> 4));
                    mma_tf32_ts_w(tmem + T_SACC, tmem + T_U + kk * 8, bk, id, 1);
                }
                mma_commit_w(bar_mma);
            }
            // ---- S10: the product completes under the next chunk's operand
            // build, and this chunk's output is read out under the next MMA ----
            pend_mma = true;
            prev_tc = tc;
            prev_L = L;
            tc = tn;
        }
        if (ctrl[2] != 0) break;  // to the drain
        if (pend_mma) {
            if (!cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid, p.polls_mma)) break;
            ph_mma++;
            pend_mma = false;
        }
        if (prev_L > 0) write_output(prev_tc, prev_L, grp);  // output of the last chunk

        // ---- final state ----
        if (p.Sf != nullptr) {
            float r[32];
            tmem_ld32(tmem + lane_base + T_SACC + 32 * grp, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) p.Sf[state_off + (32 * grp + j) * kD + ch] = r[j];
        }
    }

    // Drain: after an abort, wait for every TMA batch and product still in
    // flight, with the full bound whatever limit the main loop used, so that
    // no copy lands in shared memory after this CTA has exited and no product
    // is running when the tensor memory is released.
    cp_async_wait_all();
    if (tid == 0) {
        if (pend_qk) mbar_wait_bounded(bar_qk, ph_qk & 1, kMaxPolls);
        if (pend_v) mbar_wait_bounded(bar_v, ph_v & 1, kMaxPolls);
        if (pend_g) mbar_wait_bounded(bar_g, ph_g & 1, kMaxPolls);
        if (pend_mma) mbar_wait_bounded(bar_mma, ph_mma & 1, kMaxPolls);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

namespace {
// Bounds of the main loop's waits for the next launches (kMaxPolls unless a
// test shortens them to make a wait run out).
std::atomic<uint32_t> g_polls_tma{kMaxPolls};
std::atomic<uint32_t> g_polls_mma{kMaxPolls};
}  // namespace

void set_prefill_wait_polls(int64_t copy_polls, int64_t product_polls) {
    auto clamp = [](int64_t v) -> uint32_t {
        if (v < 0 || v > static_cast<int64_t>(kMaxPolls)) return kMaxPolls;
        return static_cast<uint32_t>(v);
    };
    g_polls_tma.store(clamp(copy_polls));
    g_polls_mma.store(clamp(product_polls));
}

uint32_t prefill_wait_polls() { return g_polls_mma.load(); }

size_t prefill_workspace_bytes(int64_t N, int B, int H) {
    (void)N;
    return (B > 0 && H > 0) ? 256 : 0;
}

namespace {

template <bool kGate, bool kCkpt = false>
cudaError_t launch_chunk(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                         const void *g_or_f, const Params &p, bool o_bf16, int num_sms,
                         cudaStream_t s) {
    if (p.B == 0 || p.H == 0) return cudaSuccess;
    cudaError_t ea = o_bf16 ? ensure_dynamic_smem(reinterpret_cast<const void *>(chunk_kernel<true, kGate, kCkpt>),
                                                  static_cast<int>(kSmemAlloc))
                            : ensure_dynamic_smem(reinterpret_cast<const void *>(chunk_kernel<false, kGate, kCkpt>),
                                                  static_cast<int>(kSmemAlloc));
    if (ea != cudaSuccess) return ea;
    CUtensorMap mq, mk, mv, mg;
    // With no tokens no tile is ever loaded (every chain is empty), but a map
    // needs a valid aligned address: the chain counter's stands in for the
    // token tensors, which may then be absent.
    const int64_t Nmap = p.N > 0 ? p.N : 1;
    auto at = [&](const void *t) -> const void * { return p.N > 0 ? t : p.counter; };
    if (!make_map(&mq, at(q), Nmap, p.H, 128, false) || !make_map(&mk, at(k), Nmap, p.H, 128, false) ||
        !make_map(&mv, at(v), Nmap, p.H, 64, true) ||
        !make_map(&mg, at(g_or_f), Nmap, p.H, 128, false, !kGate))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(p.counter, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    Params pl = p;
    pl.polls_tma = g_polls_tma.load();
    pl.polls_mma = g_polls_mma.load();
    const int chains = p.B * p.H;
    const int grid = chains < num_sms ? chains : num_sms;
    if (o_bf16)
        chunk_kernel<true, kGate, kCkpt><<<grid, kThreads, kSmemAlloc, s>>>(mq, mk, mv, mg, pl);
    else
        chunk_kernel<false, kGate, kCkpt><<<grid, kThreads, kSmemAlloc, s>>>(mq, mk, mv, mg, pl);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, const float *g, const float *beta,
                           const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
                           const float *initial_state, float *final_state, void *o, bool o_bf16,
                           void *workspace, unsigned int *err, int num_sms, cudaStream_t s) {
    const Params p{g, beta, nullptr, nullptr, 0, nullptr, 0, nullptr, cu_seqlens, B, N, H, scale,
                   initial_state, final_state, o, err, static_cast<unsigned int *>(workspace),
                   kMaxPolls, kMaxPolls, nullptr, nullptr};
    return launch_chunk<false>(q, k, v, g, p, o_bf16, num_sms, s);
}

cudaError_t launch_prefill_checkpoints(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                       const __nv_bfloat16 *v, const float *g, const float *beta,
                                       const int32_t *cu_seqlens, int B, int64_t N, int H,
                                       float scale, const float *initial_state, float *ckpt,
                                       int *split, unsigned int *counter, unsigned int *err,
                                       int num_sms, cudaStream_t s) {
    const Params p{g, beta, nullptr, nullptr, 0, nullptr, 0, nullptr, cu_seqlens, B, N, H, scale,
                   initial_state, nullptr, nullptr, err, counter, kMaxPolls, kMaxPolls, ckpt, split};
    return launch_chunk<false, true>(q, k, v, g, p, false, num_sms, s);
}

cudaError_t launch_prefill_checkpointed(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                        const __nv_bfloat16 *v, const float *g, const float *beta,
                                        const int32_t *cu_seqlens, int B, int64_t N, int H,
                                        float scale, const float *initial_state, float *final_state,
                                        void *o, bool o_bf16, float *ckpt, int *split,
                                        void *workspace, unsigned int *err, int num_sms,
                                        cudaStream_t s) {
    if (B == 0 || H == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(split, 0, static_cast<size_t>(B) * H * sizeof(int), s);
    if (e != cudaSuccess) return e;
    const Params p{g, beta, nullptr, nullptr, 0, nullptr, 0, nullptr, cu_seqlens, B, N, H, scale,
                   initial_state, final_state, o, err, static_cast<unsigned int *>(workspace),
                   kMaxPolls, kMaxPolls, ckpt, split};
    return launch_chunk<false, true>(q, k, v, g, p, o_bf16, num_sms, s);
}

cudaError_t launch_prefill_gated(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                 const __nv_bfloat16 *v, const __nv_bfloat16 *f, const void *b,
                                 bool b_bf16, const float *A_log, int alog_mode,
                                 const float *dt_bias, const int32_t *cu_seqlens, int B, int64_t N,
                                 int H, float scale, const float *initial_state,
                                 float *final_state, void *o, bool o_bf16, void *workspace,
                                 unsigned int *err, int num_sms, cudaStream_t s) {
    const Params p{nullptr, nullptr, f, b, b_bf16 ? 1 : 0, A_log, alog_mode, dt_bias, cu_seqlens,
                   B, N, H, scale, initial_state, final_state, o, err,
                   static_cast<unsigned int *>(workspace), kMaxPolls, kMaxPolls, nullptr, nullptr};
    return launch_chunk<true>(q, k, v, f, p, o_bf16, num_sms, s);
}

// ---- built-in scratch for callers that cannot allocate ---------------------------------
//
// kda_chunk_prefill_noalloc() (include/kda.h) runs the same launch as
// kda_chunk_prefill() but takes its scratch from this file-scope device array
// instead of a caller-provided workspace.  Every GPU that loads the library
// holds the array until the process exits, and every call on a device shares
// it, so calls whose kernels overlap on the GPU race on it.
namespace {
constexpr size_t kBuiltinScratchBytes = 4096;
static __device__ __align__(256) unsigned char g_builtin_scratch[kBuiltinScratchBytes];

constexpr int kMaxScratchDevices = 64;
void *g_builtin_scratch_ptr[kMaxScratchDevices];
std::mutex g_builtin_scratch_mutex;
}  // namespace

// The device address of the built-in scratch on the current device.  The
// first call on a device looks it up with cudaGetSymbolAddress (the array's
// name is a host-side stand-in, not a device address); later calls reuse it.
cudaError_t builtin_prefill_scratch(void **ptr, size_t *bytes) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_builtin_scratch_mutex);
    if (g_builtin_scratch_ptr[dev] == nullptr) {
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_builtin_scratch);
        if (e != cudaSuccess) return e;
        g_builtin_scratch_ptr[dev] = addr;
    }
    *ptr = g_builtin_scratch_ptr[dev];
    *bytes = kBuiltinScratchBytes;
    return cudaSuccess;
}

}  // namespace kda


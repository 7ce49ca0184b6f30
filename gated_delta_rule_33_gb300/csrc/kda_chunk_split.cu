// kda_chunk_split.cu -- chunked KDA prefill in two phases (sm_103a).
//
// The chunked regime of Kimi Delta Attention (data/code-audit.json, finding
// "dual-kda-execution-regimes") over packed sequences with initial and final
// state (K3_ARTIFACT_AUDIT.md section 7.1).  For a chunk of L <= 64 tokens
// starting from state S (rows r, s are tokens of the chunk, per-channel
// cumulative decay Gam_r, reference m = Gam_L / 2):
//
//   Qt = scale q e^{Gam-m},  Kr = k e^{Gam-m},  Ks = k e^{m-Gam},  Khat = k e^{Gam_L-Gam}
//   A_qk = tril(Qt Ks^T),  A_kk = diag(beta) tril(Kr Ks^T, -1),  T = (I + A_kk)^{-1}
//   W' = T beta Kr,  Ut = T beta V                            (independent of S)
//   U = Ut - W' S_op,  O = Qt S_op + A_qk U,  S <- Diag(e^{Gam_L}) S + Khat^T U
//   with S_op = Diag(e^m) S
//
// Everything on the first line of products depends only on the chunk's own
// inputs, so it is computed for all chunks of all heads at once by
// intra_kernel (chunk-parallel: every SM, two CTAs per SM) and stored as one
// "chunk record" per (chunk, head) in the workspace: the operand tiles the
// tensor cores need, already in their shared-memory image (tf32, K-major,
// 128-byte swizzle), plus Ut, e^m and e^{Gam_L}.  state_kernel then runs each
// head's serial chain: per chunk it streams the record into shared memory
// with bulk copies (the next chunk's tiles in flight during this chunk) and
// does only the state-dependent work -- the S_op / decay pass over the state
// in tensor memory and four tcgen05 MMAs.  The arithmetic is that of the
// one-kernel form in kda_chunk.cu (same operand roundings, same MMAs); only
// where the operands wait between the two phases differs.
#include "kda_chunk_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace chunk;

// ---- chunk record (one per (chunk, head)) -------------------------------------------
constexpr uint32_t REC_QT = 0;        // Qt: tf32 64 x 128, K-major sw128 image
constexpr uint32_t REC_WP = 32768;    // W': tf32 64 x 128 image
constexpr uint32_t REC_KH = 65536;    // Khat^T: tf32 128 x 64 image
constexpr uint32_t REC_AQ = 98304;    // A_qk: tf32 64 x 64 image (zero above the diagonal)
constexpr uint32_t REC_UT = 114688;   // Ut: fp32 [64 r][128 v]
constexpr uint32_t REC_EM = 147456;   // e^{m} [128], then e^{Gam_L} [128]
constexpr uint32_t kRecBytes = 148480;

// ---- intra kernel ---------------------------------------------------------------------
constexpr int kAThreads = 256;        // 8 warps: lane quarter w % 4, row half w / 4
constexpr uint32_t A_QK = 0;          // [Qt; Kr] tf32 128 x 128 (build .. MMA1), then:
constexpr uint32_t A_AKK = 0;         //   A_kk fp32 64 x 64 (akk_idx layout)
constexpr uint32_t A_T = 16384;       //   T fp32 64 x 64 row-major
constexpr uint32_t A_TB = 32768;      //   T beta tf32 image 64 x 64
constexpr uint32_t A_TB16 = 49152;    //   T beta bf16 high | low images
constexpr uint32_t A_KS = 65536;      // Ks tf32 64 x 128 (build .. MMA1), then:
constexpr uint32_t A_V = 65536;       //   V bf16 (TMA, two 64-wide swizzled boxes)
constexpr uint32_t A_AQ = 81920;      //   A_qk staging image, then:
constexpr uint32_t A_P = 81920;       //   float[4][256] inverse partial products
constexpr uint32_t A_TDIAG = 86016;   //   float[4][256] diagonal blocks of T
constexpr uint32_t A_MISC = 98304;
constexpr uint32_t AM_BETA = 0;       // float[64]
constexpr uint32_t AM_EM = 256;       // float[128]
constexpr uint32_t AM_DEC = 768;      // float[128]
constexpr uint32_t AM_PART = 1280;    // float[4][128] decay sums of the 16-row blocks
constexpr uint32_t AM_DIAG = 3328;    // float[4][256] diagonal blocks of A_kk, column-major
constexpr uint32_t AM_BAR = 7424;     // mbarriers: MMA, V
constexpr uint32_t AM_CTRL = 7440;    // int[4]: tmem base, unit, abort, decay flag
constexpr uint32_t kASmem = A_MISC + 7456;
constexpr uint32_t kASmemAlloc = kASmem + 1024;
// tensor memory (256 columns): D_A = [Qt; Kr] Ks^T, Kr^T, W'^T, Ut^T
constexpr uint32_t AT_A = 0, AT_W = 64, AT_O = 128, AT_U = 192;

struct IntraParams {
    const __nv_bfloat16 *q, *k;
    const float *g, *beta;        // unfused: log-decay [N,H,128], beta [N,H]
    const __nv_bfloat16 *f;       // fused gate: pre-activation [N,H,128]
    const void *blog;             // fused gate: beta logits [N,H]
    int blog_bf16;
    const float *A_log;
    int alog_mode;
    const float *dt_bias;
    const int32_t *cu_seqlens;
    int B;
    int64_t N;
    int H;
    float scale;
    int64_t num_slots;            // N / 64 + B
    uint8_t *records;
    unsigned int *counter;
    unsigned int *err;
};

// The sequence and chunk of a record slot: slots of sequence b start at
// floor(cu[b] / 64) + b (strictly increasing in b), so b is found by
// bisection.  Returns false for a slot that holds no chunk.
__device__ __forceinline__ bool slot_chunk(const int32_t *cu, int B, int64_t N, int64_t slot,
                                           int &b, int64_t &t0, int64_t &t1, int64_t &tc,
                                           bool &bad) {
    b = 0;
    t0 = 0;
    t1 = N;
    bad = false;
    if (cu != nullptr) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<int64_t>(cu[mid]) / kC + mid <= slot) lo = mid; else hi = mid - 1;
        }
        b = lo;
        t0 = cu[b];
        t1 = cu[b + 1];
        if (t0 < 0 || t1 < t0 || t1 > N) {
            bad = true;
            return false;
        }
    }
    const int64_t j = slot - (t0 / kC + b);
    tc = t0 + j * kC;
    return j >= 0 && tc < t1;
}

template <bool kGate>
__global__ void __launch_bounds__(kAThreads, 2) intra_kernel(const __grid_constant__ CUtensorMap tm_v,
                                                             const IntraParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *misc = smem + A_MISC;
    float *s_beta = reinterpret_cast<float *>(misc + AM_BETA);
    float *s_em = reinterpret_cast<float *>(misc + AM_EM);
    float *s_dec = reinterpret_cast<float *>(misc + AM_DEC);
    float *s_part = reinterpret_cast<float *>(misc + AM_PART);
    float *s_diag = reinterpret_cast<float *>(misc + AM_DIAG);
    uint64_t *bar_mma = reinterpret_cast<uint64_t *>(misc + AM_BAR);
    uint64_t *bar_v = bar_mma + 1;
    int *ctrl = reinterpret_cast<int *>(misc + AM_CTRL);
    float *Akk = reinterpret_cast<float *>(smem + A_AKK);
    float *Tm = reinterpret_cast<float *>(smem + A_T);
    float *s_P = reinterpret_cast<float *>(smem + A_P);
    float *s_tdiag = reinterpret_cast<float *>(smem + A_TDIAG);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int quarter = warp & 3, half = warp >> 2;
    const int ch = quarter * 32 + (tid & 31);   // channel / tensor-memory lane
    const int H = p.H;
    const int64_t num_units = p.num_slots * H;

    if (warp == 0) tmem_alloc(reinterpret_cast<uint32_t *>(&ctrl[0]), 256);
    if (tid == 0) {
        mbar_init(bar_mma, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
        prefetch_tmap(&tm_v);
        ctrl[2] = 0;
        ctrl[3] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(ctrl[0]);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint64_t d_qk = smem_desc(smem_addr(smem + A_QK), 16, 1024, kSwizzle128B);
    const uint64_t d_ks = smem_desc(smem_addr(smem + A_KS), 16, 1024, kSwizzle128B);
    const uint64_t d_tb = smem_desc(smem_addr(smem + A_TB), 16, 1024, kSwizzle128B);
    const uint64_t d_tb16 = smem_desc(smem_addr(smem + A_TB16), 16, 1024, kSwizzle128B);
    const uint64_t d_v = smem_desc(smem_addr(smem + A_V), 8192, 1024, kSwizzle128B);  // MN-major
    uint32_t ph_mma = 0, ph_v = 0;
    bool pend_v = false;
    const float kLog2e = 1.4426950408889634f;

    while (true) {
        __syncthreads();
        if (tid == 0) ctrl[1] = static_cast<int>(atomicAdd(p.counter, 1u));
        __syncthreads();
        const int64_t unit = static_cast<unsigned int>(ctrl[1]);
        if (unit >= num_units || ctrl[2] != 0) break;
        const int64_t slot = unit / H;
        const int h = static_cast<int>(unit % H);
        int b;
        int64_t t0, t1, tc;
        bool bad;
        if (!slot_chunk(p.cu_seqlens, p.B, p.N, slot, b, t0, t1, tc, bad)) {
            if (bad && tid == 0) record_device_error(p.err, kDevInvalidArg);
            continue;
        }
        const int L = static_cast<int>((t1 - tc) < kC ? (t1 - tc) : kC);
        uint8_t *rec = p.records + (slot * H + h) * static_cast<int64_t>(kRecBytes);

        // ---- cumulative decay (log2 units) of this thread's 32 rows ----
        float gam[32];
        {
            float gate_a = 0.f, gate_dt = 0.f;
            if (kGate) {
                const int ai = (p.alog_mode == 0) ? h : (p.alog_mode == 1 ? ch : h * kD + ch);
                gate_a = expf(p.A_log[ai]);
                gate_dt = p.dt_bias[h * kD + ch];
            }
            // summed per 16-row block, the blocks then combined in order: the
            // same additions, in the same order, as the one-kernel path
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int r = 32 * half + i;
                if (i == 16) {
                    s_part[(2 * half) * kD + ch] = acc;
                    acc = 0.f;
                }
                float g2 = 0.f;
                if (r < L) {
                    const int64_t idx = ((tc + r) * H + h) * kD + ch;
                    if (kGate) {
                        // log2(e) g = -exp(A_log) (log2(e) max(x, 0) + log2(1 + 2^{-log2(e)|x|})),
                        // x = f + dt_bias; log2(1 + e) as log2(u) e / (u - 1), u = 1 + e
                        // (D. Goldberg, "What every computer scientist should know about
                        // floating-point arithmetic", 1991)
                        const float x = __bfloat162float(p.f[idx]) + gate_dt;
                        const float e = fast_exp2(-kLog2e * fabsf(x));
                        const float u = 1.f + e;
                        float lg;
                        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(u));
                        lg = (u == 1.f) ? kLog2e * e : lg * __fdividef(e, u - 1.f);
                        g2 = -gate_a * (kLog2e * fmaxf(x, 0.f) + lg);
                    } else {
                        g2 = kLog2e * p.g[idx];
                    }
                }
                acc += g2;
                gam[i] = acc;
            }
            s_part[(2 * half + 1) * kD + ch] = acc;
            if (tid < kC) {
                float bt = 0.f;
                if (tid < L) {
                    const int64_t bi = (tc + tid) * H + h;
                    if (kGate) {
                        const float lg = p.blog_bf16
                                             ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p.blog)[bi])
                                             : static_cast<const float *>(p.blog)[bi];
                        bt = 1.f / (1.f + __expf(-lg));
                    } else {
                        bt = p.beta[bi];
                    }
                }
                s_beta[tid] = bt;
            }
        }
        __syncthreads();
        // prefix of each 16-row block and the chunk total, summed in block order
        float pre[2] = {0.f, 0.f}, gam_l = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < 4; ++g2) {
            const float pg = s_part[g2 * kD + ch];
            if (g2 < 2 * half) pre[0] += pg;
            if (g2 < 2 * half + 1) pre[1] += pg;
            gam_l += pg;
        }
        if (-gam_l > kMaxDecay * kLog2e) ctrl[3] = 1;
        const float m = 0.5f * gam_l;
        if (half == 0) {
            s_em[ch] = fast_exp2(m);
            s_dec[ch] = fast_exp2(gam_l);
        }
        const float ekh = fast_exp2(gam_l - m);

        // ---- operands: Qt, Kr (smem, MMA1), Ks (smem), Kr^T (TMEM); Qt and
        // Khat^T straight into the record ----
        {
            float krt[32];
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
                float khv[4];
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int i = 4 * i4 + e4;
                    const int r = 32 * half + i;
                    float qt = 0.f, kr = 0.f, ks = 0.f, kh = 0.f;
                    if (r < L) {
                        const int64_t idx = ((tc + r) * H + h) * kD + ch;
                        const float gr = pre[i >> 4] + gam[i];
                        const float e_up = fast_exp2(gr - m);   // e^{Gam_r - m}
                        const float e_dn = fast_exp2(m - gr);   // e^{m - Gam_r}
                        const float qv = __bfloat162float(p.q[idx]);
                        const float kv = __bfloat162float(p.k[idx]);
                        qt = to_tf32(p.scale * qv * e_up);
                        kr = to_tf32(kv * e_up);
                        ks = to_tf32(kv * e_dn);
                        kh = to_tf32(kv * (e_dn * ekh));
                    }
                    *reinterpret_cast<float *>(smem + A_QK + sw128_offset(r, ch, 128, 4)) = qt;
                    *reinterpret_cast<float *>(smem + A_QK + sw128_offset(r + 64, ch, 128, 4)) = kr;
                    *reinterpret_cast<float *>(smem + A_KS + sw128_offset(r, ch, 64, 4)) = ks;
                    *reinterpret_cast<float *>(rec + REC_QT + sw128_offset(r, ch, 64, 4)) = qt;
                    khv[e4] = kh;
                    krt[i] = kr;
                }
                *reinterpret_cast<float4 *>(rec + REC_KH + sw128_offset(ch, 32 * half + 4 * i4, 128, 4)) =
                    make_float4(khv[0], khv[1], khv[2], khv[3]);
            }
            tmem_st32(tmem + lane_base + AT_W + 32 * half, krt);
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- MMA1: D_A = [Qt; Kr] Ks^T ----
        if (tid == 0) {
            const uint32_t id = instr_desc(128, 64, kFmtTF32, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const uint64_t ad = d_qk + static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                const uint64_t bd = d_ks + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
                mma_tf32_ss(tmem + AT_A, ad, bd, id, kk > 0);
            }
            mma_commit(bar_mma);
        }
        cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid);
        ph_mma++;
        if (ctrl[2] != 0) break;
        // Ks is consumed: V of the chunk into its region
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_v, 16384);
            tma_load_3d(smem + A_V, &tm_v, bar_v, 0, h, static_cast<int32_t>(tc));
            tma_load_3d(smem + A_V + 8192, &tm_v, bar_v, 64, h, static_cast<int32_t>(tc));
            pend_v = true;
        }

        // ---- D_A epilogue: A_qk (staging image), A_kk (+ its diagonal blocks);
        // zero the T beta tiles (their strictly upper blocks stay zero) ----
        for (int e = tid; e < 32768 / 16; e += kAThreads)
            reinterpret_cast<float4 *>(smem + A_TB)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        {
            float d32[32];
            tmem_ld32(tmem + lane_base + AT_A + 32 * half, d32);
            tmem_wait_ld();
            if (quarter < 2) {
                const int r = ch;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int s = 32 * half + j;
                    *reinterpret_cast<float *>(smem + A_AQ + sw128_offset(r, s, 64, 4)) =
                        (s <= r) ? to_tf32(d32[j]) : 0.f;
                }
            } else {
                const int r = ch - 64;
                const float br = s_beta[r];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int s = 32 * half + j;
                    const float a = (s < r) ? br * d32[j] : 0.f;
                    Akk[akk_idx(r, s)] = a;
                    if ((r >> 4) == (s >> 4)) s_diag[(s >> 4) * 256 + (s & 15) * 16 + (r & 15)] = a;
                }
            }
        }
        __syncthreads();
        for (int e = tid; e < 16384 / 16; e += kAThreads)
            reinterpret_cast<float4 *>(rec + REC_AQ)[e] = reinterpret_cast<const float4 *>(smem + A_AQ)[e];
        __syncthreads();

        // ---- T = (I + A_kk)^{-1}, T beta into the operand tiles ----
        if (tid < 64) ut_diag_solve(s_diag, Tm, s_tdiag, smem + A_TB, smem + A_TB16, s_beta, tid);
        __syncthreads();
        ut_level1(Akk, s_tdiag, Tm, s_P, smem + A_TB, smem + A_TB16, s_beta, tid);
        ut_level2(Akk, Tm, s_P, smem + A_TB, smem + A_TB16, s_beta, tid);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- MMA2: W'^T = Kr^T (T beta)^T ;  Ut^T = V^T (T beta)^T ----
        if (tid == 0) {
            const uint32_t idw = instr_desc(128, 64, kFmtTF32, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bd = d_tb + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
                mma_tf32_ts(tmem + AT_O, tmem + AT_W + kk * 8, bd, idw, kk > 0);
            }
            if (!mbar_wait_bounded(bar_v, ph_v & 1, kMaxPolls)) {
                ctrl[2] = 1;
                record_device_error(p.err, kDevTimeout);
            } else {
                pend_v = false;
                const uint32_t idu = instr_desc(128, 64, kFmtBF16, 1, 0);
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = d_v + static_cast<uint64_t>((kk * 2048) >> 4);
                        const uint64_t bd = d_tb16 + static_cast<uint64_t>((part * 8192 + kk * 32) >> 4);
                        mma_f16_ss(tmem + AT_U, ad, bd, idu, (part | kk) != 0);
                    }
                }
            }
            mma_commit(bar_mma);
        }
        ph_v++;
        cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid);
        ph_mma++;
        if (ctrl[2] != 0) break;

        // ---- record: W' (tf32 image [r][k]), Ut ([r][v]), e^m, e^{Gam_L} ----
        {
            float w32[32];
            tmem_ld32(tmem + lane_base + AT_O + 32 * half, w32);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                *reinterpret_cast<float *>(rec + REC_WP + sw128_offset(32 * half + j, ch, 64, 4)) =
                    to_tf32(w32[j]);
            tmem_ld32(tmem + lane_base + AT_U + 32 * half, w32);
            tmem_wait_ld();
            float *ut = reinterpret_cast<float *>(rec + REC_UT);
#pragma unroll
            for (int j = 0; j < 32; ++j) ut[(32 * half + j) * kD + ch] = w32[j];
            if (tid < kD) {
                reinterpret_cast<float *>(rec + REC_EM)[tid] = s_em[tid];
                reinterpret_cast<float *>(rec + REC_EM)[kD + tid] = s_dec[tid];
            }
        }
        tc_fence_before();
    }

    // Drain: a V copy still in flight after an abort must land before exit.
    if (tid == 0) {
        if (pend_v) mbar_wait_bounded(bar_v, ph_v & 1, kMaxPolls);
        if (ctrl[3] != 0) record_device_error(p.err, kDevDecayRange);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---- state kernel -----------------------------------------------------------------------
constexpr int kBThreads = 512;        // 16 warps: lane quarter w % 4, column group w / 4
constexpr uint32_t B_XSTRIDE = 66560; // per buffer: Qt image, W' image, e^m | e^{Gam_L}
constexpr uint32_t BX_QT = 0, BX_WP = 32768, BX_ED = 65536;
constexpr uint32_t B_KH = 2 * B_XSTRIDE;        // Khat^T image
constexpr uint32_t B_AQ = B_KH + 32768;         // A_qk image
constexpr uint32_t B_MISC = B_AQ + 16384;
constexpr uint32_t BM_BAR = 0;        // mbarriers: a0, a1, b, mma
constexpr uint32_t BM_CTRL = 32;      // int[4]: tmem base, chain, abort
constexpr uint32_t kBSmem = B_MISC + 48;
constexpr uint32_t kBSmemAlloc = kBSmem + 1024;
// tensor memory (512 columns): S_acc = S^T, S_op, U^T, O^T of even / odd chunks
constexpr uint32_t BT_SACC = 0, BT_SOP = 128, BT_U = 256, BT_O0 = 320, BT_O1 = 384;

struct StateParams {
    const int32_t *cu_seqlens;
    int B;
    int64_t N;
    int H;
    const float *S0;
    float *Sf;
    void *o;
    const uint8_t *records;
    unsigned int *counter;
    unsigned int *err;
};

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

template <bool kOutBf16>
__global__ void __launch_bounds__(kBThreads, 1) state_kernel(const StateParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bar_a = reinterpret_cast<uint64_t *>(smem + B_MISC + BM_BAR);   // [2]
    uint64_t *bar_b = bar_a + 2;
    uint64_t *bar_mma = bar_a + 3;
    int *ctrl = reinterpret_cast<int *>(smem + B_MISC + BM_CTRL);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int quarter = warp & 3, grp = warp >> 2;
    const int ch = quarter * 32 + (tid & 31);
    const int H = p.H;
    const int num_chains = p.B * H;

    if (warp == 0) tmem_alloc(reinterpret_cast<uint32_t *>(&ctrl[0]), 512);
    if (tid == 0) {
        mbar_init(&bar_a[0], 1);
        mbar_init(&bar_a[1], 1);
        mbar_init(bar_b, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        ctrl[2] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(ctrl[0]);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    // (the two buffers' descriptors, phases and flags are scalars chosen with
    // ?: so that nothing is indexed by a runtime value and lands in local memory)
    const uint64_t d_qt0 = smem_desc(smem_addr(smem + BX_QT), 16, 1024, kSwizzle128B);
    const uint64_t d_qt1 = smem_desc(smem_addr(smem + B_XSTRIDE + BX_QT), 16, 1024, kSwizzle128B);
    const uint64_t d_wp0 = smem_desc(smem_addr(smem + BX_WP), 16, 1024, kSwizzle128B);
    const uint64_t d_wp1 = smem_desc(smem_addr(smem + B_XSTRIDE + BX_WP), 16, 1024, kSwizzle128B);
    const uint64_t d_kh = smem_desc(smem_addr(smem + B_KH), 16, 1024, kSwizzle128B);
    const uint64_t d_aq = smem_desc(smem_addr(smem + B_AQ), 16, 1024, kSwizzle128B);
    uint32_t ph_a0 = 0, ph_a1 = 0, ph_b = 0, ph_mma = 0;
    bool pend_a0 = false, pend_a1 = false, pend_b = false;

    while (true) {
        __syncthreads();
        if (tid == 0) ctrl[1] = static_cast<int>(atomicAdd(p.counter, 1u));
        __syncthreads();
        const int chain = ctrl[1];
        if (chain >= num_chains || ctrl[2] != 0) break;
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
        const int nck = static_cast<int>((t1 - t0 + kC - 1) / kC);
        const int64_t slot0 = t0 / kC + b;
        auto record = [&](int c) -> const uint8_t * {
            return p.records + ((slot0 + c) * H + h) * static_cast<int64_t>(kRecBytes);
        };
        auto issue_a = [&](int c, int x) {   // Qt, W', e^m | e^{Gam_L} of chunk c into buffer x
            const uint8_t *rec = record(c);
            uint8_t *dst = smem + x * B_XSTRIDE;
            mbar_arrive_expect_tx(&bar_a[x], 32768 + 32768 + 1024);
            bulk_load(dst + BX_QT, rec + REC_QT, 32768, &bar_a[x]);
            bulk_load(dst + BX_WP, rec + REC_WP, 32768, &bar_a[x]);
            bulk_load(dst + BX_ED, rec + REC_EM, 1024, &bar_a[x]);
            if (x) pend_a1 = true; else pend_a0 = true;
        };
        auto issue_b = [&](int c) {          // Khat^T, A_qk of chunk c
            const uint8_t *rec = record(c);
            mbar_arrive_expect_tx(bar_b, 32768 + 16384);
            bulk_load(smem + B_KH, rec + REC_KH, 32768, bar_b);
            bulk_load(smem + B_AQ, rec + REC_AQ, 16384, bar_b);
            pend_b = true;
        };
        // O^T of chunk c (rows r = 16 grp + j) from tensor memory to o
        auto write_output = [&](int c) {
            const int64_t tcw = t0 + static_cast<int64_t>(c) * kC;
            const int Lw = static_cast<int>((t1 - tcw) < kC ? (t1 - tcw) : kC);
            float o16[16];
            tmem_ld16(tmem + lane_base + ((c & 1) ? BT_O1 : BT_O0) + 16 * grp, o16);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = 16 * grp + j;
                if (r < Lw) {
                    const int64_t idx = ((tcw + r) * H + h) * kD + ch;
                    if (kOutBf16)
                        static_cast<__nv_bfloat16 *>(p.o)[idx] = __float2bfloat16_rn(o16[j]);
                    else
                        static_cast<float *>(p.o)[idx] = o16[j];
                }
            }
        };

        // initial state into S_acc (lane v, column k holds S[k][v])
        {
            float r32[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                r32[j] = (p.S0 != nullptr) ? p.S0[state_off + (32 * grp + j) * kD + ch] : 0.f;
            tmem_st32(tmem + lane_base + BT_SACC + 32 * grp, r32);
            tmem_wait_st();
        }
        if (tid == 0 && nck > 0) {
            issue_a(0, 0);
            issue_b(0);
        }

        for (int c = 0; c < nck; ++c) {
            const int x = c & 1;
            const uint8_t *rec = record(c);
            float u16[16];
            {
                const float *ut = reinterpret_cast<const float *>(rec + REC_UT);
#pragma unroll
                for (int j = 0; j < 16; ++j) u16[j] = ut[(16 * grp + j) * kD + ch];
            }
            if (tid == 0 && c + 1 < nck) issue_a(c + 1, x ^ 1);
            cta_wait(&bar_a[x], (x ? ph_a1 : ph_a0) & 1, &ctrl[2], p.err, tid);
            if (x) { ph_a1++; pend_a1 = false; } else { ph_a0++; pend_a0 = false; }
            if (ctrl[2] != 0) break;

            // ---- state pass: S_op = tf32(e^{m_k} S), S_acc = e^{Gam_L,k} S; Ut -> U ----
            {
                const float *em = reinterpret_cast<const float *>(smem + x * B_XSTRIDE + BX_ED);
                const float *dec = em + kD;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int c0 = 32 * grp + 16 * hh;
                    float r16[16], o16[16];
                    tmem_ld16(tmem + lane_base + BT_SACC + c0, r16);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        o16[j] = to_tf32(r16[j] * em[c0 + j]);
                        r16[j] = r16[j] * dec[c0 + j];
                    }
                    tmem_st16(tmem + lane_base + BT_SOP + c0, o16);
                    tmem_st16(tmem + lane_base + BT_SACC + c0, r16);
                }
                tmem_st16(tmem + lane_base + BT_U + 16 * grp, u16);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

            // ---- U^T -= S_op W'^T ;  O^T = S_op Qt^T ----
            if (tid == 0) {
                const uint32_t idn = instr_desc(128, 64, kFmtTF32, 0, 0, 1);
                const uint32_t ido = instr_desc(128, 64, kFmtTF32, 0, 0);
                const uint32_t to = tmem + (x ? BT_O1 : BT_O0);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint64_t bw = (x ? d_wp1 : d_wp0) + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
                    mma_tf32_ts(tmem + BT_U, tmem + BT_SOP + kk * 8, bw, idn, 1);
                }
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint64_t bq = (x ? d_qt1 : d_qt0) + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
                    mma_tf32_ts(to, tmem + BT_SOP + kk * 8, bq, ido, kk > 0);
                }
                mma_commit(bar_mma);
            }
            if (c > 0) write_output(c - 1);
            cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid);
            ph_mma++;
            if (ctrl[2] != 0) break;

            // ---- U rounded to tf32 in place (A operand of the next MMAs) ----
            {
                float v16[16];
                tmem_ld16(tmem + lane_base + BT_U + 16 * grp, v16);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) v16[j] = to_tf32(v16[j]);
                tmem_st16(tmem + lane_base + BT_U + 16 * grp, v16);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            cta_wait(bar_b, ph_b & 1, &ctrl[2], p.err, tid);
            ph_b++;
            if (tid == 0) pend_b = false;
            if (ctrl[2] != 0) break;

            // ---- S_acc^T += U^T Khat ;  O^T += U^T A_qk^T ----
            if (tid == 0) {
                const uint32_t ids = instr_desc(128, 128, kFmtTF32, 0, 0);
                const uint32_t ido = instr_desc(128, 64, kFmtTF32, 0, 0);
                const uint32_t to = tmem + (x ? BT_O1 : BT_O0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t bk = d_kh + static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    mma_tf32_ts(tmem + BT_SACC, tmem + BT_U + kk * 8, bk, ids, 1);
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ba = d_aq + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
                    mma_tf32_ts(to, tmem + BT_U + kk * 8, ba, ido, 1);
                }
                mma_commit(bar_mma);
            }
            cta_wait(bar_mma, ph_mma & 1, &ctrl[2], p.err, tid);
            ph_mma++;
            if (ctrl[2] != 0) break;
            if (tid == 0 && c + 1 < nck) issue_b(c + 1);
        }
        if (ctrl[2] != 0) break;
        if (nck > 0) write_output(nck - 1);

        if (p.Sf != nullptr) {
            float r32[32];
            tmem_ld32(tmem + lane_base + BT_SACC + 32 * grp, r32);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) p.Sf[state_off + (32 * grp + j) * kD + ch] = r32[j];
        }
        tc_fence_before();
    }

    // Drain: bulk copies still in flight after an abort must land before exit.
    if (tid == 0) {
        if (pend_a0) mbar_wait_bounded(&bar_a[0], ph_a0 & 1, kMaxPolls);
        if (pend_a1) mbar_wait_bounded(&bar_a[1], ph_a1 & 1, kMaxPolls);
        if (pend_b) mbar_wait_bounded(bar_b, ph_b & 1, kMaxPolls);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <bool kGate>
cudaError_t launch_split(const __nv_bfloat16 *v, const IntraParams &ip, const StateParams &sp,
                         bool o_bf16, int num_sms, cudaStream_t s) {
    if (ip.B == 0 || ip.H == 0) return cudaSuccess;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(intra_kernel<kGate>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kASmemAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(state_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kBSmemAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(state_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kBSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    CUtensorMap mv;
    const int64_t Nmap = ip.N > 0 ? ip.N : 1;
    if (!make_map(&mv, v, Nmap, ip.H, 64, true)) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(ip.counter, 0, 2 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    const int64_t units = ip.num_slots * ip.H;
    const int64_t agrid = units < 2 * num_sms ? units : 2 * num_sms;
    if (agrid > 0) intra_kernel<kGate><<<static_cast<int>(agrid), kAThreads, kASmemAlloc, s>>>(mv, ip);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int chains = sp.B * sp.H;
    const int bgrid = chains < num_sms ? chains : num_sms;
    if (o_bf16)
        state_kernel<true><<<bgrid, kBThreads, kBSmemAlloc, s>>>(sp);
    else
        state_kernel<false><<<bgrid, kBThreads, kBSmemAlloc, s>>>(sp);
    return cudaGetLastError();
}

}  // namespace

// Workspace of the two-phase prefill: 256 bytes of counters, then one chunk
// record per (slot, head) with slots = N / 64 + B.
size_t prefill_split_workspace_bytes(int64_t N, int B, int H) {
    if (N < 0 || B < 1 || H < 1) return 0;
    const size_t slots = static_cast<size_t>(N / kC) + static_cast<size_t>(B);
    return 256 + slots * static_cast<size_t>(H) * kRecBytes;
}

cudaError_t launch_prefill_split(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                 const __nv_bfloat16 *v, const float *g, const float *beta,
                                 const __nv_bfloat16 *f, const void *blog, bool blog_bf16,
                                 const float *A_log, int alog_mode, const float *dt_bias,
                                 const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
                                 const float *initial_state, float *final_state, void *o,
                                 bool o_bf16, void *workspace, unsigned int *err, int num_sms,
                                 cudaStream_t s) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    IntraParams ip;
    ip.q = q; ip.k = k; ip.g = g; ip.beta = beta;
    ip.f = f; ip.blog = blog; ip.blog_bf16 = blog_bf16 ? 1 : 0;
    ip.A_log = A_log; ip.alog_mode = alog_mode; ip.dt_bias = dt_bias;
    ip.cu_seqlens = cu_seqlens; ip.B = B; ip.N = N; ip.H = H; ip.scale = scale;
    ip.num_slots = N / kC + B;
    ip.records = ws + 256;
    ip.counter = reinterpret_cast<unsigned int *>(ws);
    ip.err = err;
    StateParams sp;
    sp.cu_seqlens = cu_seqlens; sp.B = B; sp.N = N; sp.H = H;
    sp.S0 = initial_state; sp.Sf = final_state; sp.o = o;
    sp.records = ws + 256;
    sp.counter = reinterpret_cast<unsigned int *>(ws) + 1;
    sp.err = err;
    return (f != nullptr) ? launch_split<true>(v, ip, sp, o_bf16, num_sms, s)
                          : launch_split<false>(v, ip, sp, o_bf16, num_sms, s);
}

}  // namespace kda

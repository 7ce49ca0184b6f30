// kda_chunk_bwd.cu -- chunked KDA backward on tcgen05 tensor cores (sm_103a).
//
// The training regime of Kimi Delta Attention in chunked form
// (data/code-audit.json, finding "dual-kda-execution-regimes": chunked KDA for
// prefill and training).  The pages print no gradient; this is the exact
// reverse mode of the chunk-level forward of kda_chunk.cu.  For one chunk of
// L <= 64 tokens of one (sequence, head) with start state S (k x v), the
// chunk-end state gradient dS' and the output gradient dO, with the per-channel
// reference m = Gam_L / 2 and the referenced operands
//   Qt = scale q e^{Gam - m}, Kr = k e^{Gam - m}, Ks = k e^{m - Gam},
//   Kh = k e^{Gam_L - Gam},  S_op = Diag(e^m) S,
//   A_qk = tril(Qt Ks^T),  kk = Kr Ks^T,  A_kk = strict_tril(diag(beta) kk),
//   T = (I + A_kk)^{-1},  W' = T diag(beta) Kr,  Ut = T diag(beta) V,
//   U = Ut - W' S_op,
// the gradients are
//   dU    = A_qk^T dO + Kh dS'
//   dS    = Diag(e^{Gam_L}) dS' + Diag(e^m) (Qt^T dO - W'^T dU)      (to the previous chunk)
//   dA_qk = tril(dO U^T),  dQt = dO S_op^T + dA_qk Ks,  dW' = -dU S_op^T,
//   dKh   = U dS'^T,
//   dT    = (dW' Kr^T + dU V^T) diag(beta),  d(beta Kr) = T^T dW',  d(beta V) = T^T dU,
//   dA_kk = -strict_tril(T^T dT T^T),
//   dKs   = dA_qk^T Qt + (diag(beta) dA_kk)^T Kr,  dKr = diag(beta) (dA_kk Ks + d(beta Kr)),
//   dbeta = rowsum(dA_kk . kk) + rowsum(d(beta Kr) . Kr) + rowsum(d(beta V) . V),
//   dv = diag(beta) d(beta V),  dq = scale dQt e^{Gam - m},
//   dk = dKr e^{Gam - m} + dKs e^{m - Gam} + dKh e^{Gam_L - Gam},
//   dGam = dKr.Kr - dKs.Ks - dKh.Kh + dQt.Qt,
//   dGam_L += colsum(dKh.Kh) + rowsum_v(dS' . Diag(e^{Gam_L}) S),
//   dg = the reverse cumulative sum of dGam over the chunk's tokens.
// (The e^{+-m} factors cancel in every product, so these equal the
// unreferenced formulas term by term.)
//
// Products.  Every matrix above is stored once, as an "image": a bf16 tile
// pair hi = bf16(x), lo = bf16(x - hi) in the 128-byte-swizzled layout of a
// [rows][cols] operand tile (cols in blocks of 64).  bf16 tcgen05 operands may
// be K-major or MN-major, so one image serves a matrix and its transpose, and
// every product is three kind::f16 MMAs per k-step (hi.hi + hi.lo + lo.hi, a
// 16-bit mantissa; the raw bf16 inputs are exact and need no low part).
// Images live in a per-CTA scratch area of the workspace (about 530 KB, L2
// resident); a product copies the rows it reads of its two operand images into
// two 64 KB shared slots (16-byte cp.async by every thread) unless a slot
// already holds them, runs its MMAs into tensor memory, and an epilogue writes
// the result's image(s), mostly into a slot whose operand is dead, and copies
// it to the scratch from there.  The chain's state gradient dS stays in
// tensor memory in fp32 for the whole sequence.
//
// The chunk-start states S come from the forward prefill kernel, which writes
// them to the workspace (fp32 [k][v] per chunk) when asked; chains whose
// forward pass had to shorten a chunk (a per-channel chunk decay beyond the
// represented range) have no 64-token-aligned states: they are reported as
// KDA_ERR_DECAY_RANGE and their gradients are written as zeros.
//
// Work decomposition: one CTA of 512 threads per (sequence, head) chain at a
// time, chains from a counter, chunks last to first.  Warp w serves lane
// quarter w % 4 (tensor-memory lanes 32 (w % 4) .. + 31, also the channel of
// the element-wise passes) and group w / 4 (16 chunk rows / columns).
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"
#include "kda_chunk_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace chunk;

constexpr int kThreads = 512;

// ---- operand images in the per-CTA scratch ----------------------------------------------
// rows x cols, split (hi tile then lo tile) unless exact; every size a multiple of 8 KB.
enum Img : int {
    I_QK,    // [128][128] rows 0-63 Qt (later dW'), rows 64-127 Kr
    I_KS,    // [64][128]  Ks
    I_KH,    // [64][128]  Kh
    I_V,     // [64][128]  v (exact bf16)
    I_TB,    // [64][64]   T diag(beta)
    I_T,     // [64][64]   T
    I_AQ,    // [64][64]   A_qk
    I_WT,    // [128][64]  -W'^T
    I_UT,    // [128][64]  U^T
    I_SO,    // [128][128] S_op^T: row v holds e^{m_k} S[k][v] over k
    I_DS,    // [128][128] dS'^T: row v holds dS'[k][v] over k (chunk-end state gradient)
    I_DU2,   // [128][128] rows 0-63 dU, rows 64-127 dO
    I_DAQ,   // [64][64]   dA_qk
    I_DT,    // [64][64]   dT
    I_Y,     // [64][64]   dT T^T
    I_DKK,   // [64][64]   dA_kk
    I_BDKK,  // [64][64]   diag(beta) dA_kk
    kNumImg
};
__host__ __device__ constexpr uint32_t img_rows(int i) {
    return (i == I_QK || i == I_WT || i == I_UT || i == I_SO || i == I_DS || i == I_DU2) ? 128 : 64;
}
__host__ __device__ constexpr uint32_t img_cols(int i) {
    return (i == I_TB || i == I_T || i == I_AQ || i == I_WT || i == I_UT || i == I_DAQ ||
            i == I_DT || i == I_Y || i == I_DKK || i == I_BDKK)
               ? 64
               : 128;
}
__host__ __device__ constexpr bool img_exact(int i) { return i == I_V; }
// bytes of one bf16 tile of the image (hi or lo)
__host__ __device__ constexpr uint32_t img_half(int i) { return img_rows(i) * img_cols(i) * 2; }
__host__ __device__ constexpr uint32_t img_bytes(int i) {
    return img_exact(i) ? img_half(i) : 2 * img_half(i);
}
__host__ __device__ constexpr uint32_t img_off(int i) {
    uint32_t o = 0;
    for (int j = 0; j < i; ++j) o += img_bytes(j);
    return o;
}
constexpr uint32_t kScratchPerCta = img_off(kNumImg);  // 540672

// ---- shared memory (bytes from a 1024-aligned base) -------------------------------------
constexpr uint32_t SLOT_A = 0;            // operand slot, 64 KB
constexpr uint32_t SLOT_B = 65536;        // operand slot, 64 KB
constexpr uint32_t OFF_AT = 131072;       // A_kk column-major fp32 [64][64]; q staged outside the inverse
constexpr uint32_t OFF_TT = 147456;       // T row-major fp32 (inverse work area)
constexpr uint32_t OFF_KK = 163840;       // kk fp32 [64][64] column-major
constexpr uint32_t OFF_MISC = 180224;
constexpr uint32_t M_BETA = 0;            // float[64]
constexpr uint32_t M_EM = 256;            // float[128] e^{m}
constexpr uint32_t M_DEC = 768;           // float[128] e^{Gam_L}
constexpr uint32_t M_PART = 1280;         // float[4][128] partial decay sums per row group
constexpr uint32_t M_DGL = 3328;          // float[128] sum_v dS'[k][v] S[k][v]
constexpr uint32_t M_SUF = 4096;          // float[4][128] dGam sums per row group; before
                                          // the assembly the per-quarter parts of M_DGL
constexpr uint32_t M_P = 6144;            // float[4][256] inverse partial products; after
                                          // the inverse the parts of dbeta ([8][64]) and of
                                          // colsum(dKh . Kh) ([4][128])
constexpr uint32_t M_T32 = 10240;         // float[16][16]
constexpr uint32_t M_TDIAG = 11264;       // float[4][16][16]
constexpr uint32_t M_BAR = 15360;         // the product mbarrier
constexpr uint32_t M_CTRL = 15376;        // int[8]: tmem base, chain, abort
constexpr uint32_t M_GL = 15936;          // float[128] Gam_L (log2 units)
constexpr uint32_t OFF_STG = OFF_MISC + 16448;  // k, v bf16 [64][128] each, the whole chunk
constexpr uint32_t kSmemBytes = OFF_STG + 32768;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

// ---- tensor memory columns (lane = M row of each product) ----
constexpr uint32_t C_DS = 0;      // dS^T fp32 (lane v, column k), the chain
constexpr uint32_t C_VB = 128;    // d(beta V)^T (lane v, column r)            transient
constexpr uint32_t C_H = 192;     // dKh^T (lane k, column r)
constexpr uint32_t C_S = 256;     // dKs^T (lane k, column s)
constexpr uint32_t C_R = 320;     // d(beta Kr)^T + (dA_kk Ks)^T (lane k, column r)
constexpr uint32_t C_TA = 384;    // transient 64 columns
constexpr uint32_t C_TB = 448;    // Ut^T -> U^T, later dQt^T (lane k, column r)

struct BwdParams {
    const __nv_bfloat16 *q, *k, *v;
    const float *g, *beta;
    const int32_t *cu_seqlens;
    int B;
    int64_t N;
    int H;
    float scale;
    const void *dO;
    int dO_bf16;
    const float *dSf;
    const float *ckpt;      // chunk-start states from the forward pass
    const int *split;       // per chain: the forward pass shortened a chunk
    float *dq, *dk, *dv, *dg, *dbeta, *dS0;
    uint8_t *scratch;       // kScratchPerCta bytes per CTA
    unsigned int *counter;
    unsigned int *err;
    uint32_t polls;
};

// ---- image stores (generic pointers into the global scratch) ------------------------------

__device__ __forceinline__ void put1(uint8_t *img, uint32_t half, uint32_t rows, int i, int j,
                                     float x) {
    const uint32_t o = sw128_offset(i, j, rows, 2);
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    *reinterpret_cast<__nv_bfloat16 *>(img + o) = hi;
    if (half != 0)
        *reinterpret_cast<__nv_bfloat16 *>(img + half + o) =
            __float2bfloat16_rn(x - __bfloat162float(hi));
}

// eight consecutive columns j0 .. j0 + 7 (j0 % 8 == 0) of row i: one 16-byte chunk each
__device__ __forceinline__ void put8(uint8_t *img, uint32_t half, uint32_t rows, int i, int j0,
                                     const float *x) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
        hw[e] = *reinterpret_cast<const uint32_t *>(&h);
        lw[e] = *reinterpret_cast<const uint32_t *>(&l);
    }
    const uint32_t o = sw128_offset(i, j0, rows, 2);
    *reinterpret_cast<uint4 *>(img + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (half != 0) *reinterpret_cast<uint4 *>(img + half + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// ---- product issue ---------------------------------------------------------------------

// One operand of a product: an image (or a row range of it) in a shared slot.
// K-major: rows are M / N, `blk` the bytes between 64-column K blocks.
// MN-major: rows are K, `blk` the bytes between 64-column M / N blocks (LBO).
struct Opd {
    uint32_t hi;       // shared address of the hi tile
    uint32_t hi_lo;    // bytes from the hi tile to the lo tile
    bool has_lo;       // false: an exact bf16 image (no lo tile)
    uint32_t blk;
    uint32_t mn;
};

__device__ __forceinline__ Opd opd(uint32_t slot, int img, uint32_t row0, bool mn) {
    Opd o;
    o.hi = slot + row0 * 128;
    o.hi_lo = img_half(img);
    o.has_lo = !img_exact(img);
    o.blk = img_rows(img) * 128;
    o.mn = mn ? 1u : 0u;
    return o;
}

__device__ __forceinline__ uint64_t desc0(const Opd &o, uint32_t base) {
    return smem_desc(base, o.mn ? o.blk : 16u, 1024, kSwizzle128B);
}

// D[tmem d] (+)= A B over `ksteps` k-steps of 16 (a multiple of 4; M = 128, N
// columns), as hi.hi + hi.lo + lo.hi per k-step, issued by one elected lane of
// the converged warp 0.  Each descriptor's low word (the start address) steps
// by a constant: 32 bytes per k-step for a K-major operand, with a jump to the
// next 64-column block after every fourth step, and eight 256-byte rows per
// k-step for an MN-major one.  The loop holds little besides the MMAs: every
// instruction of the issuing warp delays the next MMA, and an N = 64 or 128
// MMA completes in about 50 cycles, less than a longer issue path takes to
// produce it.  The loop stays rolled: the kernel is bound by its instruction
// cache, and every unrolled copy of this loop costs more than it saves.
__device__ __forceinline__ void issue(uint32_t d, const Opd &A, const Opd &B, uint32_t N, int ksteps,
                                      bool accumulate) {
    const uint32_t id = instr_desc(128, N, kFmtBF16, A.mn, B.mn);
    const uint64_t a0 = desc0(A, A.hi), b0 = desc0(B, B.hi);
    const uint32_t dh_a = static_cast<uint32_t>(a0 >> 32), dh_b = static_cast<uint32_t>(b0 >> 32);
    uint32_t ah = static_cast<uint32_t>(a0), bh = static_cast<uint32_t>(b0);
    uint32_t al = ah + (A.hi_lo >> 4), bl = bh + (B.hi_lo >> 4);
    const uint32_t sa = A.mn ? 128u : 2u, sb = B.mn ? 128u : 2u;
    const uint32_t ja = A.mn ? 512u : (A.blk >> 4), jb = B.mn ? 512u : (B.blk >> 4);
    auto dsc = [](uint32_t hi, uint32_t lo) { return (static_cast<uint64_t>(hi) << 32) | lo; };
    uint32_t acc = accumulate ? 1u : 0u;
    // after the fourth step of a block: to the next block
    const uint32_t ea = ja - 3 * sa, eb = jb - 3 * sb;
#pragma unroll 1
    for (int kk = 0; kk < ksteps; ++kk) {
        mma_f16_ss_w(d, dsc(dh_a, ah), dsc(dh_b, bh), id, acc);
        acc = 1u;
        if (B.has_lo) mma_f16_ss_w(d, dsc(dh_a, ah), dsc(dh_b, bl), id, 1u);
        if (A.has_lo) mma_f16_ss_w(d, dsc(dh_a, al), dsc(dh_b, bh), id, 1u);
        const bool last = (kk & 3) == 3;
        const uint32_t da = last ? ea : sa, db = last ? eb : sb;
        ah += da; al += da; bh += db; bl += db;
    }
}

// One halving step of a sum across lanes: lanes with bit `off` set keep the
// upper N of their 2N values, the others the lower N, each adding its
// partner's copy of the half it keeps.
template <int N>
__device__ __forceinline__ void fold(float *x, int lane, int off) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float a = x[i], b = x[i + N];
        x[i] = (up ? b : a) + __shfl_xor_sync(0xffffffffu, up ? a : b, off);
    }
}

// Sums over the 32 lanes of a warp of 16 values per lane: on return x[0] of
// lane l holds the total of value l >> 1 (16 shuffles instead of 16 x 5).
__device__ __forceinline__ float lanes_sum16(float (&x)[16], int lane) {
    fold<8>(x, lane, 16);
    fold<4>(x, lane, 8);
    fold<2>(x, lane, 4);
    fold<1>(x, lane, 2);
    return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 1);
}

// The product engine's state (identical in every thread): the image each of
// the two operand slots holds (-1: none) and which of its rows, the product
// barrier's phase, and whether a product is in flight (for the drain).
struct Sched {
    uint8_t *smem, *scr;
    uint64_t *bar_mma;
    int *abort_flag;
    unsigned int *err;
    uint32_t polls, sa, sb;
    int tid;
    int sl0, sl1;
    int lo0, hi0, lo1, hi1;  // the rows of its image each slot holds
    // one more image per slot, in its own byte layout from an offset past the
    // first image's (loaded under a product for the next one)
    int xi0, xlo0, xhi0, xi1, xlo1, xhi1;
    uint32_t xoff0, xoff1;
    uint32_t ph_mma;
    bool pend_mma;
    bool pend_copy;  // a preloaded operand's copies may still be in flight
};

// An operand: image, first row used, MN-major.
struct OpSpec {
    int img, row0, mn;
};

__device__ __forceinline__ void clear_extra(Sched &S) {
    S.xi0 = S.xi1 = -1;
    S.xoff0 = S.xoff1 = 0;
}

__device__ __forceinline__ void dirty(Sched &S, int i) {
    if (S.sl0 == i) S.sl0 = -1;
    if (S.sl1 == i) S.sl1 = -1;
    if (S.xi0 == i) S.xi0 = -1;
    if (S.xi1 == i) S.xi1 = -1;
}

__device__ __forceinline__ uint8_t *slot_ptr(const Sched &S, int sl) {
    return S.smem + (sl ? SLOT_B : SLOT_A);
}

// Slot `sl` holds rows [lo, hi) of image i (from its start); the images
// placed further on that it overlaps are gone.
__device__ __forceinline__ void set_slot(Sched &S, int sl, int i, int lo, int hi) {
    if (sl) {
        S.sl1 = i; S.lo1 = lo; S.hi1 = hi;
    } else {
        S.sl0 = i; S.lo0 = lo; S.hi0 = hi;
    }
    if (sl) {
        if (S.xoff1 < img_bytes(i)) S.xi1 = -1;
    } else {
        if (S.xoff0 < img_bytes(i)) S.xi0 = -1;
    }
}

// The slot holding rows [lo, hi) of image i and the byte offset of its
// layout there (kExtra: the second images too), or -1.
template <bool kExtra>
__device__ __forceinline__ int find_img(const Sched &S, int i, int lo, int hi, uint32_t &off) {
    off = 0;
    if (S.sl0 == i && S.lo0 <= lo && hi <= S.hi0) return 0;
    if (S.sl1 == i && S.lo1 <= lo && hi <= S.hi1) return 1;
    if (kExtra) {
        if (S.xi0 == i && S.xlo0 <= lo && hi <= S.xhi0) {
            off = S.xoff0;
            return 0;
        }
        if (S.xi1 == i && S.xlo1 <= lo && hi <= S.xhi1) {
            off = S.xoff1;
            return 1;
        }
    }
    return -1;
}

// The slot holding image i (any of its rows, any placement), or -1.
__device__ __forceinline__ int slot_of(const Sched &S, int i) {
    uint32_t off;
    return find_img<true>(S, i, 0x7fff, 0, off);
}

// Slot `sl` holds rows [lo, hi) of image i in the image's layout from byte
// `off`; whatever it overlaps in the slot is gone.
__device__ __forceinline__ void place_extra(Sched &S, int sl, int i, int lo, int hi, uint32_t off) {
    const int p = sl ? S.sl1 : S.sl0;
    if (p >= 0 && off < img_bytes(p)) {
        if (sl) S.sl1 = -1; else S.sl0 = -1;
    }
    if (sl) {
        S.xi1 = i; S.xlo1 = lo; S.xhi1 = hi; S.xoff1 = off;
    } else {
        S.xi0 = i; S.xlo0 = lo; S.xhi0 = hi; S.xoff0 = off;
    }
}
// Every thread copies 16-byte pieces between a slot and the image in the
// scratch: rows [r0, r1) of each 64-column block of the hi (and lo) tile, in
// the image's byte layout; cp.async into the slot (load) or plain 16-byte
// stores to the scratch (store).
template <bool kLoad>
__device__ __forceinline__ void copy_rows(const Sched &S, int sl, int i, uint32_t r0, uint32_t r1,
                                          uint32_t off = 0) {
    uint8_t *slot = slot_ptr(S, sl) + off;
    uint8_t *glob = S.scr + img_off(i);
    const uint32_t rows = img_rows(i);
    if (r0 == 0 && r1 == rows) {
        for (uint32_t u = S.tid; u < img_bytes(i) / 16; u += kThreads) {
            if (kLoad)
                cp_async_16(slot + u * 16, glob + u * 16, true);
            else
                *reinterpret_cast<uint4 *>(glob + u * 16) = *reinterpret_cast<const uint4 *>(slot + u * 16);
        }
        return;
    }
    // in each (tile, 64-column block) the rows are one contiguous range
    const uint32_t pieces = (r1 - r0) * 8;
#pragma unroll 1
    for (uint32_t q = 0; q < (img_exact(i) ? 1u : 2u) * (img_cols(i) / 64); ++q) {
        const uint32_t base = q * rows * 128 + r0 * 128;  // the lo tile follows the hi tile's blocks
        for (uint32_t u = S.tid; u < pieces; u += kThreads) {
            if (kLoad)
                cp_async_16(slot + base + u * 16, glob + base + u * 16, true);
            else
                *reinterpret_cast<uint4 *>(glob + base + u * 16) =
                    *reinterpret_cast<const uint4 *>(slot + base + u * 16);
        }
    }
}

// After an epilogue wrote image `i` (or the row range [r0, r1) of it) into slot
// `sl` in the image's own byte layout: makes the writes visible to the async
// proxy (the tensor core reads the slot), and the CTA copies the written bytes
// to the image in the scratch.  A whole image stays in the slot for the next
// products.
__device__ __forceinline__ void stage_store(Sched &S, int sl, int i, uint32_t r0, uint32_t r1) {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int rows = static_cast<int>(img_rows(i));
    copy_rows<false>(S, sl, i, r0, r1);
    // the slot's rows of image i: the written ones, with those it held if the
    // two ranges touch; any other slot's copy of the image is stale
    int lo = static_cast<int>(r0), hi = static_cast<int>(r1);
    const bool had = sl ? S.sl1 == i : S.sl0 == i;
    const int plo = sl ? S.lo1 : S.lo0, phi = sl ? S.hi1 : S.hi0;
    if (had && plo <= hi && lo <= phi) {
        lo = min(lo, plo);
        hi = max(hi, phi);
    }
    set_slot(S, sl, i, lo, hi);
    if (!(r0 == 0 && static_cast<int>(r1) == rows)) {
        if (sl && S.sl0 == i) S.sl0 = -1;
        if (!sl && S.sl1 == i) S.sl1 = -1;
    }
    if (S.xi0 == i) S.xi0 = -1;
    if (S.xi1 == i) S.xi1 = -1;
}

// As stage_store for an image that only the next products read, from the
// slot: no copy to the scratch (the scratch's copy stays stale, so no later
// product may miss it in the slot).
__device__ __forceinline__ void stage_only(Sched &S, int sl, int i, int r0, int r1) {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    set_slot(S, sl, i, r0, r1);
}

// An operand image to bring in while a product runs, for the products after
// it: rows [lo, hi) of image img, in its own layout from byte `off` of the
// slot that holds the product's A (rel 0) or B (rel 1) operand, or of the slot
// the product does not read (rel 2, for a product whose operands share one).
struct Pre {
    int img, lo, hi, rel;
    uint32_t off;
};

// One product term, D[tmem d] (+)= A B: copies the operand images that are not
// already in a slot (a slot keeps its images until they are overwritten or
// rewritten), issues the MMAs from warp 0, starts the copies of `pre` while
// they run, and waits for the MMAs.  Returns false when a wait ran out (the
// CTA is aborting).
template <bool kExtra = false>
__device__ __forceinline__ bool product(Sched &S, OpSpec A, OpSpec B, uint32_t d, uint32_t N,
                                     int ksteps, bool accumulate, int a_lo = 0, int a_hi = 128,
                                     const Pre *pre = nullptr) {
    const int ia = A.img, ib = B.img;
    // the rows each operand reads: K rows for an MN-major operand, the M rows
    // whose results are used (a_lo .. a_hi) for A, N rows for B
    int alo = A.mn ? A.row0 : A.row0 + a_lo, ahi = A.mn ? A.row0 + 16 * ksteps : A.row0 + a_hi;
    int blo = B.row0, bhi = B.row0 + (B.mn ? 16 * ksteps : static_cast<int>(N));
    ahi = min(ahi, static_cast<int>(img_rows(ia)));
    bhi = min(bhi, static_cast<int>(img_rows(ib)));
    if (ia == ib) {
        alo = blo = min(alo, blo);
        ahi = bhi = max(ahi, bhi);
    }
    uint32_t fa, fb;  // byte offsets of the operands' layouts in their slots
    int pa = find_img<kExtra>(S, ia, alo, ahi, fa);
    int pb = find_img<kExtra>(S, ib, blo, bhi, fb);
    int la = -1, lb = -1;
    if (pa < 0) {  // loaded at the start of the slot the other operand is not in
        pa = (pb == 0) ? 1 : 0;
        la = pa;
        fa = 0;
    }
    if (ib == ia) {
        pb = pa;
        fb = fa;
    }
    if (pb < 0) {
        pb = (pa == 0) ? 1 : 0;
        lb = pb;
        fb = 0;
    }
    if (la >= 0 || lb >= 0 || S.pend_copy) {
        // the rows it reads of each image not in a slot, by cp.async (the
        // images were written by this CTA's threads before a barrier), and
        // any preloaded rows
        if (la >= 0) copy_rows<true>(S, la, ia, alo, ahi);
        if (lb >= 0) copy_rows<true>(S, lb, ib, blo, bhi);
        cp_async_wait_all();
        fence_proxy_async_smem();  // read by the tensor core
        __syncthreads();
        if (la >= 0) set_slot(S, la, ia, alo, ahi);
        if (lb >= 0) set_slot(S, lb, ib, blo, bhi);
        S.pend_copy = false;
    }
    if (S.tid < 32) {
        __syncwarp();
        issue(d, opd((pa ? S.sb : S.sa) + fa, ia, A.row0, A.mn != 0),
              opd((pb ? S.sb : S.sa) + fb, ib, B.row0, B.mn != 0), N, ksteps, accumulate);
        mma_commit_w(S.bar_mma);
    }
    if (pre != nullptr) {  // into bytes of the slots this product does not read
        const int sl = pre->rel == 0 ? pa : pre->rel == 1 ? pb : 1 - pa;
        copy_rows<true>(S, sl, pre->img, static_cast<uint32_t>(pre->lo), static_cast<uint32_t>(pre->hi),
                        pre->off);
        place_extra(S, sl, pre->img, pre->lo, pre->hi, pre->off);
        S.pend_copy = true;
    }
    S.pend_mma = true;
    if (!cta_wait(S.bar_mma, S.ph_mma & 1, S.abort_flag, S.err, S.tid, S.polls)) return false;
    S.ph_mma++;
    S.pend_mma = false;
    return true;
}

// Starts copying rows [r0, r1) of image i into slot sl for the next product,
// under the epilogue in between: the slot's operand is dead and nothing else
// writes the slot before that product, which waits for the copies.  Called
// by every thread after a product's completion (its barrier orders the copy
// after every read of the slot).
__device__ __forceinline__ void preload(Sched &S, int sl, int i, int r0, int r1) {
    copy_rows<true>(S, sl, i, static_cast<uint32_t>(r0), static_cast<uint32_t>(r1));
    set_slot(S, sl, i, r0, r1);
    S.pend_copy = true;
}

__global__ void __launch_bounds__(kThreads, 1) chunk_bwd_kernel(const BwdParams p) {
    uint8_t *smem = smem_base();
    uint8_t *misc = smem + OFF_MISC;
    float *s_beta = reinterpret_cast<float *>(misc + M_BETA);
    float *s_em = reinterpret_cast<float *>(misc + M_EM);
    float *s_dec = reinterpret_cast<float *>(misc + M_DEC);
    float *s_part = reinterpret_cast<float *>(misc + M_PART);
    float *s_dgl = reinterpret_cast<float *>(misc + M_DGL);
    float *s_suf = reinterpret_cast<float *>(misc + M_SUF);
    // Reductions across warps go through per-warp parts added in a fixed order
    // (no shared-memory atomics), so the gradients do not depend on timing.
    float *s_dglp = s_suf;                                     // [quarter][k]
    float *s_dbp = reinterpret_cast<float *>(misc + M_P);      // [8][r]
    float *s_khp = s_dbp + 512;                                // [grp][k]
    float *s_gl = reinterpret_cast<float *>(misc + M_GL);
    float *s_kk = reinterpret_cast<float *>(smem + OFF_KK);
    float *s_at = reinterpret_cast<float *>(smem + OFF_AT);
    uint64_t *bar_mma = reinterpret_cast<uint64_t *>(misc + M_BAR);
    int *ctrl = reinterpret_cast<int *>(misc + M_CTRL);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, grp = warp >> 2;
    const int ch = quarter * 32 + lane;  // channel / tensor-memory lane
    const int H = p.H;
    const int num_chains = p.B * H;
    uint8_t *scr = p.scratch + static_cast<size_t>(blockIdx.x) * kScratchPerCta;
    auto img = [&](int i) { return scr + img_off(i); };

    if (warp == 0) tmem_alloc(reinterpret_cast<uint32_t *>(&ctrl[0]), 512);
    if (tid == 0) {
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        ctrl[2] = 0;
    }
    // the inverse's T: the blocks above the diagonal are zero (restored after
    // D_A in every chunk, whose Ks copy overwrites them)
    for (int e = tid; e < 4096 / 4; e += kThreads)
        reinterpret_cast<float4 *>(smem + OFF_TT)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(ctrl[0]);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tl = tmem + lane_base;  // this warp's lane quarter
    const uint32_t sa = smem_addr(smem + SLOT_A), sb = smem_addr(smem + SLOT_B);

    Sched S;
    S.smem = smem;
    S.scr = scr;
    S.bar_mma = bar_mma;
    S.abort_flag = &ctrl[2];
    S.err = p.err;
    S.polls = p.polls;
    S.sa = sa;
    S.sb = sb;
    S.tid = tid;
    S.sl0 = S.sl1 = -1;
    clear_extra(S);
    S.lo0 = S.hi0 = S.lo1 = S.hi1 = 0;
    S.ph_mma = 0;
    S.pend_mma = false;
    S.pend_copy = false;
    const float kLog2e = 1.4426950408889634f;
    const float kMaxChunkLog2 = kMaxChunkDecay * kLog2e;

    // Makes every thread's image and tensor-memory writes visible to the next
    // copy / product (the images are read back by the same CTA's cp.async, in
    // the generic proxy, so a CTA barrier orders them).
    auto publish = [&]() {
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
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
        const bool skip = p.split[chain] != 0;
        if (skip && tid == 0) record_device_error(p.err, kDevDecayRange);

        // ---- dS^T <- dS_final (lane v, column k holds dS[k][v]) ----
        {
            float r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                r[j] = (p.dSf != nullptr) ? p.dSf[state_off + (32 * grp + j) * kD + ch] : 0.f;
            tmem_st32(tl + C_DS + 32 * grp, r);
            tmem_wait_st();
        }

        const int64_t nchunks = (t1 - t0 + kC - 1) / kC;
        const int64_t slot0 = t0 / kC + b;
        for (int64_t c = skip ? -1 : nchunks - 1; c >= 0; --c) {
            const int64_t tc = t0 + c * kC;
            const int L = static_cast<int>((t1 - tc) < kC ? (t1 - tc) : kC);
            const float *Sc = p.ckpt + ((slot0 + c) * H + h) * (kD * kD);
            S.sl0 = S.sl1 = -1;  // every image is rewritten for this chunk
            clear_extra(S);
            // ---- B0: the chunk's rows into shared memory by 16-byte cp.async
            // (rows past the sequence zero-filled): g and dO to slot A, q to the
            // A_kk area (free until the D_A epilogue), k and v to the staging
            // area (read again later) ----
            {
                const int dob = p.dO_bf16 ? 2 : 4;  // bytes per dO element
                auto src_row = [&](int r) { return ((tc + (r < L ? r : 0)) * H + h) * kD; };
                for (int u = tid; u < kC * 32; u += kThreads) {
                    const int r = u >> 5, pc = u & 31;
                    cp_async_16(smem + SLOT_A + u * 16, p.g + src_row(r) + pc * 4, r < L);
                }
                const int dpr = 8 * dob;  // 16-byte pieces per dO row
                for (int u = tid; u < kC * dpr; u += kThreads) {
                    const int r = u / dpr, pc = u - r * dpr;
                    cp_async_16(smem + SLOT_A + 32768 + u * 16,
                                static_cast<const uint8_t *>(p.dO) + src_row(r) * dob + pc * 16, r < L);
                }
                for (int u = tid; u < kC * 16; u += kThreads) {
                    const int r = u >> 4, pc = u & 15;
                    const int64_t e = src_row(r) + pc * 8;
                    cp_async_16(smem + OFF_AT + u * 16, p.q + e, r < L);
                    cp_async_16(smem + OFF_STG + u * 16, p.k + e, r < L);
                    cp_async_16(smem + OFF_STG + 16384 + u * 16, p.v + e, r < L);
                }
                cp_async_wait_all();
            }
            __syncthreads();

            // ---- B1: cumulative decay and the chunk operand images ----
            float gam[16];
            float *gA = reinterpret_cast<float *>(smem + SLOT_A);  // g, then Gam in place
            {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {  // the forward kernel's order
                    const int r = 16 * grp + i;
                    if (r < L) acc += kLog2e * gA[r * kD + ch];
                    gam[i] = acc;
                }
                s_part[grp * kD + ch] = acc;
            }
            if (tid < kC) s_beta[tid] = tid < L ? p.beta[(tc + tid) * H + h] : 0.f;
            __syncthreads();
            float prefix = 0.f, gam_l = 0.f;
#pragma unroll
            for (int g2 = 0; g2 < 4; ++g2) {
                const float pg = s_part[g2 * kD + ch];
                if (g2 < grp) prefix += pg;
                gam_l += pg;
            }
            if (-gam_l > kMaxChunkLog2 && tid == 0) record_device_error(p.err, kDevDecayRange);
            const float m = 0.5f * gam_l;
            if (grp == 0) {
                s_em[ch] = fast_exp2(m);
                s_dec[ch] = fast_exp2(gam_l);
                s_gl[ch] = gam_l;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) gam[i] += prefix;  // Gam_r in log2 units from here on
            // Gam [64][128] over g in slot A (each thread its own elements), then
            // the operand images eight channels of one row at a time (unit u: row
            // u / 16, channels 8 (u % 16) .. + 7)
#pragma unroll
            for (int i = 0; i < 16; ++i) gA[(16 * grp + i) * kD + ch] = gam[i];
            __syncthreads();
#pragma unroll 1
            for (int u = tid; u < kC * 16; u += kThreads) {
                const int r = u >> 4, c0 = (u & 15) * 8;
                float qv[8], kv[8], vv[8], dov[8];  // rows past the sequence are zero
                {
                    const uint4 q8 = *reinterpret_cast<const uint4 *>(smem + OFF_AT + u * 16);
                    const uint4 k8 = *reinterpret_cast<const uint4 *>(smem + OFF_STG + u * 16);
                    const uint4 v8 = *reinterpret_cast<const uint4 *>(smem + OFF_STG + 16384 + u * 16);
                    const __nv_bfloat16 *qb = reinterpret_cast<const __nv_bfloat16 *>(&q8);
                    const __nv_bfloat16 *kb = reinterpret_cast<const __nv_bfloat16 *>(&k8);
                    const __nv_bfloat16 *vb = reinterpret_cast<const __nv_bfloat16 *>(&v8);
                    if (p.dO_bf16) {
                        const uint4 d8 = *reinterpret_cast<const uint4 *>(smem + SLOT_A + 32768 + u * 16);
                        const __nv_bfloat16 *db = reinterpret_cast<const __nv_bfloat16 *>(&d8);
#pragma unroll
                        for (int j = 0; j < 8; ++j) dov[j] = __bfloat162float(db[j]);
                    } else {
                        const float4 d0 = *reinterpret_cast<const float4 *>(smem + SLOT_A + 32768 + u * 32);
                        const float4 d1 = *reinterpret_cast<const float4 *>(smem + SLOT_A + 32768 + u * 32 + 16);
                        dov[0] = d0.x; dov[1] = d0.y; dov[2] = d0.z; dov[3] = d0.w;
                        dov[4] = d1.x; dov[5] = d1.y; dov[6] = d1.z; dov[7] = d1.w;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        qv[j] = __bfloat162float(qb[j]);
                        kv[j] = __bfloat162float(kb[j]);
                        vv[j] = __bfloat162float(vb[j]);
                    }
                }
                const float *gt = gA + r * kD + c0;
                float qt[8], kr[8], ks[8], kh[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float gr = gt[j], gl = s_gl[c0 + j], mj = 0.5f * gl;
                    const float eu = fast_exp2(gr - mj);
                    qt[j] = p.scale * qv[j] * eu;
                    kr[j] = kv[j] * eu;
                    ks[j] = kv[j] * fast_exp2(mj - gr);
                    kh[j] = kv[j] * fast_exp2(gl - gr);
                }
                put8(smem + SLOT_B, img_half(I_QK), 128, r, c0, qt);  // staged (slot B is free)
                put8(smem + SLOT_B, img_half(I_QK), 128, 64 + r, c0, kr);
                put8(img(I_KS), img_half(I_KS), 64, r, c0, ks);
                put8(smem + OFF_TT, img_half(I_KS), 64, r, c0, ks);  // for D_A, below
                put8(img(I_KH), img_half(I_KH), 64, r, c0, kh);
                put8(img(I_V), 0, 64, r, c0, vv);
                put8(img(I_DU2), img_half(I_DU2), 128, 64 + r, c0, dov);
            }
            stage_store(S, 1, I_QK, 0, 128);

            // ---- D_A = [Qt; Kr] Ks^T ----
            // Ks from its copy in the inverse's work areas (T and kk, both
            // free until D_A completes), standing in for slot A
            S.sa = smem_addr(smem + OFF_TT);
            set_slot(S, 0, I_KS, 0, 64);
            const bool da_ok = product(S, {I_QK, 0, 0}, {I_KS, 0, 0}, tmem + C_TA, 64, 8, false);
            S.sa = smem_addr(smem + SLOT_A);
            S.sl0 = -1;
            if (!da_ok) break;
            {
                float d16[16];
                tmem_ld16(tl + C_TA + 16 * grp, d16);
                tmem_wait_ld();
                if (quarter < 2) {  // A_qk rows r = ch
                    float a[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) a[j] = (16 * grp + j <= ch) ? d16[j] : 0.f;
                    put8(img(I_AQ), img_half(I_AQ), 64, ch, 16 * grp, a);
                    put8(img(I_AQ), img_half(I_AQ), 64, ch, 16 * grp + 8, a + 8);
                } else {  // kk rows r = ch - 64: kept, and A_kk column-major for the inverse
                    const int r = ch - 64;
                    const float br = s_beta[r];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s = 16 * grp + j;
                        s_kk[s * 64 + r] = d16[j];
                        s_at[s * 64 + r] = (s < r) ? br * d16[j] : 0.f;
                    }
                }
            }
            {
                // Ks's copy is consumed: the blocks of T above its diagonal
                // back to zero (the inverse leaves them alone and reads them)
                float *T = reinterpret_cast<float *>(smem + OFF_TT);
                for (int e = tid; e < kC * kC; e += kThreads)
                    if (((e & 63) >> 4) > (e >> 10)) T[e] = 0.f;
            }
            dirty(S, I_AQ);
            __syncthreads();

            // ---- T = (I + A_kk)^{-1} on warps 0-3 (fp32, row-major); meanwhile
            // warps 4-15 (B2) form the S_op^T and dS'^T images (row v = the
            // lane) and sum_v dS' S from the chunk-start state S, brought into
            // slot A.  Then T diag(beta) and T as split images staged in slot B
            // by every thread (row tid / 8, columns 8 (tid % 8) .. + 7), T
            // also stored to its image ----
            {
                float *T = reinterpret_cast<float *>(smem + OFF_TT);
                if (warp >= 4) {
                    // the checkpoint S into slot A (its Ks is dead since D_A),
                    // in flight while the dS' image is formed; each image is
                    // staged in slot B (QK's copy there is given up: the W'
                    // product copies its rows back) and then copied to the
                    // scratch with coalesced stores
                    const int bt = tid - 128;  // 0 .. 383
                    for (int u = bt; u < 4096; u += kThreads - 128)
                        cp_async_16(smem + SLOT_A + u * 16, Sc + u * 4, true);
                    uint8_t *stage = smem + SLOT_B;
                    auto copy_out = [&](int i) {
                        named_sync(2, kThreads - 128);
                        for (uint32_t u = bt; u < img_bytes(i) / 16; u += kThreads - 128)
                            *reinterpret_cast<uint4 *>(img(i) + u * 16) =
                                *reinterpret_cast<const uint4 *>(stage + u * 16);
                        named_sync(2, kThreads - 128);
                    };
                    // 16-column units of k: warps 4-7 take units 0, 3, 6, warps
                    // 8-11 units 1, 4, 7 and warps 12-15 units 2, 5
#pragma unroll 1
                    for (int u = grp - 1; u < 8; u += 3) {
                        const int k0 = 16 * u;
                        float ds[16];
                        tmem_ld16(tl + C_DS + k0, ds);
                        tmem_wait_ld();
                        put8(stage, img_half(I_DS), 128, ch, k0, ds);
                        put8(stage, img_half(I_DS), 128, ch, k0 + 8, ds + 8);
                    }
                    copy_out(I_DS);
                    cp_async_wait_all();
                    named_sync(2, kThreads - 128);
                    const float *Ss = reinterpret_cast<const float *>(smem + SLOT_A);
#pragma unroll 1
                    for (int u = grp - 1; u < 8; u += 3) {
                        const int k0 = 16 * u;
                        float ds[16], sv[16], so[16];
                        tmem_ld16(tl + C_DS + k0, ds);
#pragma unroll
                        for (int j = 0; j < 16; ++j) sv[j] = Ss[(k0 + j) * kD + ch];
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) so[j] = s_em[k0 + j] * sv[j];
                        put8(stage, img_half(I_SO), 128, ch, k0, so);
                        put8(stage, img_half(I_SO), 128, ch, k0 + 8, so + 8);
#pragma unroll
                        for (int j = 0; j < 16; ++j) so[j] = ds[j] * sv[j];
                        const float t = lanes_sum16(so, lane);
                        if ((lane & 1) == 0) s_dglp[quarter * kD + k0 + (lane >> 1)] = t;
                    }
                    copy_out(I_SO);  // its barriers also order the parts above
                    if (bt < kD)
                        s_dgl[bt] = ((s_dglp[bt] + s_dglp[kD + bt]) + s_dglp[2 * kD + bt]) +
                                    s_dglp[3 * kD + bt];
                } else {
                    float *Tdiag = reinterpret_cast<float *>(misc + M_TDIAG);
                    float *T32c = reinterpret_cast<float *>(misc + M_T32);
                    float *P = reinterpret_cast<float *>(misc + M_P);
                    // T complete in its row-major form; the split images are formed
                    // from it by the whole CTA
                    const TRowMajor out{T};
                    if (tid < 64) {
                        ut_diag_solve(s_at, T, Tdiag, out, tid);
                        __syncwarp();
                        ut_level1<TRowMajor, 4>(s_at, T, Tdiag, P, T, T32c, out, tid);
                    }
                    inverse_sync();
                    ut_level2<TRowMajor, 4>(s_at, T, Tdiag, T32c, P, out, tid);
                }
                __syncthreads();
                // the checkpoint in slot A is dead: the W' product's Kr rows
                // meanwhile
                preload(S, 0, I_QK, 64, 128);
                // A_kk is consumed: q again into its area for the assembly
                for (int u = tid; u < kC * 16; u += kThreads) {
                    const int r = u >> 4, pc = u & 15;
                    cp_async_16(smem + OFF_AT + u * 16, p.q + ((tc + (r < L ? r : 0)) * H + h) * kD + pc * 8,
                                r < L);
                }
                const int r = tid >> 3, c0 = (tid & 7) * 8;
                const float4 t0 = *reinterpret_cast<const float4 *>(T + r * 64 + c0);
                const float4 t1 = *reinterpret_cast<const float4 *>(T + r * 64 + c0 + 4);
                const float t8[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                float tb8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) tb8[j] = t8[j] * s_beta[c0 + j];
                put8(smem + SLOT_B, img_half(I_TB), 64, r, c0, tb8);
                put8(smem + SLOT_B + img_bytes(I_TB), img_half(I_T), 64, r, c0, t8);
                put8(img(I_T), img_half(I_T), 64, r, c0, t8);
            }
            fence_proxy_async_smem();
            publish();
            set_slot(S, 1, I_TB, 0, 64);

            // Epilogues below write their image into a slot whose operand is
            // dead (the image's own byte layout) and copy it to the scratch from
            // there; a whole image stays in the slot for the products that
            // follow.

            // ---- W'^T = Kr^T (T beta)^T and Ut^T = V^T (T beta)^T; -W'^T image
            // in V's slot ----
            if (!product(S, {I_QK, 64, 1}, {I_TB, 0, 0}, tmem + C_TA, 64, 4, false)) break;
            if (!product(S, {I_V, 0, 1}, {I_TB, 0, 0}, tmem + C_TB, 64, 4, false)) break;
            preload(S, S.sl0 == I_TB ? 0 : 1, I_SO, 0, 128);
            {
                const int sl = (S.sl0 == I_V) ? 0 : 1;
                float w16[16];
                tmem_ld16(tl + C_TA + 16 * grp, w16);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) w16[j] = -w16[j];
                put8(slot_ptr(S, sl), img_half(I_WT), 128, ch, 16 * grp, w16);
                put8(slot_ptr(S, sl), img_half(I_WT), 128, ch, 16 * grp + 8, w16 + 8);
                stage_store(S, sl, I_WT, 0, 128);
            }

            // ---- U^T = Ut^T + S_op^T (-W'^T); U^T image in S_op's slot ----
            if (!product(S, {I_SO, 0, 0}, {I_WT, 0, 1}, tmem + C_TB, 64, 8, true)) break;
            preload(S, S.sl0 == I_WT ? 0 : 1, I_DS, 0, 128);
            {
                const int sl = (S.sl0 == I_SO) ? 0 : 1;
                float u16[16];
                tmem_ld16(tl + C_TB + 16 * grp, u16);
                tmem_wait_ld();
                put8(slot_ptr(S, sl), img_half(I_UT), 128, ch, 16 * grp, u16);
                put8(slot_ptr(S, sl), img_half(I_UT), 128, ch, 16 * grp + 8, u16 + 8);
                stage_store(S, sl, I_UT, 0, 128);
            }

            // ---- dU^T = dS'^T Kh + dO^T A_qk ; dU into rows 0-63 of DU2, which
            // stays in its slot ----
            {
                // A_qk for the next product into Kh's slot, past Kh (32 KB)
                const Pre pre_aq{I_AQ, 0, 64, 1, 32768};
                if (!product(S, {I_DS, 0, 0}, {I_KH, 0, 0}, tmem + C_TA, 64, 8, false, 0, 128, &pre_aq))
                    break;
            }
            if (!product<true>(S, {I_DU2, 64, 1}, {I_AQ, 0, 1}, tmem + C_TA, 64, 4, true)) break;
            preload(S, slot_of(S, I_AQ), I_QK, 0, 64);
            {
                const int sl = (S.sl0 == I_DU2) ? 0 : 1;
                float d16[16];
                tmem_ld16(tl + C_TA + 16 * grp, d16);  // dU^T[v = ch][r]
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    put1(slot_ptr(S, sl), img_half(I_DU2), 128, 16 * grp + j, ch, d16[j]);
                stage_store(S, sl, I_DU2, 0, 64);
            }

            // ---- P^T = dO^T Qt - dU^T W'^T... ; dS <- e^{Gam_L} dS' + e^m P ----
            if (!product(S, {I_DU2, 64, 1}, {I_QK, 0, 1}, tmem + C_TA, 128, 4, false)) break;
            if (!product(S, {I_DU2, 0, 1}, {I_WT, 0, 0}, tmem + C_TA, 128, 4, true)) break;
            preload(S, S.sl0 == I_WT ? 0 : 1, I_UT, 0, 128);
            {
                float pv[32], ds[32];
                tmem_ld32(tl + C_TA + 32 * grp, pv);
                tmem_ld32(tl + C_DS + 32 * grp, ds);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int kq = 32 * grp + j;
                    ds[j] = s_dec[kq] * ds[j] + s_em[kq] * pv[j];
                }
                tmem_st32(tl + C_DS + 32 * grp, ds);
                tmem_wait_st();
            }
            tc_fence_before();  // (no global image was written since the last publish)
            __syncthreads();
            tc_fence_after();

            // ---- dA_qk = tril(dO U^T) (lanes 64-127 of [dU; dO] U^T) ----
            if (!product(S, {I_DU2, 0, 0}, {I_UT, 0, 1}, tmem + C_TA, 64, 8, false, 64, 128)) break;  // lanes 64-127
            {
                const int sl = (S.sl0 == I_UT) ? 0 : 1;
                if (quarter >= 2) {
                    const int r = ch - 64;
                    float d16[16];
                    tmem_ld16(tl + C_TA + 16 * grp, d16);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) d16[j] = (16 * grp + j <= r) ? d16[j] : 0.f;
                    put8(slot_ptr(S, sl), img_half(I_DAQ), 64, r, 16 * grp, d16);
                    put8(slot_ptr(S, sl), img_half(I_DAQ), 64, r, 16 * grp + 8, d16 + 8);
                }
                stage_store(S, sl, I_DAQ, 0, 64);
            }

            // ---- [-dW'^T | dQt^T] = S_op [dU; dO]^T (DU2 still in its slot) ;
            // dKs^T = Qt^T dA_qk ; dQt^T += Ks^T dA_qk^T ----
            if (!product(S, {I_SO, 0, 1}, {I_DU2, 0, 0}, tmem + C_TA, 128, 8, false)) break;
            {
                // Ks for the next product into dA_qk's slot, past dA_qk (16 KB)
                const Pre pre_ks{I_KS, 0, 64, 1, 16384};
                if (!product(S, {I_QK, 0, 1}, {I_DAQ, 0, 1}, tmem + C_S, 64, 4, false, 0, 128, &pre_ks))
                    break;
            }
            if (!product<true>(S, {I_KS, 0, 1}, {I_DAQ, 0, 0}, tmem + C_TB, 64, 4, true)) break;
            preload(S, 1 - slot_of(S, I_DAQ), I_DS, 0, 128);
            {
                // -dW'^T[k = ch][r]: dW'[r][k] into rows 0-63 of the QK image (Qt is
                // dead), staged in the slot dA_qk used
                const int sl = (S.sl0 == I_DAQ) ? 0 : 1;
                float d16[16];
                tmem_ld16(tl + C_TA + 16 * grp, d16);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    put1(slot_ptr(S, sl), img_half(I_QK), 128, 16 * grp + j, ch, -d16[j]);
                stage_store(S, sl, I_QK, 0, 64);
            }

            // ---- dKh^T = dS' U^T ----
            if (!product(S, {I_DS, 0, 1}, {I_UT, 0, 1}, tmem + C_H, 64, 8, false)) break;

            // ---- dT = (dW' Kr^T + dU V^T) diag(beta) (lanes 0-63) ----
            {
                // v for the next product into the other slot, at 48 KB (its
                // images are dead)
                const Pre pre_v{I_V, 0, 64, 2, 49152};
                if (!product(S, {I_QK, 0, 0}, {I_QK, 64, 0}, tmem + C_TA, 64, 8, false, 0, 64, &pre_v))
                    break;  // lanes 0-63
            }
            if (!product<true>(S, {I_DU2, 0, 0}, {I_V, 0, 0}, tmem + C_TA, 64, 8, true, 0, 64)) break;  // lanes 0-63
            preload(S, S.sl0 == I_DU2 ? 0 : 1, I_QK, 0, 64);
            if (quarter < 2) {
                float d16[16];
                tmem_ld16(tl + C_TA + 16 * grp, d16);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) d16[j] *= s_beta[16 * grp + j];
                put8(slot_ptr(S, slot_of(S, I_V)), img_half(I_DT), 64, ch, 16 * grp, d16);
                put8(slot_ptr(S, slot_of(S, I_V)), img_half(I_DT), 64, ch, 16 * grp + 8, d16 + 8);
            }
            stage_store(S, slot_of(S, I_V), I_DT, 0, 64);

            // ---- d(beta Kr)^T = dW'^T T and d(beta V)^T = dU^T T ----
            if (!product(S, {I_QK, 0, 1}, {I_T, 0, 1}, tmem + C_R, 64, 4, false)) break;
            if (!product(S, {I_DU2, 0, 1}, {I_T, 0, 1}, tmem + C_VB, 64, 4, false)) break;
            preload(S, S.sl0 == I_DU2 ? 0 : 1, I_DT, 0, 64);
            {
                // d(beta V)^T[v = ch][r]: dv = beta_r d(beta V); dbeta += sum_v d(beta V) v.
                // d(beta Kr)^T[k = ch][r]: dbeta += sum_k d(beta Kr) Kr.
                float vb[16], rb[16], vv[16], kr[16];
                tmem_ld16(tl + C_VB + 16 * grp, vb);
                tmem_ld16(tl + C_R + 16 * grp, rb);
                const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_STG);
#pragma unroll
                for (int j = 0; j < 16; ++j) {  // staged rows (zero past the sequence)
                    const int r = 16 * grp + j;
                    vv[j] = __bfloat162float(ks[8192 + r * kD + ch]);
                    kr[j] = __bfloat162float(ks[r * kD + ch]);
                }
                tmem_wait_ld();
                float sum[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r = 16 * grp + j;
                    if (r < L) p.dv[((tc + r) * H + h) * kD + ch] = s_beta[r] * vb[j];
                    sum[j] = vb[j] * vv[j] + rb[j] * kr[j] * fast_exp2(gam[j] - m);
                }
                const float t = lanes_sum16(sum, lane);
                if ((lane & 1) == 0) s_dbp[quarter * kC + 16 * grp + (lane >> 1)] = t;
            }

            // ---- Y = dT T^T (lanes 0-63) ----
            if (!product(S, {I_DT, 0, 0}, {I_T, 0, 0}, tmem + C_TA, 64, 4, false)) break;
            if (quarter < 2) {
                float d16[16];
                tmem_ld16(tl + C_TA + 16 * grp, d16);
                tmem_wait_ld();
                put8(slot_ptr(S, S.sl0 == I_DT ? 0 : 1), img_half(I_Y), 64, ch, 16 * grp, d16);
                put8(slot_ptr(S, S.sl0 == I_DT ? 0 : 1), img_half(I_Y), 64, ch, 16 * grp + 8, d16 + 8);
            }
            stage_only(S, S.sl0 == I_DT ? 0 : 1, I_Y, 0, 64);  // read from the slot only

            // ---- dA_kk = -strict_tril(T^T Y) (lanes 0-63); dbeta += rowsum(dA_kk kk) ----
            if (!product(S, {I_T, 0, 1}, {I_Y, 0, 1}, tmem + C_TA, 64, 4, false)) break;
            // Kr's rows for the dKs product into Y's slot meanwhile; beta dA_kk
            // staged in T's slot (read from there only), dA_kk to the scratch
            const int sy = S.sl0 == I_Y ? 0 : 1;
            preload(S, sy, I_QK, 64, 128);
            if (quarter < 2) {
                const int r = ch;
                float d16[16], bd[16];
                tmem_ld16(tl + C_TA + 16 * grp, d16);
                tmem_wait_ld();
                float part = 0.f;
                const float br = s_beta[r];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int s = 16 * grp + j;
                    d16[j] = (s < r) ? -d16[j] : 0.f;
                    bd[j] = br * d16[j];
                    part += d16[j] * s_kk[s * 64 + r];
                }
                s_dbp[(4 + grp) * kC + r] = part;
                put8(img(I_DKK), img_half(I_DKK), 64, r, 16 * grp, d16);
                put8(img(I_DKK), img_half(I_DKK), 64, r, 16 * grp + 8, d16 + 8);
                uint8_t *sb = slot_ptr(S, 1 - sy);
                put8(sb, img_half(I_BDKK), 64, r, 16 * grp, bd);
                put8(sb, img_half(I_BDKK), 64, r, 16 * grp + 8, bd + 8);
            }
            dirty(S, I_DKK);
            stage_only(S, 1 - sy, I_BDKK, 0, 64);

            // ---- dKs^T += Kr^T (beta dA_kk) ; (dA_kk Ks)^T into C_R ----
            {
                // Ks for the next product into beta dA_kk's slot, past it (16 KB)
                const Pre pre_ks2{I_KS, 0, 64, 1, 16384};
                if (!product(S, {I_QK, 64, 1}, {I_BDKK, 0, 1}, tmem + C_S, 64, 4, true, 0, 128, &pre_ks2))
                    break;
            }
            if (!product<true>(S, {I_KS, 0, 1}, {I_DKK, 0, 0}, tmem + C_R, 64, 4, true)) break;

            // ---- assembly: dq, dk, dg, dbeta (lane k = ch, rows r = 16 grp + j) ----
            cp_async_wait_all();  // q staged after the inverse
            __syncthreads();
            {
                const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_AT);
                const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_STG);
                float dgam[16], khsum = 0.f;
#pragma unroll
                for (int j0 = 0; j0 < 16; j0 += 8) {  // eight rows at a time
                    float dqt[8], dkh[8], dks[8], dkr[8], qv[8], kv[8];
                    tmem_ld8(tl + C_TB + 16 * grp + j0, dqt);
                    tmem_ld8(tl + C_H + 16 * grp + j0, dkh);
                    tmem_ld8(tl + C_S + 16 * grp + j0, dks);
                    tmem_ld8(tl + C_R + 16 * grp + j0, dkr);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int r = 16 * grp + j0 + j;
                        qv[j] = __bfloat162float(qs[r * kD + ch]);
                        kv[j] = __bfloat162float(ks[r * kD + ch]);
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int r = 16 * grp + j0 + j;
                        const float gr = gam[j0 + j];
                        dgam[j0 + j] = 0.f;
                        if (r < L) {
                            const int64_t e = ((tc + r) * H + h) * kD + ch;
                            const float eu = fast_exp2(gr - m), ed = fast_exp2(m - gr);
                            const float eh = fast_exp2(gam_l - gr);
                            const float Qt = p.scale * qv[j] * eu, Kr = kv[j] * eu, Ks = kv[j] * ed;
                            const float Kh = kv[j] * eh;
                            const float dKr = s_beta[r] * dkr[j];
                            p.dq[e] = p.scale * dqt[j] * eu;
                            p.dk[e] = dKr * eu + dks[j] * ed + dkh[j] * eh;
                            const float khp = dkh[j] * Kh;
                            dgam[j0 + j] = dKr * Kr - dks[j] * Ks - khp + dqt[j] * Qt;
                            khsum += khp;
                        }
                    }
                }
                // suffix sums over the chunk's rows: this group's rows, then the later groups
                float run = 0.f;
#pragma unroll
                for (int j = 15; j >= 0; --j) {
                    run += dgam[j];
                    dgam[j] = run;
                }
                s_suf[grp * kD + ch] = run;
                s_khp[grp * kD + ch] = khsum;
                __syncthreads();
                float later = 0.f;
#pragma unroll
                for (int g2 = 0; g2 < 4; ++g2)
                    if (g2 > grp) later += s_suf[g2 * kD + ch];
                // dGam_L = colsum(dKh . Kh) + e^{Gam_L} sum_v dS' S, added to every row
                const float khs = ((s_khp[ch] + s_khp[kD + ch]) + s_khp[2 * kD + ch]) +
                                  s_khp[3 * kD + ch];
                const float dgl = khs + s_dec[ch] * s_dgl[ch];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r = 16 * grp + j;
                    if (r < L) p.dg[((tc + r) * H + h) * kD + ch] = dgam[j] + later + dgl;
                }
                if (tid < L) {
                    float db = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) db += s_dbp[i * kC + tid];
                    p.dbeta[(tc + tid) * H + h] = db;
                }
            }
            // the gradients are not read back: a plain barrier before the next chunk
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }
        if (ctrl[2] != 0) break;

        // ---- dS0 ----
        if (p.dS0 != nullptr) {
            float r[32];
            tmem_ld32(tl + C_DS + 32 * grp, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) p.dS0[state_off + (32 * grp + j) * kD + ch] = skip ? 0.f : r[j];
        }
        if (skip) {  // chains without 64-token-aligned checkpoints: zero gradients
            for (int64_t e = t0 * kD + tid; e < t1 * kD; e += kThreads) {
                const int64_t t = e / kD, c2 = e % kD;
                const int64_t i = (t * H + h) * kD + c2;
                p.dq[i] = 0.f;
                p.dk[i] = 0.f;
                p.dv[i] = 0.f;
                p.dg[i] = 0.f;
                if (c2 == 0) p.dbeta[t * H + h] = 0.f;
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    // Drain: wait for a product still in flight (full bound) and this thread's
    // copies before the tensor memory is released and the CTA exits.
    cp_async_wait_all();
    if (tid == 0 && S.pend_mma) mbar_wait_bounded(bar_mma, S.ph_mma & 1, kMaxPolls);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

namespace {
size_t split_flags_bytes(int B, int H) {
    return ((static_cast<size_t>(B) * H * sizeof(int) + 255) / 256) * 256;
}
size_t checkpoint_states_bytes(int64_t N, int B, int H) {
    return (static_cast<size_t>(N / kC) + static_cast<size_t>(B)) * H * kD * kD * sizeof(float);
}
}  // namespace

size_t chunk_checkpoint_flags_bytes(int B, int H) { return split_flags_bytes(B, H); }

size_t chunk_checkpoints_bytes(int64_t N, int B, int H) {
    return split_flags_bytes(B, H) + checkpoint_states_bytes(N, B, H);
}

size_t chunk_bwd_from_checkpoints_workspace_bytes(int ctas) {
    return 512 + static_cast<size_t>(ctas) * kScratchPerCta;
}

// Workspace of the self-contained backward: the forward pass's counter (512
// bytes), the checkpoint buffer (flags and states), then the workspace of the
// backward from checkpoints (its counter and the per-CTA scratch).
size_t chunk_bwd_workspace_bytes(int64_t N, int B, int H, int ctas) {
    return 512 + chunk_checkpoints_bytes(N, B, H) + chunk_bwd_from_checkpoints_workspace_bytes(ctas);
}

cudaError_t launch_chunk_backward_from_checkpoints(
    const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *g,
    const float *beta, const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
    const void *checkpoints, const void *dO, bool dO_bf16, const float *dSf, float *dq, float *dk,
    float *dv, float *dg, float *dbeta, float *dS0, void *workspace, int ctas, unsigned int *err,
    cudaStream_t s) {
    if (B == 0 || H == 0) return cudaSuccess;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e = cudaMemsetAsync(ws, 0, 512, s);  // the chain counter
    if (e != cudaSuccess) return e;
    e = ensure_dynamic_smem(reinterpret_cast<const void *>(chunk_bwd_kernel), static_cast<int>(kSmemAlloc));
    if (e != cudaSuccess) return e;
    const uint8_t *cp = static_cast<const uint8_t *>(checkpoints);
    BwdParams p;
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.cu_seqlens = cu_seqlens; p.B = B; p.N = N; p.H = H; p.scale = scale;
    p.dO = dO; p.dO_bf16 = dO_bf16 ? 1 : 0; p.dSf = dSf;
    p.split = reinterpret_cast<const int *>(cp);
    p.ckpt = reinterpret_cast<const float *>(cp + split_flags_bytes(B, H));
    p.dq = dq; p.dk = dk; p.dv = dv; p.dg = dg; p.dbeta = dbeta; p.dS0 = dS0;
    p.scratch = ws + 512;
    p.counter = reinterpret_cast<unsigned int *>(ws);
    p.err = err;
    p.polls = prefill_wait_polls();
    chunk_bwd_kernel<<<ctas, kThreads, kSmemAlloc, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_chunk_backward(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                  const __nv_bfloat16 *v, const float *g, const float *beta,
                                  const int32_t *cu_seqlens, int B, int64_t N, int H, float scale,
                                  const float *S0, const void *dO, bool dO_bf16, const float *dSf,
                                  float *dq, float *dk, float *dv, float *dg, float *dbeta,
                                  float *dS0, void *workspace, int ctas, unsigned int *err,
                                  int num_sms, cudaStream_t s) {
    if (B == 0 || H == 0) return cudaSuccess;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *checkpoints = ws + 512;
    int *split = reinterpret_cast<int *>(checkpoints);
    float *ckpt = reinterpret_cast<float *>(checkpoints + split_flags_bytes(B, H));
    cudaError_t e = cudaMemsetAsync(ws, 0, 512 + split_flags_bytes(B, H), s);
    if (e != cudaSuccess) return e;
    // forward pass: chunk-start states only
    e = launch_prefill_checkpoints(q, k, v, g, beta, cu_seqlens, B, N, H, scale, S0, ckpt, split,
                                   reinterpret_cast<unsigned int *>(ws), err, num_sms, s);
    if (e != cudaSuccess) return e;
    return launch_chunk_backward_from_checkpoints(
        q, k, v, g, beta, cu_seqlens, B, N, H, scale, checkpoints, dO, dO_bf16, dSf, dq, dk, dv, dg,
        dbeta, dS0, ws + 512 + chunk_checkpoints_bytes(N, B, H), ctas, err, s);
}

}  // namespace kda

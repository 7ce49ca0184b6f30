// kda_gate_spec_x2.cuh -- the binary32 gate specification of kda_gate_spec.cuh
// evaluated on packed pairs (used by the gate kernel, kda_gate.cu), bit for bit
// equal to the scalar functions there.  Not part of the public ABI.
#pragma once

#include "kda_f32x2.cuh"
#include "kda_gate_spec.cuh"

namespace kda {
namespace gate_spec {

// Two elements per instruction where the operation is +, -, x or fma;
// divisions, conversions and the special cases per element.

// a / b rounded to nearest even, for the divisions of the common path below
// (a normal or +0, b in [1, 2.5], the quotient normal or +0), two at a time,
// by Markstein's method (P. W. Markstein, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): the
// special-function unit's reciprocal refined by one Newton step, the quotient,
// its remainder (exact in an fma) and one correction.  Over every operand pair
// the common path can form, the result equals IEEE division bit for bit
// (checked exhaustively on the device: kda_debug_check_gate_division).
__device__ __forceinline__ float rcp_sfu(float b) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(b));
    return y;
}
__device__ __forceinline__ uint64_t div2_common(uint64_t a, uint64_t b) {
    const float2 bb = f2_split(b);
    const uint64_t nb = f2(-bb.x, -bb.y);
    const uint64_t y0 = f2(rcp_sfu(bb.x), rcp_sfu(bb.y));
    const uint64_t y1 = f2_fma(y0, f2_fma(nb, y0, f2(1.0f, 1.0f)), y0);
    const uint64_t q0 = f2_mul(a, y1);
    return f2_fma(f2_fma(nb, q0, a), y1, q0);
}

__device__ __forceinline__ uint64_t gate_exp_x2(float x0, float x1) {
    const uint64_t x = f2(x0, x1);
    const uint64_t n_f = f2_sub(f2_fma(x, f2(0x1.715476p+0f, 0x1.715476p+0f), f2(0x1.8p23f, 0x1.8p23f)),
                                f2(0x1.8p23f, 0x1.8p23f));
    uint64_t r = f2_fma(n_f, f2(-0x1.62e43p-1f, -0x1.62e43p-1f), x);
    r = f2_fma(n_f, f2(0x1.05c61p-29f, 0x1.05c61p-29f), r);
    uint64_t p = f2(0x1.a01a02p-13f, 0x1.a01a02p-13f);
    p = f2_fma(p, r, f2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
    p = f2_fma(p, r, f2(0x1.111112p-7f, 0x1.111112p-7f));
    p = f2_fma(p, r, f2(0x1.555556p-5f, 0x1.555556p-5f));
    p = f2_fma(p, r, f2(0x1.555556p-3f, 0x1.555556p-3f));
    p = f2_fma(p, r, f2(0.5f, 0.5f));
    p = f2_fma(p, r, f2(1.0f, 1.0f));
    p = f2_fma(p, r, f2(1.0f, 1.0f));
    const float2 nf = f2_split(n_f);
    const int n0 = __float2int_rz(nf.x), n1 = __float2int_rz(nf.y);
    const int h0 = n0 / 2, h1 = n1 / 2;
    const float2 v = f2_split(f2_mul(f2_mul(p, f2(pow2_of(h0), pow2_of(h1))),
                                     f2(pow2_of(n0 - h0), pow2_of(n1 - h1))));
    const float r0 = (x0 != x0) ? x0 : (x0 > 88.75f ? kInf : (x0 < -104.0f ? 0.0f : v.x));
    const float r1 = (x1 != x1) ? x1 : (x1 > 88.75f ? kInf : (x1 < -104.0f ? 0.0f : v.y));
    return f2(r0, r1);
}

// u = 2^e m with m in [sqrt(1/2), sqrt(2)]: returns e as a float, m in m_out
__device__ __forceinline__ float log1p_reduce(float u, float &m_out) {
    const uint32_t ubits = __float_as_uint(u);
    int e = static_cast<int>(ubits >> 23) - 127;
    float m = __uint_as_float((ubits & 0x007fffffu) | 0x3f800000u);
    if (m > 0x1.6a09e6p+0f) {
        m = __fmul_rn(m, 0.5f);
        e += 1;
    }
    m_out = m;
    return static_cast<float>(e);
}

__device__ __forceinline__ uint64_t gate_log1p_x2(uint64_t y) {
    const uint64_t one = f2(1.0f, 1.0f);
    const uint64_t u = f2_add(one, y);
    const float2 y2 = f2_split(y), u2 = f2_split(u);
    float m0, m1;
    const float e0 = log1p_reduce(u2.x, m0), e1 = log1p_reduce(u2.y, m1);
    const uint64_t f = f2_sub(f2(m0, m1), one);
    const float2 num = f2_split(f2_sub(y, f2_sub(u, one)));
    const float2 fs = f2_split(f), den = f2_split(f2_add(f2(2.0f, 2.0f), f));
    const uint64_t corr = f2(__fdiv_rn(num.x, u2.x), __fdiv_rn(num.y, u2.y));
    const uint64_t s = f2(__fdiv_rn(fs.x, den.x), __fdiv_rn(fs.y, den.y));
    const uint64_t z = f2_mul(s, s);
    uint64_t R = f2(0x1.745d18p-3f, 0x1.745d18p-3f);
    R = f2_fma(R, z, f2(0x1.c71c72p-3f, 0x1.c71c72p-3f));
    R = f2_fma(R, z, f2(0x1.24924ap-2f, 0x1.24924ap-2f));
    R = f2_fma(R, z, f2(0x1.99999ap-2f, 0x1.99999ap-2f));
    R = f2_fma(R, z, f2(0x1.555556p-1f, 0x1.555556p-1f));
    // The rest per element: a packed product that feeds a packed sum may be
    // contracted into one fma by the assembler, which would change the bits.
    const float2 Rp = f2_split(R), zp = f2_split(z), sp = f2_split(s), cp = f2_split(corr);
    auto tail = [](float Ri, float zi, float si, float fi, float ci, float efi) {
        const float Rz = __fmul_rn(Ri, zi);
        const float t = __fmul_rn(si, __fsub_rn(fi, Rz));
        const float low = __fsub_rn(__fmaf_rn(efi, -0x1.05c61p-29f, ci), t);
        return __fmaf_rn(efi, 0x1.62e43p-1f, __fadd_rn(fi, low));
    };
    const float2 v = make_float2(tail(Rp.x, zp.x, sp.x, fs.x, cp.x, e0),
                                 tail(Rp.y, zp.y, sp.y, fs.y, cp.y, e1));
    auto special = [](float yy, float vv) {
        if (yy != yy || yy == kInf) return yy;
        if (yy <= -1.0f) return (yy == -1.0f) ? -kInf : __uint_as_float(0x7fc00000u);
        return vv;
    };
    return f2(special(y2.x, v.x), special(y2.y, v.y));
}

// The common case, both |x| < 87: exp(-|x|) has n = round(-|x| / ln2) in
// [-126, 0] and a normal result, and log1p sees y in (2^-126, 1].  There the
// special-case branches of the specification cannot trigger and scaling p by
// 2^n in one multiply gives the same bits as the two-step scaling (p 2^(n/2)
// is exact, so only the final product rounds, in both forms).
__device__ __forceinline__ uint64_t softplus_x2_common(float x0, float x1) {
    const uint64_t x = f2(-fabsf(x0), -fabsf(x1));
    const uint64_t n_f = f2_sub(f2_fma(x, f2(0x1.715476p+0f, 0x1.715476p+0f), f2(0x1.8p23f, 0x1.8p23f)),
                                f2(0x1.8p23f, 0x1.8p23f));
    uint64_t r = f2_fma(n_f, f2(-0x1.62e43p-1f, -0x1.62e43p-1f), x);
    r = f2_fma(n_f, f2(0x1.05c61p-29f, 0x1.05c61p-29f), r);
    uint64_t p = f2(0x1.a01a02p-13f, 0x1.a01a02p-13f);
    p = f2_fma(p, r, f2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
    p = f2_fma(p, r, f2(0x1.111112p-7f, 0x1.111112p-7f));
    p = f2_fma(p, r, f2(0x1.555556p-5f, 0x1.555556p-5f));
    p = f2_fma(p, r, f2(0x1.555556p-3f, 0x1.555556p-3f));
    p = f2_fma(p, r, f2(0.5f, 0.5f));
    p = f2_fma(p, r, f2(1.0f, 1.0f));
    p = f2_fma(p, r, f2(1.0f, 1.0f));
    const float2 nf = f2_split(n_f);
    const uint64_t y = f2_mul(p, f2(pow2_of(__float2int_rz(nf.x)), pow2_of(__float2int_rz(nf.y))));
    // log1p(y), y in (2^-126, 1]
    const uint64_t one = f2(1.0f, 1.0f);
    const uint64_t u = f2_add(one, y);
    const float2 u2 = f2_split(u);
    // u = 1 + y in (1, 2]: exponent 0 and m = u, or (u > sqrt 2, u = 2
    // included) exponent 1 and m = u / 2 -- what log1p_reduce gives there
    const bool h0 = u2.x > 0x1.6a09e6p+0f, h1 = u2.y > 0x1.6a09e6p+0f;
    const float e0 = h0 ? 1.0f : 0.0f, e1 = h1 ? 1.0f : 0.0f;
    const uint64_t f = f2_sub(f2_mul(u, f2(h0 ? 0.5f : 1.0f, h1 ? 0.5f : 1.0f)), one);
    const float2 fs = f2_split(f);
    const float2 cp = f2_split(div2_common(f2_sub(y, f2_sub(u, one)), u));
    const uint64_t s = div2_common(f, f2_add(f2(2.0f, 2.0f), f));
    const uint64_t z = f2_mul(s, s);
    uint64_t R = f2(0x1.745d18p-3f, 0x1.745d18p-3f);
    R = f2_fma(R, z, f2(0x1.c71c72p-3f, 0x1.c71c72p-3f));
    R = f2_fma(R, z, f2(0x1.24924ap-2f, 0x1.24924ap-2f));
    R = f2_fma(R, z, f2(0x1.99999ap-2f, 0x1.99999ap-2f));
    R = f2_fma(R, z, f2(0x1.555556p-1f, 0x1.555556p-1f));
    const float2 Rp = f2_split(R), zp = f2_split(z), sp = f2_split(s);
    auto tail = [](float Ri, float zi, float si, float fi, float ci, float efi) {
        const float Rz = __fmul_rn(Ri, zi);
        const float t = __fmul_rn(si, __fsub_rn(fi, Rz));
        const float low = __fsub_rn(__fmaf_rn(efi, -0x1.05c61p-29f, ci), t);
        return __fmaf_rn(efi, 0x1.62e43p-1f, __fadd_rn(fi, low));
    };
    const uint64_t lg = f2(tail(Rp.x, zp.x, sp.x, fs.x, cp.x, e0), tail(Rp.y, zp.y, sp.y, fs.y, cp.y, e1));
    // max(x, 0) + log1p: the sign of a zero max cannot show, log1p(e) > 0
    return f2_add(f2(fmaxf(x0, 0.0f), fmaxf(x1, 0.0f)), lg);
}

// g of two elements: gate_g(f0, dt0, a0) and gate_g(f1, dt1, a1)
__device__ __forceinline__ float2 gate_g_x2(float f0, float f1, float dt0, float dt1, float a0,
                                            float a1) {
    const float2 x = f2_split(f2_add(f2(f0, f1), f2(dt0, dt1)));
    uint64_t sp;
    if (fabsf(x.x) < 87.0f && fabsf(x.y) < 87.0f) {
        sp = softplus_x2_common(x.x, x.y);
    } else {
        const uint64_t e = gate_exp_x2(-fabsf(x.x), -fabsf(x.y));
        sp = f2_add(f2(x.x > 0.0f ? x.x : 0.0f, x.y > 0.0f ? x.y : 0.0f), gate_log1p_x2(e));
    }
    const float2 v = f2_split(f2_mul(f2(a0, a1), sp));
    return make_float2(-v.x, -v.y);
}

}  // namespace gate_spec
}  // namespace kda

// kda_gate_spec.cuh -- the binary32 specification of the KDA gate, shared by
// the gate kernel (kda_gate.cu) and the gated decode (kda_decode.cu), so that
// both produce the same bits:
//
//   g[n,h,c]  = -(exp(A_log[.]) * softplus(f[n,h,c] + dt_bias[h,c]))
//   beta[n,h] = 1 / (1 + exp(-b[n,h]))
//
// Every operation is an explicitly rounded intrinsic (__fadd_rn, __fmul_rn,
// __fmaf_rn, __fdiv_rn ...), which the compiler never contracts or reorders,
// and exp/log1p are this library's own:
//   exp:   Cody-Waite reduction (Cody and Waite, "Software Manual for the
//          Elementary Functions", 1980): n = round(x / ln2), r = x - n ln2 with
//          ln2 = head + tail, exp(r) by its Taylor polynomial through r^7 in
//          Horner form, 2^n applied as two exact powers of two.
//   log1p: u = 1 + y = 2^e m, m in [sqrt(1/2), sqrt(2)], f = m - 1,
//          s = f / (2 + f), log m = f - s (f - R(s^2)) with
//          R(z) = sum_j 2 z^j / (2j + 1) through z^5 (the atanh series,
//          Abramowitz and Stegun 4.1.27), plus c = (y - (u - 1)) / u for the
//          rounding of 1 + y and e ln2 with ln2 = head + tail.
#pragma once

#include "kda_internal.cuh"

namespace kda {
namespace gate_spec {

constexpr float kInf = __builtin_huge_valf();

__device__ __forceinline__ float pow2_of(int e) {  // 2^e, e in [-126, 127]
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

__device__ __forceinline__ float gate_exp(float x) {
    if (x != x) return x;
    if (x > 88.75f) return kInf;
    if (x < -104.0f) return 0.0f;
    const float kLog2e = 0x1.715476p+0f;
    const float kLn2Head = 0x1.62e43p-1f;
    const float kLn2Tail = -0x1.05c61p-29f;
    const float kShift = 0x1.8p23f;
    // n = round-to-nearest(x / ln2), exact inside the fma
    const float n_f = __fsub_rn(__fmaf_rn(x, kLog2e, kShift), kShift);
    float r = __fmaf_rn(n_f, -kLn2Head, x);
    r = __fmaf_rn(n_f, -kLn2Tail, r);
    // Taylor coefficients 1/j! for j = 7 .. 2, then 1, 1
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int n = __float2int_rz(n_f);
    const int half = n / 2;  // truncating division
    return __fmul_rn(__fmul_rn(p, pow2_of(half)), pow2_of(n - half));
}

__device__ __forceinline__ float gate_log1p(float y) {
    if (y != y) return y;
    if (y == kInf) return y;
    if (y <= -1.0f) return (y == -1.0f) ? -kInf : __uint_as_float(0x7fc00000u);
    const float kLn2Head = 0x1.62e43p-1f;
    const float kLn2Tail = -0x1.05c61p-29f;
    const float kSqrt2 = 0x1.6a09e6p+0f;
    const float u = __fadd_rn(1.0f, y);
    const uint32_t ubits = __float_as_uint(u);
    int e = static_cast<int>(ubits >> 23) - 127;
    float m = __uint_as_float((ubits & 0x007fffffu) | 0x3f800000u);
    if (m > kSqrt2) {
        m = __fmul_rn(m, 0.5f);
        e += 1;
    }
    const float f = __fsub_rn(m, 1.0f);
    const float corr = __fdiv_rn(__fsub_rn(y, __fsub_rn(u, 1.0f)), u);
    const float s = __fdiv_rn(f, __fadd_rn(2.0f, f));
    const float z = __fmul_rn(s, s);
    // 2/11, 2/9, 2/7, 2/5, 2/3
    float R = 0x1.745d18p-3f;
    R = __fmaf_rn(R, z, 0x1.c71c72p-3f);
    R = __fmaf_rn(R, z, 0x1.24924ap-2f);
    R = __fmaf_rn(R, z, 0x1.99999ap-2f);
    R = __fmaf_rn(R, z, 0x1.555556p-1f);
    R = __fmul_rn(R, z);
    const float t = __fmul_rn(s, __fsub_rn(f, R));
    const float ef = static_cast<float>(e);
    const float low = __fsub_rn(__fmaf_rn(ef, kLn2Tail, corr), t);
    return __fmaf_rn(ef, kLn2Head, __fadd_rn(f, low));
}

__device__ __forceinline__ float gate_softplus(float x) {
    const float positive = (x > 0.0f) ? x : 0.0f;
    return __fadd_rn(positive, gate_log1p(gate_exp(-fabsf(x))));
}

__device__ __forceinline__ float gate_sigmoid(float b) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, gate_exp(-b)));
}

__device__ __forceinline__ float gate_g(float f, float dt, float a) {
    return -__fmul_rn(a, gate_softplus(__fadd_rn(f, dt)));
}

__device__ __forceinline__ float alog_at(const float *A_log, int mode, int h, int c, int K) {
    return mode == 0 ? A_log[h] : (mode == 1 ? A_log[c] : A_log[static_cast<int64_t>(h) * K + c]);
}

}  // namespace gate_spec
}  // namespace kda

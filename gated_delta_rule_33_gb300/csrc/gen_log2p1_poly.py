"""Coefficients of the polynomial that the chunked prefill kernel uses for
log2(1 + e), e in [0, 1], in its in-kernel gate (softplus of the decay).

log2(1 + e) = e * P(e), with P the degree-7 Chebyshev interpolant of
log2(1 + e) / e on [0, 1] (interpolation at the Chebyshev points of the first
kind; L. N. Trefethen, "Approximation Theory and Approximation Practice",
SIAM 2013, chapters 3-4), converted to monomial form in e and rounded to fp32.
Run it to print the coefficients (lowest degree first) and the largest
relative error of the fp32 Horner evaluation on a fine grid of [0, 1]."""
import numpy as np

DEGREE = 7


def coefficients(n=DEGREE):
    k = np.arange(n + 1)
    x = np.cos((2 * k + 1) * np.pi / (2 * (n + 1)))  # nodes on [-1, 1]
    e = (x + 1) / 2
    c = np.polynomial.chebyshev.chebfit(x, np.log2(1 + e) / e, n)
    in_x = np.polynomial.Polynomial(np.polynomial.chebyshev.cheb2poly(c))
    in_e = in_x(np.polynomial.Polynomial([-1.0, 2.0]))  # x = 2e - 1
    return in_e.coef.astype(np.float32)


def max_rel_error(co, points=200001):
    e = np.linspace(0, 1, points).astype(np.float32)[1:]
    acc = np.full_like(e, co[-1])
    for a in co[-2::-1]:  # fp32 fused multiply-add per step
        acc = (acc.astype(np.float64) * e + np.float64(a)).astype(np.float32)
    val = (acc.astype(np.float64) * e).astype(np.float32)
    ref = np.log2(1 + e.astype(np.float64))
    return float(np.max(np.abs(val - ref) / ref))


if __name__ == "__main__":
    co = coefficients()
    for i, a in enumerate(co):
        print(f"c{i} = {float(a):.9g}f")
    print("max relative error", max_rel_error(co))

"""Pins for the oracle's fp32 gate specification.

The gate is g = -exp(A_log) softplus(f + dt_bias), beta = sigmoid(b)
(parameters as in K3_ARTIFACT_AUDIT.md sections 4.1 and 5.1; beta as a
sigmoid of the raw gate, per finding 1 of the Kimi-K3 expert-parallel
adapter review).  The oracle evaluates it with its own binary32 exp and
log1p; these tests pin those against fp64 libm (numpy) and against exact
special values.
"""
import math

import numpy as np
import pytest

import oracle


def ulp_error(approx, exact):
    ex32 = np.asarray(exact, dtype=np.float64).astype(np.float32)
    spacing = np.spacing(np.abs(ex32)).astype(np.float64)
    return np.abs(np.asarray(approx, dtype=np.float64) - exact) / spacing


def strided_float32(stride, lo, hi):
    bits = np.arange(0, 2 ** 32, stride, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    return x[np.isfinite(x) & (x >= lo) & (x <= hi)]


def test_exp_within_one_ulp_of_libm():
    x = strided_float32(251, -103.0, 88.72)
    err = ulp_error(oracle.exp_f32_array(x), np.exp(x.astype(np.float64)))
    assert err.max() < 1.0


def test_exp_subnormal_and_limits():
    x = np.linspace(-103.9, -87.4, 20001).astype(np.float32)
    y = oracle.exp_f32_array(x)
    ref = np.exp(x.astype(np.float64))
    # absolute error at most one subnormal spacing (2^-149) or one ulp
    tiny = 2.0 ** -149
    assert np.all(np.abs(y - ref) <= np.maximum(tiny, np.spacing(ref.astype(np.float32))))
    assert oracle.exp_f32(0.0) == 1.0
    assert oracle.exp_f32(-200.0) == 0.0
    assert math.isinf(oracle.exp_f32(89.0))
    assert math.isinf(oracle.exp_f32(float("inf")))
    assert oracle.exp_f32(float("-inf")) == 0.0
    assert math.isnan(oracle.exp_f32(float("nan")))
    assert np.isfinite(oracle.exp_f32(88.72))


def test_log1p_within_one_ulp_of_libm():
    x = strided_float32(241, -0.999, 3.0e38)
    ref = np.log1p(x.astype(np.float64))
    keep = np.abs(ref) > 1e-37
    err = ulp_error(oracle.log1p_f32_array(x[keep]), ref[keep])
    assert err.max() < 1.0


def test_log1p_special_values():
    assert oracle.log1p_f32(0.0) == 0.0
    assert oracle.log1p_f32(-1.0) == float("-inf")
    assert math.isnan(oracle.log1p_f32(-2.0))
    assert oracle.log1p_f32(float("inf")) == float("inf")
    assert oracle.log1p_f32(1e-30) == np.float32(1e-30)


def test_softplus_and_sigmoid_pins():
    # softplus(0) = ln 2 to within one ulp; sigmoid(0) = 1/2 exactly
    ln2 = np.float32(math.log(2.0))
    assert abs(oracle.softplus_f32(0.0) - float(ln2)) <= float(np.spacing(ln2))
    assert oracle.sigmoid_f32(0.0) == 0.5
    assert oracle.sigmoid_f32(-200.0) == 0.0
    assert oracle.sigmoid_f32(200.0) == 1.0
    xs = np.linspace(-40, 40, 4001).astype(np.float32)
    sp = np.array([oracle.softplus_f32(v) for v in xs])
    ref = np.logaddexp(0.0, xs.astype(np.float64))
    assert ulp_error(sp, ref).max() < 2.0
    sg = np.array([oracle.sigmoid_f32(v) for v in xs])
    ref = 1.0 / (1.0 + np.exp(-xs.astype(np.float64)))
    assert ulp_error(sg, ref).max() < 2.0
    # monotone non-decreasing on a sorted grid
    assert np.all(np.diff(sp) >= 0) and np.all(np.diff(sg) >= 0)


@pytest.mark.parametrize("mode", [oracle.ALOG_PER_HEAD, oracle.ALOG_PER_CHANNEL,
                                  oracle.ALOG_PER_HEAD_CHANNEL])
def test_gate_matches_fp64_composition(mode):
    r = np.random.default_rng(mode)
    N, H, K = 37, 3, 24
    f = r.standard_normal((N, H, K)).astype(np.float32)
    b = r.standard_normal((N, H)).astype(np.float32) * 3
    shape = {oracle.ALOG_PER_HEAD: (H,), oracle.ALOG_PER_CHANNEL: (K,),
             oracle.ALOG_PER_HEAD_CHANNEL: (H, K)}[mode]
    A_log = r.normal(-0.15, 0.3, shape).astype(np.float32)
    dt = r.normal(-4.6, 1.2, (H, K)).astype(np.float32)
    g, beta = oracle.gate(f, b, A_log, dt, mode)
    if mode == oracle.ALOG_PER_HEAD:
        a = np.exp(A_log.astype(np.float64))[None, :, None]
    elif mode == oracle.ALOG_PER_CHANNEL:
        a = np.exp(A_log.astype(np.float64))[None, None, :]
    else:
        a = np.exp(A_log.astype(np.float64))[None]
    x = (f + dt[None]).astype(np.float32).astype(np.float64)
    g_ref = -a * np.logaddexp(0.0, x)
    assert ulp_error(g, g_ref).max() < 4.0
    assert np.all(g <= 0)
    beta_ref = 1.0 / (1.0 + np.exp(-b.astype(np.float64)))
    assert ulp_error(beta, beta_ref).max() < 2.0
    assert np.all((beta >= 0) & (beta <= 1))

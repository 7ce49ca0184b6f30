"""Pins for the pre-step oracle (depthwise causal conv, kernel 4, SiLU, per-head
L2 norm), against things other than the oracle itself: a hand-worked example,
the impulse response, numpy's own convolution, closed forms of SiLU, unit
norms, and the packed-batch / carried-state structure."""
import json
import os

import numpy as np
import pytest

from oracle import shortconv as sc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_handworked_example():
    ex = json.load(open(os.path.join(GOLDEN, "shortconv_handworked.json")))
    x = np.array(ex["x"])[:, None]
    w = np.array(ex["w"])[None, :]
    st = np.array(ex["state"])[:, None]
    y, fin = sc.causal_conv(x, w, st)
    np.testing.assert_array_equal(y[:, 0], ex["conv"])
    np.testing.assert_array_equal(fin[:, 0], ex["final_state"])


def test_impulse_response_reads_taps_in_order():
    r = np.random.default_rng(0)
    C, L = 5, 12
    w = r.standard_normal((C, 4))
    for p in (0, 4, 10):
        x = np.zeros((L, C))
        x[p] = 1.0
        y, _ = sc.causal_conv(x, w)
        for j in range(L):
            d = j - p
            expect = w[:, 3 - d] if 0 <= d <= 3 else np.zeros(C)
            np.testing.assert_array_equal(y[j], expect)


def test_matches_numpy_convolve():
    r = np.random.default_rng(1)
    C, L = 7, 40
    x = r.standard_normal((L, C))
    w = r.standard_normal((C, 4))
    y, fin = sc.causal_conv(x, w)
    for c in range(C):
        ref = np.convolve(x[:, c], w[c, ::-1])[:L]
        np.testing.assert_allclose(y[:, c], ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(fin, x[-3:])


def test_silu_closed_forms():
    a = np.linspace(-30, 30, 241)
    s = sc.silu(a)
    assert sc.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(s - sc.silu(-a), a, rtol=0, atol=1e-12)   # x s(x) + x s(-x) = x
    np.testing.assert_allclose(sc.silu(np.array([40.0])), [40.0], rtol=1e-15)
    assert abs(sc.silu(np.array([-40.0]))[0]) < 1e-15
    np.testing.assert_allclose(sc.silu(np.array([1.0])), [1.0 / (1.0 + np.exp(-1.0))], rtol=1e-15)


def test_norm_gives_unit_heads_and_v_is_unnormalised():
    r = np.random.default_rng(2)
    H, D, N = 3, 128, 20
    x = r.standard_normal((N, H * D))
    w = r.standard_normal((H * D, 4)) * 0.5
    yq, _ = sc.short_conv(x, w, norm_dim=D)
    yv, _ = sc.short_conv(x, w, norm_dim=None)
    norms = np.linalg.norm(yq.reshape(N, H, D), axis=-1)
    np.testing.assert_allclose(norms, 1.0, rtol=1e-6)
    conv, _ = sc.causal_conv(x, w)
    np.testing.assert_allclose(yv, conv / (1 + np.exp(-conv)), rtol=1e-14)
    # the norm is a positive per-head rescale of the SiLU output
    ratio = yq.reshape(N, H, D) / yv.reshape(N, H, D)
    np.testing.assert_allclose(ratio, ratio[..., :1] * np.ones((1, 1, D)), rtol=1e-12)


def test_packed_batch_equals_separate_calls():
    r = np.random.default_rng(3)
    C = 256
    lens = [5, 0, 1, 2, 17, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = r.standard_normal((cu[-1], C))
    w = r.standard_normal((C, 4))
    S0 = r.standard_normal((len(lens), 3, C))
    y, fin = sc.short_conv(x, w, cu, S0, norm_dim=128)
    for s, L in enumerate(lens):
        ys, fs = sc.short_conv(x[cu[s]:cu[s + 1]], w, None, S0[s:s + 1], norm_dim=128)
        np.testing.assert_array_equal(y[cu[s]:cu[s + 1]], ys)
        np.testing.assert_array_equal(fin[s], fs[0])
    np.testing.assert_array_equal(fin[1], S0[1])                # empty: state passes through
    np.testing.assert_array_equal(fin[2], np.concatenate([S0[2, 1:], x[cu[2]:cu[3]]]))
    np.testing.assert_array_equal(fin[3], np.concatenate([S0[3, 2:], x[cu[3]:cu[4]]]))


@pytest.mark.parametrize("split", [1, 2, 3, 9])
def test_carried_state_equals_one_call(split):
    r = np.random.default_rng(4)
    C, L = 128, 12
    x = r.standard_normal((L, C))
    w = r.standard_normal((C, 4))
    S0 = r.standard_normal((1, 3, C))
    y, fin = sc.short_conv(x, w, None, S0, norm_dim=128)
    y1, f1 = sc.short_conv(x[:split], w, None, S0, norm_dim=128)
    y2, f2 = sc.short_conv(x[split:], w, None, f1, norm_dim=128)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(f2, fin)


def test_one_token_steps_equal_one_call():
    r = np.random.default_rng(5)
    C, L = 128, 6
    x = r.standard_normal((L, C))
    w = r.standard_normal((C, 4))
    y, fin = sc.short_conv(x, w, None, None)
    st = np.zeros((1, 3, C))
    for t in range(L):
        yt, st = sc.short_conv(x[t:t + 1], w, None, st)
        np.testing.assert_allclose(yt[0], y[t], rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(st, fin)

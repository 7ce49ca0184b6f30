"""Pins for the oracle's reverse mode (oracle.recurrent_backward), against
the forward recurrence it differentiates: central finite differences of the
scalar L = <dO, o> + <dS_T, S_T> for every input element of small problems,
Euler's identity for the inputs the outputs are homogeneous in, and the
closed form of a one-token step."""
import numpy as np
import pytest

import oracle


def problem(lens, H=2, K=3, V=2, seed=0, s0=True, dsf=True):
    r = np.random.default_rng(seed)
    N = sum(lens)
    q = r.standard_normal((N, H, K))
    k = r.standard_normal((N, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((N, H, V))
    g = -0.4 * np.abs(r.standard_normal((N, H, K)))
    beta = r.uniform(0.1, 0.9, (N, H))
    B = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    S0 = r.standard_normal((B, H, K, V)) * 0.5 if s0 else None
    dO = r.standard_normal((N, H, V))
    dSf = r.standard_normal((B, H, K, V)) if dsf else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu=cu, S0=S0, dO=dO, dSf=dSf)


def loss(p, scale, **over):
    a = dict(p, **over)
    o, S = oracle.recurrent(a["q"], a["k"], a["v"], a["g"], a["beta"], cu_seqlens=a["cu"],
                            scale=scale, initial_state=a["S0"], nthreads=1)
    L = float((a["dO"] * o).sum())
    if a["dSf"] is not None:
        L += float((a["dSf"] * S).sum())
    return L


def grads(p, scale):
    return oracle.recurrent_backward(p["q"], p["k"], p["v"], p["g"], p["beta"], p["dO"],
                                     cu_seqlens=p["cu"], scale=scale, initial_state=p["S0"],
                                     dS_final=p["dSf"], nthreads=1)


@pytest.mark.parametrize("lens,scale,s0,dsf", [([6], 1.0, False, False), ([6], 0.7, True, True),
                                                ([3, 0, 4, 1], 1.3, True, True)])
def test_finite_differences_every_element(lens, scale, s0, dsf):
    p = problem(lens, s0=s0, dsf=dsf, seed=len(lens))
    dq, dk, dv, dg, dbeta, dS0 = grads(p, scale)
    h = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv), ("g", dg), ("beta", dbeta),
                       ("S0", dS0 if s0 else None)):
        if grad is None:
            continue
        x = p[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            fd[idx] = (loss(p, scale, **{name: xp}) - loss(p, scale, **{name: xm})) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-7, err_msg=name)


def test_euler_identities():
    """o is linear in q; (o, S_T) is homogeneous of degree 1 in (v, S0)."""
    p = problem([9, 5], H=3, K=4, V=3, seed=5)
    scale = 0.9
    dq, dk, dv, dg, dbeta, dS0 = grads(p, scale)
    o, S = oracle.recurrent(p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=p["cu"],
                            scale=scale, initial_state=p["S0"])
    Lo = float((p["dO"] * o).sum())
    L = Lo + float((p["dSf"] * S).sum())
    np.testing.assert_allclose(float((dq * p["q"]).sum()), Lo, rtol=1e-12)
    np.testing.assert_allclose(float((dv * p["v"]).sum() + (dS0 * p["S0"]).sum()), L, rtol=1e-12)


def test_one_token_closed_form():
    r = np.random.default_rng(7)
    K, V, scale, b = 5, 4, 0.8, 0.35
    q, k, v, dO = r.standard_normal((1, 1, K)), r.standard_normal((1, 1, K)), \
        r.standard_normal((1, 1, V)), r.standard_normal((1, 1, V))
    g = -np.abs(r.standard_normal((1, 1, K)))
    beta = np.full((1, 1), b)
    dq, dk, dv, dg, dbeta, dS0 = oracle.recurrent_backward(q, k, v, g, beta, dO, scale=scale)
    qs, kk, vv, do = scale * q[0, 0], k[0, 0], v[0, 0], dO[0, 0]
    np.testing.assert_allclose(dq[0, 0], scale * b * (vv @ do) * kk, rtol=1e-13)
    np.testing.assert_allclose(dk[0, 0], b * (vv @ do) * qs, rtol=1e-13)
    np.testing.assert_allclose(dv[0, 0], b * (kk @ qs) * do, rtol=1e-13)
    np.testing.assert_allclose(dbeta[0, 0], (kk @ qs) * (vv @ do), rtol=1e-13)
    assert np.all(dg == 0.0)          # zero initial state: the decay acts on nothing
    np.testing.assert_allclose(dS0[0, 0], np.outer(np.exp(g[0, 0]), np.ones(V)) *
                               (np.outer(qs, do) - b * np.outer(kk, kk @ np.outer(qs, do))),
                               rtol=1e-12, atol=1e-14)

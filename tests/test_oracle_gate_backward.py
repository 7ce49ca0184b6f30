"""Pins for oracle/gate_backward.py: central finite differences of the fp64
gate L = <dg, g> + <dbeta, beta>, with g = -exp(A_log) log(1 + exp(f + dt_bias))
and beta = 1 / (1 + exp(-b)) written out here, for every input element."""
import numpy as np
import pytest

from oracle import gate_backward as gb


def gate64(f, b, A_log, dt, mode):
    N, H, K = f.shape
    A = {0: lambda: np.repeat(A_log[:, None], K, 1), 1: lambda: np.repeat(A_log[None, :], H, 0),
         2: lambda: A_log.reshape(H, K)}[mode]()
    g = -np.exp(A)[None] * np.log1p(np.exp(f + dt[None]))
    beta = 1.0 / (1.0 + np.exp(-b))
    return g, beta


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_finite_differences(mode):
    r = np.random.default_rng(mode)
    N, H, K = 3, 2, 4
    f = r.standard_normal((N, H, K))
    b = r.standard_normal((N, H))
    A_log = r.normal(-0.15, 0.3, {0: (H,), 1: (K,), 2: (H, K)}[mode])
    dt = r.normal(-1.0, 1.0, (H, K))
    dg = r.standard_normal((N, H, K))
    dbeta = r.standard_normal((N, H))

    def loss(f_, b_, A_, dt_):
        g, beta = gate64(f_, b_, A_, dt_, mode)
        return float((dg * g).sum() + (dbeta * beta).sum())

    df, db, dA, ddt = gb.gate_backward(f, b, A_log, dt, dg, dbeta, mode)
    h = 1e-6
    for name, x, grad in (("f", f, df), ("b", b, db), ("A_log", A_log, dA), ("dt", dt, ddt)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"f": (f, b, A_log, dt), "b": (f, b, A_log, dt), "A_log": (f, b, A_log, dt),
                    "dt": (f, b, A_log, dt)}[name]
            pos = ("f", "b", "A_log", "dt").index(name)
            ap, am = list(args), list(args)
            ap[pos], am[pos] = xp, xm
            fd[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_without_beta():
    r = np.random.default_rng(9)
    f = r.standard_normal((2, 1, 3))
    df, db, dA, ddt = gb.gate_backward(f, None, np.zeros(3), np.zeros((1, 3)),
                                       np.ones((2, 1, 3)), None, 1)
    assert db is None
    # a = 1, dt = 0: df = -sigmoid(f)
    np.testing.assert_allclose(df, -1.0 / (1.0 + np.exp(-f)), rtol=1e-14)

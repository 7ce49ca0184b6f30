"""Gradients of the KDA gate -- test infrastructure only (see oracle/__init__).

The gate (K3_ARTIFACT_AUDIT.md sections 4.1 and 5.1; the KDA layer of the
Kimi-K3 checkpoint) maps its inputs to the log-decay and the delta-rule step:

    x = f + dt_bias,  a = exp(A_log),  g = -a * softplus(x),  beta = sigmoid(b)

Its derivatives, written out in fp64 (softplus' = sigmoid, sigmoid' =
sigmoid (1 - sigmoid), d g / d A_log = g):

    df = dg * (-a * sigmoid(x)),     d dt_bias[h, c] = sum over tokens of df
    d A_log = sum of dg * g over every axis A_log is broadcast along
    db = dbeta * beta * (1 - beta)

Pinned (tests/test_oracle_gate_backward.py) by central finite differences of
the fp64 gate written out in the test, for every input element and all three
A_log layouts.
"""
from __future__ import annotations

import numpy as np

ALOG_PER_HEAD = 0
ALOG_PER_CHANNEL = 1
ALOG_PER_HEAD_CHANNEL = 2


def _alog_hk(A_log, mode, H, K):
    A = np.asarray(A_log, dtype=np.float64)
    if mode == ALOG_PER_HEAD:
        return np.broadcast_to(A[:, None], (H, K))
    if mode == ALOG_PER_CHANNEL:
        return np.broadcast_to(A[None, :], (H, K))
    return A.reshape(H, K)


def _sigmoid(x):
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def gate_backward(f, b, A_log, dt_bias, dg, dbeta, mode=ALOG_PER_CHANNEL):
    """f, dg [N, H, K]; b, dbeta [N, H] or None; A_log per mode; dt_bias [H, K].
    Returns (df [N,H,K], db [N,H] or None, dA_log (shape of A_log), ddt_bias [H,K])."""
    f = np.asarray(f, dtype=np.float64)
    N, H, K = f.shape
    dg = np.asarray(dg, dtype=np.float64)
    a = np.exp(_alog_hk(A_log, mode, H, K))
    x = f + np.asarray(dt_bias, dtype=np.float64)[None]
    sp = np.logaddexp(0.0, x)
    g = -a[None] * sp
    df = dg * (-a[None] * _sigmoid(x))
    ddt = df.sum(axis=0)
    t = (dg * g).sum(axis=0)                 # [H, K]
    if mode == ALOG_PER_HEAD:
        dA = t.sum(axis=1)
    elif mode == ALOG_PER_CHANNEL:
        dA = t.sum(axis=0)
    else:
        dA = t
    db = None
    if b is not None:
        s = _sigmoid(np.asarray(b, dtype=np.float64))
        db = np.asarray(dbeta, dtype=np.float64) * s * (1.0 - s)
    return df, db, dA, ddt

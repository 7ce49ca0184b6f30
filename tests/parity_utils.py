"""Helpers shared by the GPU parity tests: run libkda on cuda:0 and the CPU
oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances: relative L2 error against the fp64 oracle.
O_TOL = 2e-3
STATE_TOL = 1e-3

DEV = torch.device("cuda:0")


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    denom = np.linalg.norm(b)
    if denom == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / denom)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def oracle_gate(x):
    """The oracle's fp32 gate on the exact stored values of f and b."""
    return oracle.gate(x.f.float().numpy(), x.b.float().numpy(), x.A_log.numpy(),
                       x.dt_bias.numpy(), x.alog_mode)


def gpu_gate(kda, x):
    return kda.gate(x.f.to(DEV), x.b.to(DEV), x.A_log.to(DEV), x.dt_bias.to(DEV), x.alog_mode)


def oracle_prefill(x, g, beta, heads=None, scale=1.0):
    """fp64 recurrence for all heads or a subset (heads are independent)."""
    q, k, v = f64(x.q), f64(x.k), f64(x.v)
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    S0 = None if x.initial_state is None else f64(x.initial_state)
    if heads is not None:
        q, k, v, g = q[:, heads], k[:, heads], v[:, heads], g[:, heads]
        beta = beta[:, heads]
        if S0 is not None:
            S0 = S0[:, heads]
    cu = None if x.cu_seqlens is None else x.cu_seqlens.numpy()
    return oracle.recurrent(q, k, v, g, beta, cu_seqlens=cu, scale=scale, initial_state=S0)

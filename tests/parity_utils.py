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


def per_unit_rel_l2(a, b, cu_seqlens=None):
    """Largest relative L2 error over the (sequence, head) units of a token
    tensor [N, H, D] (``cu_seqlens`` splits N; None = one sequence) or of a
    state tensor [B, H, K, V] (``cu_seqlens`` ignored).  Units whose reference
    is all zero (empty sequences) are skipped.  One wrong chunk, head or
    sequence shows here even where the error pooled over the whole tensor stays
    under its bound."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    worst = 0.0
    if a.ndim == 4:
        units = [(a[i, h], b[i, h]) for i in range(a.shape[0]) for h in range(a.shape[1])]
    else:
        cu = [0, a.shape[0]] if cu_seqlens is None else [int(c) for c in np.asarray(cu_seqlens)]
        units = [(a[cu[i]:cu[i + 1], h], b[cu[i]:cu[i + 1], h])
                 for i in range(len(cu) - 1) for h in range(a.shape[1])]
    for ua, ub in units:
        nb = np.linalg.norm(ub)
        if nb == 0:
            continue
        worst = max(worst, float(np.linalg.norm(ua - ub) / nb))
    return worst


def assert_parity(o_g, o_ref, S_g, S_ref, cu_seqlens=None):
    """The prefill bounds, pooled over the tensors and for every (sequence,
    head) unit on its own: o within O_TOL and the final state within
    STATE_TOL."""
    cu = None if cu_seqlens is None else np.asarray(cu_seqlens)
    e_o, e_s = rel_l2(o_g, o_ref), rel_l2(S_g, S_ref)
    u_o, u_s = per_unit_rel_l2(o_g, o_ref, cu), per_unit_rel_l2(S_g, S_ref)
    assert e_o <= O_TOL, f"o rel-L2 {e_o:.3e}"
    assert e_s <= STATE_TOL, f"state rel-L2 {e_s:.3e}"
    assert u_o <= O_TOL, f"o rel-L2 of the worst (sequence, head) {u_o:.3e}"
    assert u_s <= STATE_TOL, f"state rel-L2 of the worst (sequence, head) {u_s:.3e}"
    return e_o, e_s


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

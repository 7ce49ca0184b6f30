"""CPU oracle for the KDA input pre-step -- test infrastructure only.

The Kimi-K3 checkpoint stores one depthwise causal convolution per projection
stream, ``q/k/v_conv1d.weight`` of shape [12288, 1, 4] in fp32 (96 heads x 128
dims, kernel size 4; K3_ARTIFACT_AUDIT.md section 4.1, KDA tensor table).  The
pages give only the weight shape; the readings taken where they are silent:

* causal, no bias (the checkpoint lists no bias tensor): for channel c and a
  token at position p of its sequence,
      y[p, c] = sum_{j=0..3} w[c, j] * x[p - 3 + j, c],
  so tap 3 weighs the current token and tap 0 the token three back;
* positions before the sequence start read the sequence's carried conv state
  (the last three inputs of the previous segment, oldest first), zero when
  there is none; sequences of a packed batch never see each other;
* the convolution output goes through SiLU, a * sigmoid(a);
* q and k are then L2-normalised per (token, head) over the head dimension:
  y / sqrt(sum y^2 + eps) with eps = 1e-6; v is not normalised;
* the carried state after a segment is its last three inputs (state rows
  filling in when the segment is shorter than three tokens).

Everything here is fp64 numpy on the exact input values (bf16 inputs widened
exactly, fp32 weights).  Plain loops over sequences and taps, no blocking.

Pins (tests/test_oracle_shortconv.py): the impulse response reads the taps
in order; each channel equals numpy's full convolution with the reversed taps;
SiLU closed forms; unit norms; packed batch = separate calls; a split segment
with its carried state = one call; one-token steps = one call.
"""
from __future__ import annotations

import numpy as np

KERNEL = 4
EPS = 1e-6


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def silu(a):
    a = np.asarray(a, dtype=np.float64)
    return a / (1.0 + np.exp(-a))


def causal_conv(x, w, state=None):
    """One segment.  x [L, C], w [C, 4], state [3, C] or None (zeros).
    Returns (conv output [L, C] before the activation, new state [3, C])."""
    x = _f64(x)
    w = _f64(w)
    L, C = x.shape
    prev = np.zeros((KERNEL - 1, C)) if state is None else _f64(state)
    xp = np.concatenate([prev, x], axis=0)          # row i holds position i - 3
    y = np.zeros((L, C))
    for j in range(KERNEL):                         # tap j reads position p - 3 + j
        y += w[:, j][None, :] * xp[j:j + L]
    return y, xp[L:L + KERNEL - 1].copy()


def l2norm_heads(a, head_dim, eps=EPS):
    """Normalise each group of head_dim consecutive channels of each row."""
    a = _f64(a)
    L, C = a.shape
    g = a.reshape(L, C // head_dim, head_dim)
    n = np.sqrt((g * g).sum(axis=-1, keepdims=True) + eps)
    return (g / n).reshape(L, C)


def short_conv(x, w, cu_seqlens=None, state=None, norm_dim=None, eps=EPS):
    """The pre-step over a packed batch.

    x [N, C] (one projection stream, C = H * head_dim), w [C, 4],
    cu_seqlens int [B+1] or None (one sequence), state [B, 3, C] or None.
    norm_dim: head_dim for q and k (L2 norm per head), None for v.
    Returns (y [N, C] fp64, final_state [B, 3, C] fp64)."""
    x = _f64(x)
    N, C = x.shape
    cu = np.array([0, N]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    B = len(cu) - 1
    y = np.zeros((N, C))
    final = np.zeros((B, KERNEL - 1, C))
    for s in range(B):
        lo, hi = int(cu[s]), int(cu[s + 1])
        st = None if state is None else _f64(state)[s]
        a, final[s] = causal_conv(x[lo:hi], w, st)
        a = silu(a)
        if norm_dim is not None and hi > lo:
            a = l2norm_heads(a, norm_dim, eps)
        y[lo:hi] = a
    return y, final

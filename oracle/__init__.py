"""CPU oracle for Kimi Delta Attention (KDA) -- test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the libkda C-ABI
library and ``gated_delta_rule_33_gb300``) never imports it, and it never
imports the product: the two share nothing but the seeded input generators.

The C source ``kdaref.c`` holds the oracle proper:

* ``recurrent``  -- the fp64 token-by-token KDA recurrence
  S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T,
  o_t = S_t^T (scale q_t); the two KDA regimes (chunked prefill, recurrent
  decode) are named in the Kimi-K3 code audit, data/code-audit.json, finding
  "dual-kda-execution-regimes".
* ``chunked``    -- the same result via the fp64 chunked (WY/UT) form.
* ``recurrent_backward`` -- the reverse mode of the recurrence (gradients of
  q, k, v, g, beta and the initial state): the training regime ("chunked KDA
  for training", code-audit.json, finding "dual-kda-execution-regimes").
* ``gate``       -- the fp32 gate specification g = -exp(A_log) softplus(f +
  dt_bias), beta = sigmoid(b), built on the oracle's own binary32 exp/log1p
  (parameters as in K3_ARTIFACT_AUDIT.md sections 4.1 and 5.1).

Pins (see tests/test_oracle_*.py): brute-force matrix products, the product
form of the state, chunked-vs-recurrent equivalence, the delta-rule
invariant, closed-form special cases, a Frobenius-norm bound, varlen and
continuation structure, linearity, and ulp error of exp/log1p against
fp64 libm.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kdaref.c")
_LIB = os.path.join(_HERE, "libkdaref.so")
_lock = threading.Lock()
_lib = None

ALOG_PER_HEAD = 0
ALOG_PER_CHANNEL = 1
ALOG_PER_HEAD_CHANNEL = 2


def build(force: bool = False) -> str:
    """Compile kdaref.c into libkdaref.so (plain gcc, no contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", _LIB + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        f32 = ctypes.c_float
        for name in ("kdaref_exp_f32", "kdaref_log1p_f32", "kdaref_softplus_f32",
                     "kdaref_sigmoid_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [f32]
            fn.restype = f32
        P = ctypes.c_void_p
        for name in ("kdaref_exp_f32_array", "kdaref_log1p_f32_array"):
            fn = getattr(lib, name)
            fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            fn.restype = None
        lib.kdaref_gate_f32.argtypes = [P, P, P, ctypes.c_int, P, P, P, ctypes.c_int64,
                                        ctypes.c_int, ctypes.c_int]
        lib.kdaref_gate_f32.restype = None
        common = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_double, P, P, P]
        lib.kdaref_recurrent.argtypes = common + [ctypes.c_int]
        lib.kdaref_recurrent.restype = ctypes.c_int
        lib.kdaref_chunked.argtypes = common + [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.kdaref_chunked.restype = ctypes.c_int
        c_i, c_i64, c_d = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.kdaref_recurrent_backward.argtypes = [P, P, P, P, P, P, c_i, c_i64, c_i, c_i, c_i,
                                                  c_d, P, P, P, P, P, P, P, P, P, c_i]
        lib.kdaref_recurrent_backward.restype = c_i
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# --- scalar fp32 specification ------------------------------------------------

def exp_f32(x: float) -> float:
    return _load().kdaref_exp_f32(float(x))


def log1p_f32(y: float) -> float:
    return _load().kdaref_log1p_f32(float(y))


def softplus_f32(x: float) -> float:
    return _load().kdaref_softplus_f32(float(x))


def sigmoid_f32(x: float) -> float:
    return _load().kdaref_sigmoid_f32(float(x))


def exp_f32_array(x) -> np.ndarray:
    """exp_f32 element-wise over an array."""
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty_like(flat)
    _load().kdaref_exp_f32_array(_ptr(flat), _ptr(out), flat.size)
    return out.reshape(np.shape(x))


def log1p_f32_array(x) -> np.ndarray:
    """log1p_f32 element-wise over an array."""
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty_like(flat)
    _load().kdaref_log1p_f32_array(_ptr(flat), _ptr(out), flat.size)
    return out.reshape(np.shape(x))


# --- gate ---------------------------------------------------------------------

def gate(f, b, A_log, dt_bias, alog_mode: int = ALOG_PER_CHANNEL):
    """fp32 gate spec. f [N,H,K] (fp32 values; bf16 inputs widened exactly),
    b [N,H] logits or None, A_log per alog_mode, dt_bias [H,K].
    Returns (g [N,H,K] fp32, beta [N,H] fp32 or None)."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    N, H, K = f.shape
    A_log = np.ascontiguousarray(A_log, dtype=np.float32)
    expect = {ALOG_PER_HEAD: (H,), ALOG_PER_CHANNEL: (K,), ALOG_PER_HEAD_CHANNEL: (H, K)}
    if A_log.shape != expect[alog_mode]:
        raise ValueError(f"A_log shape {A_log.shape} does not match mode {alog_mode}")
    dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32).reshape(H, K)
    g = np.empty_like(f)
    beta = None
    if b is not None:
        b = np.ascontiguousarray(b, dtype=np.float32).reshape(N, H)
        beta = np.empty((N, H), dtype=np.float32)
    _load().kdaref_gate_f32(_ptr(f), _ptr(b), _ptr(A_log), alog_mode, _ptr(dt_bias), _ptr(g),
                            _ptr(beta), N, H, K)
    return g, beta


# --- recurrence / chunked -----------------------------------------------------

def _run(fn_name, q, k, v, g, beta, cu_seqlens, scale, initial_state, extra, nthreads):
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    N, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is None:
        B = 1
        cu = None
    else:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        B = cu.shape[0] - 1
    S0 = _f64(initial_state)
    if S0 is not None and S0.shape != (B, H, K, V):
        raise ValueError(f"initial_state shape {S0.shape} != {(B, H, K, V)}")
    o = np.zeros((N, H, V), dtype=np.float64)
    S = np.zeros((B, H, K, V), dtype=np.float64)
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = getattr(_load(), fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu), B, N,
                                   H, K, V, float(scale), _ptr(S0), _ptr(o), _ptr(S), *extra, nt)
    if rc != 0:
        raise ValueError(f"{fn_name} rejected its arguments (code {rc})")
    return o, S


def recurrent(q, k, v, g, beta, cu_seqlens=None, scale=1.0, initial_state=None, nthreads=None):
    """fp64 KDA recurrence. q,k [N,H,K], v [N,H,V], g [N,H,K], beta [N,H].
    Returns (o [N,H,V] fp64, final_state [B,H,K,V] fp64)."""
    return _run("kdaref_recurrent", q, k, v, g, beta, cu_seqlens, scale, initial_state, (),
                nthreads)


def chunked(q, k, v, g, beta, cu_seqlens=None, scale=1.0, initial_state=None, chunk=64,
            frame=16, nthreads=None):
    """fp64 chunked (WY/UT) KDA; frame < chunk uses the per-frame factorisation."""
    return _run("kdaref_chunked", q, k, v, g, beta, cu_seqlens, scale, initial_state,
                (int(chunk), int(frame)), nthreads)


def recurrent_backward(q, k, v, g, beta, dO, cu_seqlens=None, scale=1.0, initial_state=None,
                       dS_final=None, nthreads=None):
    """Reverse mode of ``recurrent``: given dO [N,H,V] and dS_final [B,H,K,V]
    (None: zero), returns (dq, dk, dv, dg [N,H,K or V], dbeta [N,H],
    dS0 [B,H,K,V]) in fp64."""
    q, k, v, g, beta, dO = (_f64(a) for a in (q, k, v, g, beta, dO))
    N, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is None:
        B, cu = 1, None
    else:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        B = cu.shape[0] - 1
    S0, dSf = _f64(initial_state), _f64(dS_final)
    for name, a in (("initial_state", S0), ("dS_final", dSf)):
        if a is not None and a.shape != (B, H, K, V):
            raise ValueError(f"{name} shape {a.shape} != {(B, H, K, V)}")
    dq, dk, dg = (np.zeros((N, H, K)) for _ in range(3))
    dv = np.zeros((N, H, V))
    dbeta = np.zeros((N, H))
    dS0 = np.zeros((B, H, K, V))
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = _load().kdaref_recurrent_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu), B, N, H, K, V, float(scale),
        _ptr(S0), _ptr(dO), _ptr(dSf), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
        _ptr(dS0), nt)
    if rc != 0:
        raise ValueError(f"kdaref_recurrent_backward rejected its arguments (code {rc})")
    return dq, dk, dv, dg, dbeta, dS0


def decode(q, k, v, g, beta, state, scale=1.0, nthreads=None):
    """One recurrent step per sequence. q,k,g [B,H,K], v [B,H,V], beta [B,H],
    state [B,H,K,V]. Returns (o [B,H,V], new_state [B,H,K,V]) in fp64."""
    Bn = np.shape(q)[0]
    cu = np.arange(Bn + 1, dtype=np.int32)
    return recurrent(q, k, v, g, beta, cu_seqlens=cu, scale=scale, initial_state=state,
                     nthreads=nthreads)

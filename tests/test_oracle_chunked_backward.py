"""Pins for oracle/chunked_backward.py, the chunked (WY/UT) reverse mode: its
chunk forward reproduces the recurrence, and its gradients equal the
recurrent reverse mode of kdaref.c (pinned by finite differences in
test_oracle_backward.py) for every chunk length, ragged tails, empty
sequences, initial states, final-state gradients and a query scale."""
import numpy as np
import pytest

import oracle
from oracle import chunked_backward as cb
from gated_delta_rule_33_gb300 import synth


def _problem(lengths, H, D, seed, s0=True):
    x = synth.make_inputs(sum(lengths), H=H, D=D, seed=seed, lengths=lengths,
                          s0_std=0.05 if s0 else 0.0)
    g, beta = oracle.gate(x.f.float().numpy(), x.b.numpy(), x.A_log.numpy(), x.dt_bias.numpy(),
                          x.alog_mode)
    r = np.random.default_rng(seed + 100)
    N, B = sum(lengths), len(lengths)
    dO = r.standard_normal((N, H, D))
    dSf = r.standard_normal((B, H, D, D)) * 0.1
    S0 = None if x.initial_state is None else x.initial_state.double().numpy()
    return (x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy(), g.astype(np.float64),
            beta.astype(np.float64), x.cu_seqlens.numpy(), S0, dO, dSf)


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


@pytest.mark.parametrize("chunk", [4, 7, 16])
def test_chunk_forward_reproduces_the_recurrence(chunk):
    q, k, v, g, beta, cu, S0, _, _ = _problem([23, 0, 9], H=2, D=8, seed=1)
    o_ref, S_ref = oracle.recurrent(q, k, v, g, beta, cu_seqlens=cu, scale=0.7, initial_state=S0)
    for b in range(len(cu) - 1):
        t0, t1 = cu[b], cu[b + 1]
        for h in range(2):
            S = S0[b, h].copy()
            for c0 in range(t0, t1, chunk):
                c1 = min(c0 + chunk, t1)
                O, S = cb.chunk_forward(q[c0:c1, h], k[c0:c1, h], v[c0:c1, h], g[c0:c1, h],
                                        beta[c0:c1, h], S, 0.7)
                assert _rel(O, o_ref[c0:c1, h]) < 1e-12
            assert _rel(S, S_ref[b, h]) < 1e-12


@pytest.mark.parametrize("chunk", [1, 4, 5, 16, 64])
@pytest.mark.parametrize("s0", [False, True])
def test_chunked_gradients_equal_the_recurrent_reverse_mode(chunk, s0):
    q, k, v, g, beta, cu, S0, dO, dSf = _problem([37, 0, 12, 64], H=2, D=8, seed=2 + chunk, s0=s0)
    ref = oracle.recurrent_backward(q, k, v, g, beta, dO, cu_seqlens=cu, scale=0.9,
                                    initial_state=S0, dS_final=dSf)
    got = cb.chunked_backward(q, k, v, g, beta, dO, cu_seqlens=cu, scale=0.9, initial_state=S0,
                              dS_final=dSf, chunk=chunk)
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta", "dS0"), got, ref):
        assert _rel(a, b) < 1e-10, f"{name}: {_rel(a, b)}"


def test_chunked_gradients_at_k3_head_width():
    # d = 128 and the K3 decay distribution, one 150-token sequence, chunk 64
    q, k, v, g, beta, cu, S0, dO, dSf = _problem([150], H=1, D=128, seed=5)
    ref = oracle.recurrent_backward(q, k, v, g, beta, dO, cu_seqlens=cu, initial_state=S0,
                                    dS_final=dSf)
    got = cb.chunked_backward(q, k, v, g, beta, dO, cu_seqlens=cu, initial_state=S0,
                              dS_final=dSf, chunk=64)
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta", "dS0"), got, ref):
        assert _rel(a, b) < 1e-10, f"{name}: {_rel(a, b)}"

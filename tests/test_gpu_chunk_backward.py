"""GPU parity of kda_chunk_backward, the chunked tensor-core backward, against
the oracle's fp64 reverse mode (oracle.recurrent_backward) on the same q, k,
v, beta, g (the gate is bit-exact on both sides), dO and final-state gradient.

Tolerance: every gradient within relative L2 1e-3, pooled over the tensor and
for each (sequence, head) on its own.  The bound comes from the precision of
the chunked forms: the chunk-start states come from the tf32 forward (state
error about 4e-4), and a numpy emulation of a tf32 chunked backward against
the fp64 reverse mode gave 3.5e-4 .. 5.2e-4 on every gradient; the bf16
high/low split products used here are more precise than tf32 (a 16-bit
significand).  The shapes follow the exact-match shape set of
K3_ARTIFACT_AUDIT.md section 7.3 (one chunk, partial tails, several chunks,
varlen with empty sequences) plus the K3 head count at T = 4096 on sampled
heads."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_33_gb300 import synth
from parity_utils import DEV, f64, gpu_gate, oracle_gate, per_unit_rel_l2, rel_l2

pytestmark = pytest.mark.gpu
GRAD_TOL = 1e-3
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def make_case(lens=None, N=None, H=3, seed=0, s0=True, dsf=True, do_dtype=torch.bfloat16):
    x = synth.make_inputs(N, H=H, seed=seed, lengths=lens, s0_std=0.05 if s0 else 0.0)
    gen = torch.Generator().manual_seed(seed + 1000)
    dO = torch.randn(x.N, H, 128, generator=gen).to(do_dtype)
    dSf = torch.randn(x.B, H, 128, 128, generator=gen) * 0.1 if dsf else None
    return x, dO, dSf


def run_case(lib, x, dO, dSf, scale, heads=None, want_dS0=True, g=None):
    if g is None:
        g, beta = gpu_gate(lib, x)
        g_ref, b_ref = oracle_gate(x)
    else:
        _, beta = gpu_gate(lib, x)
        _, b_ref = oracle_gate(x)
        g_ref = g.cpu().numpy()
    cu = None if x.cu_seqlens is None else x.cu_seqlens.to(DEV)
    S0 = None if x.initial_state is None else x.initial_state.to(DEV)
    out = lib.backward_chunked(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, dO.to(DEV),
                               cu_seqlens=cu, scale=scale, initial_state=S0,
                               dS_final=None if dSf is None else dSf.to(DEV), want_dS0=want_dS0)
    assert lib.kda_get_last_device_error() == 0
    sel = slice(None) if heads is None else heads
    S0r = None if x.initial_state is None else f64(x.initial_state)[:, sel]
    dSr = None if dSf is None else f64(dSf)[:, sel]
    cu_np = None if x.cu_seqlens is None else x.cu_seqlens.numpy()
    ref = oracle.recurrent_backward(f64(x.q)[:, sel], f64(x.k)[:, sel], f64(x.v)[:, sel],
                                    np.asarray(g_ref, np.float64)[:, sel],
                                    np.asarray(b_ref, np.float64)[:, sel], f64(dO)[:, sel],
                                    cu_seqlens=cu_np, scale=scale, initial_state=S0r,
                                    dS_final=dSr, nthreads=8)
    for name, a, r in zip(NAMES, out, ref):
        if a is None:
            continue
        a64 = f64(a)[:, sel]
        assert np.isfinite(a64).all(), name
        err = rel_l2(a64, r)
        assert err <= GRAD_TOL, f"{name}: rel L2 {err:.3e}"
        unit = per_unit_rel_l2(a64, r, cu_np)
        assert unit <= GRAD_TOL, f"{name}: rel L2 of the worst (sequence, head) {unit:.3e}"
    return out


@pytest.mark.parametrize("N,s0,dsf,do_dtype,scale", [
    (1, False, False, torch.bfloat16, 1.0),
    (16, True, False, torch.float32, 1.0),
    (64, True, True, torch.bfloat16, 1.0),
    (65, False, True, torch.float32, 0.8),
    (200, True, True, torch.bfloat16, 1.0),
])
def test_single_sequence(lib, N, s0, dsf, do_dtype, scale):
    x, dO, dSf = make_case(N=N, s0=s0, dsf=dsf, do_dtype=do_dtype, seed=N)
    run_case(lib, x, dO, dSf, scale)


def test_varlen_with_short_and_empty_sequences(lib):
    x, dO, dSf = make_case(lens=[0, 1, 17, 130, 64, 33, 0, 5], H=2, seed=3)
    out = run_case(lib, x, dO, dSf, 128 ** -0.5)
    # an empty sequence passes dS_final straight through to dS0
    np.testing.assert_array_equal(out[5][0].cpu().numpy(), dSf[0].numpy())
    np.testing.assert_array_equal(out[5][6].cpu().numpy(), dSf[6].numpy())


def test_without_dS0(lib):
    x, dO, dSf = make_case(N=70, H=2, seed=4)
    out = run_case(lib, x, dO, dSf, 1.0, want_dS0=False)
    assert out[5] is None


def test_more_chains_than_ctas(lib):
    """200 sequences x 2 heads: the persistent CTAs take several chains each."""
    lens = synth.varlen_lengths(200, 1, 90, seed=9)
    x, dO, dSf = make_case(lens=lens, H=2, seed=9)
    run_case(lib, x, dO, dSf, 1.0)


def test_k3_t4096_sampled_heads(lib):
    """T = 4096, H = 96 in one launch (the training shape of the K3 layer);
    the oracle checks three heads."""
    x, dO, dSf = make_case(N=4096, H=96, seed=5)
    run_case(lib, x, dO, dSf, 1.0, heads=[0, 41, 95])


def test_agrees_with_the_recurrent_backward(lib):
    """The chunked and the token-by-token backward on the same inputs."""
    x, dO, dSf = make_case(lens=[150, 77], H=4, seed=6)
    g, beta = gpu_gate(lib, x)
    args = (x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, dO.to(DEV))
    kw = dict(cu_seqlens=x.cu_seqlens.to(DEV), initial_state=x.initial_state.to(DEV),
              dS_final=dSf.to(DEV))
    a = lib.backward_chunked(*args, **kw)
    b = lib.backward(*args, **kw)
    assert lib.kda_get_last_device_error() == 0
    for name, ga, gb in zip(NAMES, a, b):
        assert rel_l2(f64(ga), f64(gb)) <= GRAD_TOL, name


def test_chunk_decay_beyond_range_is_reported(lib):
    """A head whose chunk decay exceeds one chunk's range (-5 per token, 320
    per 64 tokens) has no aligned checkpoints: KDA_ERR_DECAY_RANGE, zero
    gradients for it, the other head still correct."""
    x, dO, dSf = make_case(N=130, H=2, seed=7)
    g, _ = gpu_gate(lib, x)
    g[:, 1] = -5.0
    dq, dk, dv, dg, dbeta, dS0 = lib.backward_chunked(
        x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, gpu_gate(lib, x)[1], dO.to(DEV),
        initial_state=x.initial_state.to(DEV), dS_final=dSf.to(DEV))
    assert lib.kda_get_last_device_error() == 11   # KDA_ERR_DECAY_RANGE
    for t in (dq, dk, dv, dg, dbeta, dS0):
        assert float(t[:, 1].abs().max()) == 0.0
    # head 0 as the oracle computes it
    _, b_ref = oracle_gate(x)
    ref = oracle.recurrent_backward(f64(x.q)[:, :1], f64(x.k)[:, :1], f64(x.v)[:, :1],
                                    f64(g)[:, :1], np.asarray(b_ref, np.float64)[:, :1],
                                    f64(dO)[:, :1], initial_state=f64(x.initial_state)[:, :1],
                                    dS_final=f64(dSf)[:, :1])
    for name, a, r in zip(NAMES, (dq, dk, dv, dg, dbeta, dS0), ref):
        assert rel_l2(f64(a)[:, :1], r) <= GRAD_TOL, name


def test_product_wait_that_runs_out_is_reported_then_next_call_is_correct(lib):
    """The backward's bounded waits on its tensor-core products (and those of
    its checkpointing forward pass) give up at the first poll under the test
    hook: KDA_ERR_DEVICE_TIMEOUT is recorded, every product still completes
    before the kernel exits, and a normal call right after is correct."""
    x, dO, dSf = make_case(lens=[130, 0, 60], H=2, seed=9)
    g, beta = gpu_gate(lib, x)
    assert lib.kda_get_last_device_error() == 0
    try:
        lib.kda_debug_set_wait_limit(-1, 0)
        lib.backward_chunked(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, dO.to(DEV),
                             cu_seqlens=x.cu_seqlens.to(DEV),
                             initial_state=x.initial_state.to(DEV), dS_final=dSf.to(DEV))
        st = lib.kda_get_last_device_error()
    finally:
        lib.kda_debug_set_wait_limit(-1, -1)
    assert st == 7, lib.kda_status_string(st)   # KDA_ERR_DEVICE_TIMEOUT
    run_case(lib, x, dO, dSf, 1.0)


def test_two_calls_write_the_same_bits(lib):
    """Every cross-warp sum (dg's decay terms, dbeta) is added in a fixed
    order: repeated calls on the same inputs give identical gradients."""
    x, dO, dSf = make_case(lens=[130, 7, 64, 200], H=8, seed=12)
    g, beta = gpu_gate(lib, x)
    args = (x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, dO.to(DEV))
    kw = dict(cu_seqlens=x.cu_seqlens.to(DEV), initial_state=x.initial_state.to(DEV),
              dS_final=dSf.to(DEV))
    first = lib.backward_chunked(*args, **kw)
    for _ in range(3):
        again = lib.backward_chunked(*args, **kw)
        for name, a, b in zip(NAMES, first, again):
            assert torch.equal(a, b), name
    assert lib.kda_get_last_device_error() == 0

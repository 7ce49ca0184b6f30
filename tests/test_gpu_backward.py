"""GPU parity of kda_recurrent_backward against the oracle's fp64 reverse mode
(oracle.recurrent_backward), on the same q, k, v, beta and g (the gate is
bit-exact on both sides) and the same dO.  The kernel runs in fp32, so every
gradient tensor must match within relative L2 1e-4."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_33_gb300 import synth
from parity_utils import DEV, f64, gpu_gate, oracle_gate, rel_l2

pytestmark = pytest.mark.gpu
GRAD_TOL = 1e-4
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def make_case(lens=None, N=None, H=3, seed=0, s0=True, dsf=True, do_dtype=torch.bfloat16):
    x = synth.make_inputs(N, H=H, seed=seed, lengths=lens, s0_std=0.05 if s0 else 0.0)
    gen = torch.Generator().manual_seed(seed + 1000)
    dO = torch.randn(x.N, H, 128, generator=gen).to(do_dtype)
    dSf = torch.randn(x.B, H, 128, 128, generator=gen) * 0.1 if dsf else None
    return x, dO, dSf


def run_case(lib, x, dO, dSf, scale, heads=None, want_dS0=True):
    g, beta = gpu_gate(lib, x)
    cu = None if x.cu_seqlens is None else x.cu_seqlens.to(DEV)
    S0 = None if x.initial_state is None else x.initial_state.to(DEV)
    out = lib.backward(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, dO.to(DEV), cu_seqlens=cu,
                       scale=scale, initial_state=S0,
                       dS_final=None if dSf is None else dSf.to(DEV), want_dS0=want_dS0)
    assert lib.kda_get_last_device_error() == 0
    g_ref, b_ref = oracle_gate(x)
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
        err = rel_l2(f64(a)[:, sel], r)
        assert err <= GRAD_TOL, f"{name}: rel L2 {err:.3e}"
    return out


@pytest.mark.parametrize("N,s0,dsf,do_dtype,scale", [
    (1, False, False, torch.bfloat16, 1.0),
    (16, True, False, torch.float32, 1.0),
    (100, True, True, torch.bfloat16, 0.8),
    (257, False, True, torch.float32, 1.0),
])
def test_single_sequence(lib, N, s0, dsf, do_dtype, scale):
    x, dO, dSf = make_case(N=N, s0=s0, dsf=dsf, do_dtype=do_dtype, seed=N)
    run_case(lib, x, dO, dSf, scale)


def test_varlen_with_short_and_empty_sequences(lib):
    x, dO, dSf = make_case(lens=[0, 1, 17, 40, 16, 33, 0, 5], H=2, seed=3)
    out = run_case(lib, x, dO, dSf, 1.0)
    # an empty sequence passes dS_final straight through to dS0
    np.testing.assert_array_equal(out[5][0].cpu().numpy(), dSf[0].numpy())


def test_without_dS0(lib):
    x, dO, dSf = make_case(N=40, H=2, seed=4)
    out = run_case(lib, x, dO, dSf, 1.0, want_dS0=False)
    assert out[5] is None


def test_t1024_four_heads(lib):
    x, dO, dSf = make_case(N=1024, H=4, seed=5)
    run_case(lib, x, dO, dSf, 1.0)


def test_k3_size_sampled_heads(lib):
    """T=4096, 96 heads on the GPU; the oracle checks two heads."""
    x, dO, dSf = make_case(N=4096, H=96, seed=6, s0=False, dsf=False)
    run_case(lib, x, dO, dSf, 1.0, heads=[7, 88])


def test_bad_cu_seqlens_reports(lib):
    x, dO, dSf = make_case(lens=[10, 10], H=1, seed=7)
    x.cu_seqlens[1] = 25
    g, beta = gpu_gate(lib, x)
    lib.backward(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, dO.to(DEV),
                 cu_seqlens=x.cu_seqlens.to(DEV))
    assert lib.kda_get_last_device_error() == 1


# --- gate backward -------------------------------------------------------------------------

@pytest.mark.parametrize("N,H,mode,f_fp32,b_bf16,with_beta", [
    (4096, 96, synth.ALOG_PER_CHANNEL, False, False, True),
    (300, 3, synth.ALOG_PER_HEAD, True, True, True),
    (77, 2, synth.ALOG_PER_HEAD_CHANNEL, False, False, False),
    (1, 1, synth.ALOG_PER_CHANNEL, False, False, True)])
def test_gate_backward(lib, N, H, mode, f_fp32, b_bf16, with_beta):
    """kda_gate_backward against the fp64 chain rule of the gate
    (oracle/gate_backward.py): every output within 1e-5 relative L2."""
    from oracle import gate_backward as gb
    x = synth.make_inputs(N, H=H, D=128, seed=N + mode, alog_mode=mode)
    f = x.f.float() if f_fp32 else x.f
    b = (x.b.to(torch.bfloat16) if b_bf16 else x.b) if with_beta else None
    gen = torch.Generator().manual_seed(N)
    dg = torch.randn(N, H, 128, generator=gen)
    dbeta = torch.randn(N, H, generator=gen) if with_beta else None
    df, db, dA, ddt = lib.gate_backward(f.to(DEV), None if b is None else b.to(DEV),
                                        x.A_log.to(DEV), x.dt_bias.to(DEV), dg.to(DEV),
                                        None if dbeta is None else dbeta.to(DEV), alog_mode=mode)
    assert lib.kda_get_last_device_error() == 0
    ref = gb.gate_backward(f.double().numpy(), None if b is None else b.double().numpy(),
                           x.A_log.double().numpy(), x.dt_bias.double().numpy(),
                           dg.double().numpy(), None if dbeta is None else dbeta.double().numpy(),
                           mode)
    for name, a, r in zip(("df", "db", "dA_log", "ddt_bias"), (df, db, dA, ddt), ref):
        if r is None:
            assert a is None
            continue
        err = rel_l2(f64(a), r)
        assert err <= 1e-5, f"{name}: rel L2 {err:.2e}"


def test_gate_backward_is_deterministic(lib):
    x = synth.make_inputs(2000, H=4, D=128, seed=5)
    dg = torch.randn(2000, 4, 128, device=DEV)
    dbeta = torch.randn(2000, 4, device=DEV)
    args = (x.f.to(DEV), x.b.to(DEV), x.A_log.to(DEV), x.dt_bias.to(DEV), dg, dbeta)
    r1 = lib.gate_backward(*args)
    r2 = lib.gate_backward(*args)
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)

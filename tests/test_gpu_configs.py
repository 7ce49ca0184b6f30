"""GPU parity on the two larger workloads, checked on sampled heads.

* Varlen packed prefill: 8 sequences with lengths drawn uniformly from
  [512, 8192], 96 heads, d = 128, zero initial states.
* Long context: one sequence of 65536 tokens with a nonzero initial state,
  followed by 128 single-token recurrent decode steps on fresh tokens; the
  outputs and the state after the last step are compared with one fp64
  oracle run over all 65664 tokens.
The oracle runs the sampled heads only (heads are independent)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_33_gb300 import synth
from parity_utils import (DEV, O_TOL, STATE_TOL, assert_parity, f64, gpu_gate, oracle_gate,
                          per_unit_rel_l2, rel_l2)

pytestmark = pytest.mark.gpu


def test_varlen_k3_batch(lib):
    lengths = synth.varlen_lengths(8, 512, 8192, seed=0)
    x = synth.make_inputs(lengths=lengths, H=96, D=128, seed=0)
    g, beta = gpu_gate(lib, x)
    o, Sf = lib.prefill(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, x.cu_seqlens.to(DEV),
                        1.0, None)
    assert lib.kda_get_last_device_error() == 0
    heads = [0, 47, 95]
    g_ref, b_ref = oracle_gate(x)
    o_ref, S_ref = oracle.recurrent(f64(x.q)[:, heads], f64(x.k)[:, heads], f64(x.v)[:, heads],
                                    g_ref[:, heads], b_ref[:, heads],
                                    cu_seqlens=x.cu_seqlens.numpy())
    assert_parity(f64(o)[:, heads], o_ref, f64(Sf)[:, heads], S_ref, x.cu_seqlens)


def test_long_context_then_decode(lib):
    T, H, steps = 65536, 96, 128
    heads = [5, 77]
    x = synth.make_inputs(T, H=H, D=128, seed=0, s0_std=0.05, device=DEV)
    g, beta = lib.gate(x.f, x.b, x.A_log, x.dt_bias, x.alog_mode)
    o, S = lib.prefill(x.q, x.k, x.v, g, beta, None, 1.0, x.initial_state, o_dtype=torch.float32)
    assert lib.kda_get_last_device_error() == 0
    # 128 decode steps on fresh tokens (their own seeded draws)
    d = synth.make_inputs(steps, H=H, D=128, seed=1, device=DEV)
    dg, dbeta = lib.gate(d.f, d.b, x.A_log, x.dt_bias, x.alog_mode)
    outs = []
    for t in range(steps):
        outs.append(lib.decode(d.q[t:t + 1].clone(), d.k[t:t + 1].clone(), d.v[t:t + 1].clone(),
                               dg[t:t + 1].clone(), dbeta[t:t + 1].clone(), S, 1.0,
                               o_dtype=torch.float32))
    od = torch.cat(outs)
    torch.cuda.synchronize()
    # oracle: the same 65664 tokens on the sampled heads, from the same S0
    sel = torch.tensor(heads, device=DEV)

    def cat(a, b):
        return torch.cat([a[:, sel], b[:, sel]]).cpu()
    f_all = cat(x.f, d.f).float().numpy()
    b_all = cat(x.b, d.b).numpy()
    g_ref, b_ref = oracle.gate(f_all, b_all, x.A_log.cpu().numpy(),
                               x.dt_bias[sel].cpu().numpy(), x.alog_mode)
    o_ref, S_ref = oracle.recurrent(cat(x.q, d.q).double().numpy(), cat(x.k, d.k).double().numpy(),
                                    cat(x.v, d.v).double().numpy(), g_ref, b_ref,
                                    initial_state=x.initial_state[:, sel].cpu().double().numpy())
    o_gpu = np.concatenate([f64(o[:, sel]), f64(od[:, sel])])
    assert_parity(o_gpu[:T], o_ref[:T], f64(S[:, sel]), S_ref)
    assert rel_l2(o_gpu[T:], o_ref[T:]) <= O_TOL
    assert per_unit_rel_l2(o_gpu[T:], o_ref[T:]) <= O_TOL
    # the prefill leg chunk by chunk: every 64-token chunk of every sampled head
    for c0 in range(0, T, 64):
        blk_ref = o_ref[c0:c0 + 64]
        assert per_unit_rel_l2(o_gpu[c0:c0 + 64], blk_ref) <= O_TOL, f"chunk at {c0}"

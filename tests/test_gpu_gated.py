"""GPU parity of the chunked prefill with the gate computed inside the kernel
(kda_chunk_prefill_gated): o and final states against the fp64 oracle, whose
g and beta come from the oracle's own fp32 gate specification."""
import numpy as np
import pytest
import torch

from gated_delta_rule_33_gb300 import synth
from parity_utils import (DEV, O_TOL, STATE_TOL, assert_parity, f64, oracle_gate, oracle_prefill,
                          rel_l2)

pytestmark = pytest.mark.gpu


def run_gated(lib, x, scale=1.0, o_dtype=torch.bfloat16, b_bf16=False):
    b = x.b.to(torch.bfloat16) if b_bf16 else x.b
    cu = None if x.cu_seqlens is None else x.cu_seqlens.to(DEV)
    S0 = None if x.initial_state is None else x.initial_state.to(DEV)
    o, Sf = lib.prefill_gated(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), x.f.to(DEV), b.to(DEV),
                              x.A_log.to(DEV), x.dt_bias.to(DEV), x.alog_mode, cu, scale, S0,
                              o_dtype=o_dtype)
    assert lib.kda_get_last_device_error() == 0
    return o, Sf, b


def check_gated(lib, x, scale=1.0, o_dtype=torch.bfloat16, b_bf16=False, heads=None):
    o, Sf, b = run_gated(lib, x, scale, o_dtype, b_bf16)
    x_ref = x
    if b_bf16:
        x_ref = synth.KDAInputs(x.q, x.k, x.v, x.f, b.float(), x.A_log, x.dt_bias, x.alog_mode,
                                x.cu_seqlens, x.initial_state)
    g_ref, beta_ref = oracle_gate(x_ref)
    o_ref, S_ref = oracle_prefill(x, g_ref, beta_ref, heads=heads, scale=scale)
    o_g, S_g = f64(o), f64(Sf)
    if heads is not None:
        o_g, S_g = o_g[:, heads], S_g[:, heads]
    assert_parity(o_g, o_ref, S_g, S_ref, x.cu_seqlens)


@pytest.mark.parametrize("lengths,H", [([16], 1), ([65], 2), ([17, 31], 2), ([200], 3)])
@pytest.mark.parametrize("b_bf16", [False, True])
def test_gated_shape_set(lib, lengths, H, b_bf16):
    x = synth.make_inputs(lengths=lengths, H=H, D=128, seed=11 + H)
    check_gated(lib, x, b_bf16=b_bf16)


@pytest.mark.parametrize("mode", [synth.ALOG_PER_HEAD, synth.ALOG_PER_CHANNEL,
                                  synth.ALOG_PER_HEAD_CHANNEL])
def test_gated_alog_modes_state_scale(lib, mode):
    x = synth.make_inputs(lengths=[150, 0, 70], H=4, D=128, seed=mode, s0_std=0.05,
                          alog_mode=mode)
    check_gated(lib, x, scale=128 ** -0.5, o_dtype=torch.float32)


def test_gated_k3_full_size_sampled_heads(lib):
    x = synth.make_inputs(4096, H=96, D=128, seed=0)
    check_gated(lib, x, heads=[3, 50, 94])


def test_gated_as_accurate_as_unfused_path(lib):
    """Same inputs through kda_gate_fused + kda_chunk_prefill and through the
    fused kernel.  Each path carries its own tf32 rounding, so they are compared
    through the oracle: the fused path must be within the tolerances and no less
    accurate than the unfused one (to 20 % plus 1e-5)."""
    x = synth.make_inputs(lengths=[300, 129], H=8, D=128, seed=5, s0_std=0.05)
    o1, S1, _ = run_gated(lib, x, o_dtype=torch.float32)
    g, beta = lib.gate(x.f.to(DEV), x.b.to(DEV), x.A_log.to(DEV), x.dt_bias.to(DEV), x.alog_mode)
    o2, S2 = lib.prefill(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, x.cu_seqlens.to(DEV),
                         1.0, x.initial_state.to(DEV), o_dtype=torch.float32)
    g_ref, beta_ref = oracle_gate(x)
    o_ref, S_ref = oracle_prefill(x, g_ref, beta_ref)
    e_o1, e_s1 = rel_l2(f64(o1), o_ref), rel_l2(f64(S1), S_ref)
    e_o2, e_s2 = rel_l2(f64(o2), o_ref), rel_l2(f64(S2), S_ref)
    assert e_o1 <= O_TOL and e_s1 <= STATE_TOL
    assert e_o1 <= 1.2 * e_o2 + 1e-5, (e_o1, e_o2)
    assert e_s1 <= 1.2 * e_s2 + 1e-5, (e_s1, e_s2)

"""GPU parity of kda_recurrent_decode_indexed: a pool of cached states
addressed by slot, fp32 or bf16 state storage.

fp32 pool: outputs and updated states within the parity tolerances.  bf16
pool: the oracle starts from the same bf16 state values; outputs within 2e-3
and the stored state within the bf16 rounding bound: relative L2 <= 2^-8
(the unit roundoff of bf16; the fp32 arithmetic before the final rounding
adds ~1e-6)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_33_gb300 import synth
from parity_utils import DEV, O_TOL, STATE_TOL, f64, rel_l2

pytestmark = pytest.mark.gpu

BF16_STATE_TOL = 2.0 ** -8


def make_case(B, slots, H=4, state_dtype=torch.float32, seed=3):
    d = synth.make_decode_inputs(B, H=H, seed=seed)
    P = max(int(s) for s in slots) + 3
    gen = torch.Generator().manual_seed(seed + 100)
    pool = (torch.randn(P, H, 128, 128, generator=gen) * 0.05).to(state_dtype)
    return d, pool


def oracle_indexed(d, pool_cpu, slots):
    g_ref, b_ref = oracle.gate(d.f.float().numpy(), d.b.numpy(), d.A_log.numpy(),
                               d.dt_bias.numpy(), d.alog_mode)
    act = [i for i, s in enumerate(slots) if s >= 0]
    S = pool_cpu.double().numpy()[[slots[i] for i in act]]
    o, Sn = oracle.decode(f64(d.q)[act], f64(d.k)[act], f64(d.v)[act], g_ref[act], b_ref[act], S)
    return act, o, Sn


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_indexed_decode(lib, state_dtype):
    slots = [5, 0, -1, 7, 2, -1, 1]
    d, pool = make_case(len(slots), slots, state_dtype=state_dtype)
    g, beta = lib.gate(d.f.to(DEV), d.b.to(DEV), d.A_log.to(DEV), d.dt_bias.to(DEV), d.alog_mode)
    pool_dev = pool.to(DEV)
    idx = torch.tensor(slots, dtype=torch.int32, device=DEV)
    o = lib.decode_indexed(d.q.to(DEV), d.k.to(DEV), d.v.to(DEV), g, beta, pool_dev, idx,
                           o_dtype=torch.float32)
    assert lib.kda_get_last_device_error() == 0
    act, o_ref, S_ref = oracle_indexed(d, pool, slots)
    assert rel_l2(f64(o)[act], o_ref) <= O_TOL
    inactive = [i for i, s in enumerate(slots) if s < 0]
    assert float(o[inactive].abs().max()) == 0.0
    S_gpu = pool_dev.cpu().double().numpy()
    tol = STATE_TOL if state_dtype == torch.float32 else BF16_STATE_TOL
    assert rel_l2(S_gpu[[slots[i] for i in act]], S_ref) <= tol
    untouched = [p for p in range(pool.shape[0]) if p not in slots]
    np.testing.assert_array_equal(S_gpu[untouched], pool.double().numpy()[untouched])


def test_indexed_decode_matches_dense_decode(lib):
    """slots = 0..B-1 on an fp32 pool is kda_recurrent_decode."""
    B = 6
    d = synth.make_decode_inputs(B, H=3, seed=8)
    g, beta = lib.gate(d.f.to(DEV), d.b.to(DEV), d.A_log.to(DEV), d.dt_bias.to(DEV), d.alog_mode)
    s1 = d.state.to(DEV)
    s2 = d.state.to(DEV)
    o1 = lib.decode(d.q.to(DEV), d.k.to(DEV), d.v.to(DEV), g, beta, s1, o_dtype=torch.float32)
    o2 = lib.decode_indexed(d.q.to(DEV), d.k.to(DEV), d.v.to(DEV), g, beta, s2,
                            torch.arange(B, dtype=torch.int32, device=DEV), o_dtype=torch.float32)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_indexed_decode_out_of_range_slot(lib):
    slots = [0, 9]
    d, pool = make_case(2, [0, 1], H=2)   # pool of 4 slots; slot 9 is out of range
    g, beta = lib.gate(d.f.to(DEV), d.b.to(DEV), d.A_log.to(DEV), d.dt_bias.to(DEV), d.alog_mode)
    pool_dev = pool.to(DEV)
    o = lib.decode_indexed(d.q.to(DEV), d.k.to(DEV), d.v.to(DEV), g, beta, pool_dev,
                           torch.tensor(slots, dtype=torch.int32, device=DEV),
                           o_dtype=torch.float32)
    assert lib.kda_get_last_device_error() == 1   # KDA_ERR_INVALID_ARG
    assert float(o[1].abs().max()) == 0.0
    np.testing.assert_array_equal(pool_dev[1:].cpu().numpy(), pool[1:].numpy())


@pytest.mark.parametrize("state_dtype,mode,f_fp32,b_bf16", [
    (torch.float32, synth.ALOG_PER_CHANNEL, False, False),
    (torch.bfloat16, synth.ALOG_PER_HEAD, True, True),
    (torch.float32, synth.ALOG_PER_HEAD_CHANNEL, False, True)])
def test_gated_decode_equals_gate_then_decode(lib, state_dtype, mode, f_fp32, b_bf16):
    """kda_recurrent_decode_gated forms g and beta with the gate's own binary32
    operations, so it must equal kda_gate_fused + the indexed decode bit for
    bit, and match the oracle."""
    slots = [3, -1, 0, 2]
    d = synth.make_decode_inputs(len(slots), H=3, seed=21, alog_mode=mode)
    P = 5
    gen = torch.Generator().manual_seed(77)
    pool = (torch.randn(P, 3, 128, 128, generator=gen) * 0.05).to(state_dtype)
    f = d.f.float() if f_fp32 else d.f
    b = d.b.to(torch.bfloat16) if b_bf16 else d.b
    q, k, v = d.q.to(DEV), d.k.to(DEV), d.v.to(DEV)
    idx = torch.tensor(slots, dtype=torch.int32, device=DEV)
    g, beta = lib.gate(f.to(DEV), b.to(DEV), d.A_log.to(DEV), d.dt_bias.to(DEV), mode)
    pool1, pool2 = pool.to(DEV), pool.to(DEV)
    o1 = lib.decode_indexed(q, k, v, g, beta, pool1, idx, o_dtype=torch.float32)
    o2 = lib.decode_gated(q, k, v, f.to(DEV), b.to(DEV), d.A_log.to(DEV), d.dt_bias.to(DEV),
                          pool2, alog_mode=mode, state_indices=idx, o_dtype=torch.float32)
    assert lib.kda_get_last_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(pool1, pool2)
    g_ref, b_ref = oracle.gate(f.float().numpy(), b.float().numpy(), d.A_log.numpy(),
                               d.dt_bias.numpy(), mode)
    act = [i for i, s in enumerate(slots) if s >= 0]
    S = pool.double().numpy()[[slots[i] for i in act]]
    o_ref, S_ref = oracle.decode(f64(d.q)[act], f64(d.k)[act], f64(d.v)[act], g_ref[act],
                                 b_ref[act], S)
    assert rel_l2(f64(o2)[act], o_ref) <= O_TOL
    tol = STATE_TOL if state_dtype == torch.float32 else BF16_STATE_TOL
    assert rel_l2(pool2.cpu().double().numpy()[[slots[i] for i in act]], S_ref) <= tol


def test_gated_decode_dense_slots(lib):
    """state_indices NULL: slot b for sequence b over an fp32 [B, H, 128, 128] state."""
    d = synth.make_decode_inputs(4, H=2, seed=22)
    s1, s2 = d.state.to(DEV), d.state.to(DEV)
    g, beta = lib.gate(d.f.to(DEV), d.b.to(DEV), d.A_log.to(DEV), d.dt_bias.to(DEV), d.alog_mode)
    o1 = lib.decode(d.q.to(DEV), d.k.to(DEV), d.v.to(DEV), g, beta, s1)
    o2 = lib.decode_gated(d.q.to(DEV), d.k.to(DEV), d.v.to(DEV), d.f.to(DEV), d.b.to(DEV),
                          d.A_log.to(DEV), d.dt_bias.to(DEV), s2, alog_mode=d.alog_mode)
    assert lib.kda_get_last_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(s1, s2)

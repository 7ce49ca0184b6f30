"""GPU parity: libkda on cuda:0 (through the C ABI) against the CPU oracle.

Gate: bit-exact.  Prefill and decode: relative L2 error <= 2e-3 on outputs and
<= 1e-3 on states against the fp64 recurrence, on the same seeded inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_33_gb300 import synth
from parity_utils import (DEV, O_TOL, STATE_TOL, assert_parity, f64, gpu_gate, oracle_gate,
                          oracle_prefill, rel_l2)

pytestmark = pytest.mark.gpu


# --- gate -----------------------------------------------------------------------------------

def test_gate_fast_division_is_ieee_division(lib):
    """The gate kernel's common path divides by Markstein's method (an fma
    correction of a refined reciprocal) instead of IEEE division; over every
    operand pair that path can form (about 1.07e9) the quotients are the same
    bits, so the gate stays bit-exact to its specification."""
    assert lib.kda_debug_check_gate_division() == 0


@pytest.mark.parametrize("mode", [synth.ALOG_PER_HEAD, synth.ALOG_PER_CHANNEL,
                                  synth.ALOG_PER_HEAD_CHANNEL])
def test_gate_bit_exact_k3_shape(lib, mode):
    x = synth.make_inputs(333, H=96, D=128, seed=mode, alog_mode=mode)
    g, beta = gpu_gate(lib, x)
    g_ref, beta_ref = oracle_gate(x)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g.cpu().numpy(), g_ref)
    np.testing.assert_array_equal(beta.cpu().numpy(), beta_ref)


def test_gate_bit_exact_fp32_inputs_and_generic_k(lib):
    # fp32 f and b, channel count not a multiple of 8 (the scalar path)
    x = synth.make_inputs(97, H=3, D=20, seed=5, dtype=torch.float32)
    x.b = x.b * 8.0  # push the sigmoid into its tails as well
    g, beta = gpu_gate(lib, x)
    g_ref, beta_ref = oracle_gate(x)
    np.testing.assert_array_equal(g.cpu().numpy(), g_ref)
    np.testing.assert_array_equal(beta.cpu().numpy(), beta_ref)


def test_gate_bit_exact_bf16_logits_and_extremes(lib):
    x = synth.make_inputs(64, H=4, D=128, seed=9)
    # extreme pre-activations: softplus tails, exp under/overflow of the pieces
    ext = torch.tensor([0.0, -0.0, 1e-30, -90.0, 90.0, 200.0, -200.0, 17.0, -17.0, 88.7])
    x.f = x.f.float()
    x.f.view(-1)[: ext.numel()] = ext
    x.f = x.f.to(torch.bfloat16)
    b16 = x.b.to(torch.bfloat16)
    g, beta = lib.gate(x.f.to(DEV), b16.to(DEV), x.A_log.to(DEV), x.dt_bias.to(DEV), x.alog_mode)
    g_ref, beta_ref = oracle.gate(x.f.float().numpy(), b16.float().numpy(), x.A_log.numpy(),
                                  x.dt_bias.numpy(), x.alog_mode)
    np.testing.assert_array_equal(g.cpu().numpy(), g_ref)
    np.testing.assert_array_equal(beta.cpu().numpy(), beta_ref)


def test_gate_without_beta(lib):
    x = synth.make_inputs(16, H=2, D=128, seed=2)
    g, beta = lib.gate(x.f.to(DEV), None, x.A_log.to(DEV), x.dt_bias.to(DEV), x.alog_mode)
    assert beta is None
    g_ref, _ = oracle_gate(x)
    np.testing.assert_array_equal(g.cpu().numpy(), g_ref)


# --- prefill --------------------------------------------------------------------------------

def run_prefill(lib, x, scale=1.0, o_dtype=torch.bfloat16):
    g, beta = gpu_gate(lib, x)
    cu = None if x.cu_seqlens is None else x.cu_seqlens.to(DEV)
    S0 = None if x.initial_state is None else x.initial_state.to(DEV)
    o, Sf = lib.prefill(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, cu, scale, S0,
                        o_dtype=o_dtype)
    assert lib.kda_get_last_device_error() == 0
    return o, Sf, g, beta


def check_prefill(lib, x, scale=1.0, o_dtype=torch.bfloat16, heads=None):
    o, Sf, g, beta = run_prefill(lib, x, scale, o_dtype)
    g_ref, beta_ref = oracle_gate(x)
    o_ref, S_ref = oracle_prefill(x, g_ref, beta_ref, heads=heads, scale=scale)
    o_g, S_g = f64(o), f64(Sf)
    if heads is not None:
        o_g, S_g = o_g[:, heads], S_g[:, heads]
    assert np.isfinite(o_g).all() and np.isfinite(S_g).all()
    return assert_parity(o_g, o_ref, S_g, S_ref, x.cu_seqlens)


# The exact-match shape set of K3_ARTIFACT_AUDIT.md section 7.3: one chunk, a
# partial tail, two chunks, multi-chunk multi-head, the K3 head count, and
# varlen with partial chunks (chunk 64, d = 128 here).
@pytest.mark.parametrize("lengths,H", [([16], 1), ([17], 1), ([32], 1), ([65], 2), ([17], 96),
                                       ([17, 31], 2), ([64], 2), ([128], 2), ([200], 3),
                                       ([1], 2)])
@pytest.mark.parametrize("o_dtype", [torch.bfloat16, torch.float32])
def test_prefill_shape_set(lib, lengths, H, o_dtype):
    x = synth.make_inputs(lengths=lengths, H=H, D=128, seed=len(lengths) * 7 + H)
    check_prefill(lib, x, o_dtype=o_dtype)


def test_prefill_initial_state_and_scale(lib):
    x = synth.make_inputs(lengths=[150, 64, 3], H=4, D=128, seed=3, s0_std=0.05)
    check_prefill(lib, x, scale=128 ** -0.5, o_dtype=torch.float32)


def test_prefill_varlen_with_empty_sequences(lib):
    x = synth.make_inputs(lengths=[0, 70, 0, 129, 1, 0], H=3, D=128, seed=4, s0_std=0.05)
    o, Sf, g, beta = run_prefill(lib, x, o_dtype=torch.float32)
    g_ref, beta_ref = oracle_gate(x)
    o_ref, S_ref = oracle_prefill(x, g_ref, beta_ref)
    assert_parity(f64(o), o_ref, f64(Sf), S_ref, x.cu_seqlens)
    # empty sequences: final state equals the initial state
    for i in (0, 2, 5):
        np.testing.assert_array_equal(Sf[i].cpu().numpy(), x.initial_state[i].numpy())


def test_prefill_tiny_config_padded(lib):
    """The d=16 oracle-scale case, zero-padded to d=128 (padded channels stay 0)."""
    x = synth.tiny_config()
    g_ref, beta_ref = oracle.gate(x.f.numpy(), x.b.numpy(), x.A_log.numpy(), x.dt_bias.numpy(),
                                  x.alog_mode)
    q16, k16, v16 = x.q.to(torch.bfloat16), x.k.to(torch.bfloat16), x.v.to(torch.bfloat16)
    o_ref, S_ref = oracle.recurrent(q16.double().numpy(), k16.double().numpy(),
                                    v16.double().numpy(), g_ref, beta_ref)

    def pad(t, dtype):
        out = torch.zeros(*t.shape[:-1], 128, dtype=dtype)
        out[..., :16] = t
        return out.to(DEV)
    g = pad(torch.from_numpy(g_ref), torch.float32)
    beta = torch.from_numpy(beta_ref).to(DEV)
    o, Sf = lib.prefill(pad(q16, torch.bfloat16), pad(k16, torch.bfloat16),
                        pad(v16, torch.bfloat16), g, beta, None, 1.0, None,
                        o_dtype=torch.float32)
    assert rel_l2(f64(o)[..., :16], o_ref) <= O_TOL
    assert rel_l2(f64(Sf)[..., :16, :16], S_ref) <= STATE_TOL
    assert float(o[..., 16:].abs().max()) == 0.0
    assert float(Sf[..., 16:, :].abs().max()) == 0.0 and float(Sf[..., :, 16:].abs().max()) == 0.0


def test_prefill_k3_full_size_sampled_heads(lib):
    """T = 4096, H = 96, d = 128 in the launch configuration the benchmark
    times; the oracle checks four sampled heads."""
    x = synth.make_inputs(4096, H=96, D=128, seed=0)
    check_prefill(lib, x, heads=[0, 31, 64, 95])


def test_prefill_bad_cu_seqlens_sets_device_error(lib):
    x = synth.make_inputs(lengths=[10, 20], H=2, D=128, seed=6)
    g, beta = gpu_gate(lib, x)
    cu = torch.tensor([0, 25, 20], dtype=torch.int32, device=DEV)  # not monotone
    o, Sf = lib.prefill(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, cu, 1.0, None)
    assert lib.kda_get_last_device_error() == 1  # KDA_ERR_INVALID_ARG
    assert lib.kda_get_last_device_error() == 0  # cleared


# --- decode ---------------------------------------------------------------------------------

def run_decode(lib, d, o_dtype=torch.bfloat16, scale=1.0):
    g, beta = lib.gate(d.f.to(DEV), d.b.to(DEV), d.A_log.to(DEV), d.dt_bias.to(DEV), d.alog_mode)
    state = d.state.to(DEV)
    o = lib.decode(d.q.to(DEV), d.k.to(DEV), d.v.to(DEV), g, beta, state, scale, o_dtype=o_dtype)
    return o, state


def oracle_decode(d, sel=None, scale=1.0):
    g_ref, b_ref = oracle.gate(d.f.float().numpy(), d.b.numpy(), d.A_log.numpy(),
                               d.dt_bias.numpy(), d.alog_mode)
    q, k, v, S = f64(d.q), f64(d.k), f64(d.v), f64(d.state) if sel is None else None
    if sel is not None:
        bs, hs = sel
        q, k, v = q[bs][:, hs], k[bs][:, hs], v[bs][:, hs]
        g_ref, b_ref = g_ref[bs][:, hs], b_ref[bs][:, hs]
        S = d.state[bs][:, hs].double().numpy()
    return oracle.decode(q, k, v, g_ref, b_ref, S, scale=scale)


@pytest.mark.parametrize("o_dtype", [torch.bfloat16, torch.float32])
def test_decode_small(lib, o_dtype):
    d = synth.make_decode_inputs(6, H=5, seed=11)
    o, state = run_decode(lib, d, o_dtype, scale=0.75)
    o_ref, S_ref = oracle_decode(d, scale=0.75)
    assert rel_l2(f64(o), o_ref) <= O_TOL
    assert rel_l2(f64(state), S_ref) <= STATE_TOL


def test_decode_full_size_sampled(lib):
    """256 sequences x 96 heads (1.6 GB of state) in the launch configuration the
    benchmark times; the oracle checks a seeded sample of 16 sequences x 6 heads."""
    d = synth.make_decode_inputs(256, H=96, seed=0)
    o, state = run_decode(lib, d)
    r = np.random.default_rng(0)
    bs = np.sort(r.choice(256, 16, replace=False))
    hs = np.sort(r.choice(96, 6, replace=False))
    o_ref, S_ref = oracle_decode(d, sel=(bs, hs))
    o_g = f64(o)[bs][:, hs]
    S_g = state[torch.from_numpy(bs).to(DEV)][:, torch.from_numpy(hs).to(DEV)].cpu().double().numpy()
    assert rel_l2(o_g, o_ref) <= O_TOL
    assert rel_l2(S_g, S_ref) <= STATE_TOL


def test_prefill_then_decode_continuation(lib):
    """Prefill T1 tokens, then decode the next tokens one by one from its final
    state; compare with one long oracle run (the continuation structure)."""
    T1, T2, H = 100, 12, 2
    x = synth.make_inputs(T1 + T2, H=H, D=128, seed=21, s0_std=0.05)
    g_ref, beta_ref = oracle_gate(x)
    o_ref, S_ref = oracle_prefill(x, g_ref, beta_ref)
    g, beta = gpu_gate(lib, x)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    o1, S = lib.prefill(q[:T1].contiguous(), k[:T1].contiguous(), v[:T1].contiguous(),
                        g[:T1].contiguous(), beta[:T1].contiguous(), None, 1.0,
                        x.initial_state.to(DEV), o_dtype=torch.float32)
    outs = [o1]
    for t in range(T1, T1 + T2):
        # clone(): fresh 16-byte-aligned buffers (a one-token slice of beta is not)
        ot = lib.decode(q[t:t + 1].clone(), k[t:t + 1].clone(), v[t:t + 1].clone(),
                        g[t:t + 1].clone(), beta[t:t + 1].clone(), S, 1.0,
                        o_dtype=torch.float32)
        outs.append(ot)
    o = torch.cat(outs)
    assert rel_l2(f64(o), o_ref) <= O_TOL
    assert rel_l2(f64(S), S_ref) <= STATE_TOL


def test_prefill_many_short_sequences(lib):
    """200 sequences of 1..40 tokens x 2 heads: more chains than SMs, every
    chunk a partial one."""
    lens = synth.varlen_lengths(200, 1, 40, seed=5)
    x = synth.make_inputs(lengths=lens, H=2, D=128, seed=23, s0_std=0.05)
    check_prefill(lib, x, o_dtype=torch.float32)


# --- strong decay: chunks whose decay exceeds what one chunk represents ----------------------

def _strong_decay_g(x, g_ref, case):
    """g for the strong-decay cases: every channel at -5 per token (-320 over a
    64-token chunk), or one head with a mix of hard channels (-5 per token;
    -300 every seventh token in a few) and the soft K3 channels."""
    g = np.array(g_ref, dtype=np.float32, copy=True)
    if case == "all_hard":
        g[:] = -5.0
    else:
        g[:, 0, :32] = -5.0
        g[::7, 0, 32:40] = -300.0
    return g


@pytest.mark.parametrize("case", ["all_hard", "mixed"])
@pytest.mark.parametrize("o_dtype", [torch.bfloat16, torch.float32])
def test_prefill_strong_decay_matches_oracle(lib, case, o_dtype):
    """Per-channel chunk decays far beyond one chunk's range (and single tokens
    beyond e^-160) are computed, not refused: the kernel shortens such chunks.
    Parity with the fp64 recurrence on the same g."""
    x = synth.make_inputs(lengths=[200, 77, 1], H=2, D=128, seed=8, s0_std=0.05)
    g_ref, beta_ref = oracle_gate(x)
    g_np = _strong_decay_g(x, g_ref, case)
    g, beta = torch.from_numpy(g_np).to(DEV), torch.from_numpy(beta_ref).to(DEV)
    o, Sf = lib.prefill(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta, x.cu_seqlens.to(DEV), 1.0,
                        x.initial_state.to(DEV), o_dtype=o_dtype)
    assert lib.kda_get_last_device_error() == 0
    o_ref, S_ref = oracle_prefill(x, g_np, beta_ref)
    assert np.isfinite(f64(o)).all() and np.isfinite(f64(Sf)).all()
    assert_parity(f64(o), o_ref, f64(Sf), S_ref, x.cu_seqlens)


@pytest.mark.parametrize("hard", ["all", "some_channels"])
def test_prefill_gated_strong_decay_matches_oracle(lib, hard):
    """The gate fused into the kernel with A_log = 2 and f = 30 (g about -190
    per token: each token a chunk of its own), in every channel or in the first
    32 channels of each head beside the soft K3 ones."""
    x = synth.make_inputs(lengths=[130, 64, 9], H=2, D=128, seed=12, s0_std=0.05)
    f = x.f.float()
    A_log = x.A_log.clone()
    sl = slice(None) if hard == "all" else slice(0, 32)
    f[..., sl] = 30.0
    A_log[sl] = 2.0
    x.f = f.to(torch.bfloat16)
    x.A_log = A_log
    o, Sf = lib.prefill_gated(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), x.f.to(DEV), x.b.to(DEV),
                              x.A_log.to(DEV), x.dt_bias.to(DEV), x.alog_mode,
                              x.cu_seqlens.to(DEV), 1.0, x.initial_state.to(DEV),
                              o_dtype=torch.float32)
    assert lib.kda_get_last_device_error() == 0
    g_ref, beta_ref = oracle_gate(x)
    assert g_ref[..., sl].max() < -100.0
    o_ref, S_ref = oracle_prefill(x, g_ref, beta_ref)
    assert np.isfinite(f64(o)).all() and np.isfinite(f64(Sf)).all()
    assert_parity(f64(o), o_ref, f64(Sf), S_ref, x.cu_seqlens)


def test_prefill_positive_g_is_reported(lib):
    """g must be a log-decay (g <= 0): a positive entry sets INVALID_ARG in the
    device error word."""
    x = synth.make_inputs(96, H=2, D=128, seed=13)
    g, beta = gpu_gate(lib, x)
    g[40, 1, 7] = 0.25
    lib.prefill(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), g, beta)
    assert lib.kda_get_last_device_error() == 1   # KDA_ERR_INVALID_ARG
    assert lib.kda_get_last_device_error() == 0

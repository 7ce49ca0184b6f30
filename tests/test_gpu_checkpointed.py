"""GPU tests of the training pair kda_chunk_prefill_checkpointed /
kda_chunk_backward_checkpointed (the chunked regime for training,
code-audit.json finding "dual-kda-execution-regimes"): the forward pass keeps
the state at every 64-token chunk start, and the backward reads those states
instead of running the forward again.

- The checkpointed prefill writes the same o and final state as
  kda_chunk_prefill, bit for bit.
- Each stored chunk-start state equals the oracle's fp64 recurrence run over
  the tokens before it, within the prefill's state bound (1e-3 relative L2).
- The checkpointed backward writes the same gradients as the self-contained
  kda_chunk_backward, bit for bit, and so stays within that test's bound of
  the oracle's reverse mode (checked here too on two varlen cases: bf16 dO
  with empty sequences, and fp32 dO with a query scale and ragged tails).
- A (sequence, head) whose chunk had to be shortened is marked in the flags
  and the backward reports KDA_ERR_DECAY_RANGE with zero gradients for it."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_33_gb300 import synth
from parity_utils import DEV, STATE_TOL, f64, gpu_gate, oracle_gate, rel_l2

pytestmark = pytest.mark.gpu
GRAD_TOL = 1e-3
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def make_case(lens=None, N=None, H=3, seed=0):
    x = synth.make_inputs(N, H=H, seed=seed, lengths=lens, s0_std=0.05)
    gen = torch.Generator().manual_seed(seed + 1000)
    dO = torch.randn(x.N, H, 128, generator=gen).to(torch.bfloat16)
    dSf = torch.randn(x.B, H, 128, 128, generator=gen) * 0.1
    return x, dO, dSf


def device_args(x):
    cu = None if x.cu_seqlens is None else x.cu_seqlens.to(DEV)
    return x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), cu, x.initial_state.to(DEV)


def unpack(ckpt, B, H):
    """(split flags [B, H], states [slots, H, 128, 128]) of a checkpoint buffer."""
    flags = ckpt[:B * H * 4].view(torch.int32).view(B, H)
    head = ((B * H * 4 + 255) // 256) * 256
    states = ckpt[head:].view(torch.float32).view(-1, H, 128, 128)
    return flags, states


@pytest.mark.parametrize("lens,H,o_dtype", [
    (None, 2, torch.bfloat16),
    ([0, 1, 17, 130, 64, 33, 0, 5], 2, torch.float32),
    ([200, 64, 129], 3, torch.bfloat16),
])
def test_prefill_checkpointed_matches_prefill_and_the_oracle_states(lib, lens, H, o_dtype):
    x, _, _ = make_case(lens=lens, N=None if lens else 190, H=H, seed=11)
    q, k, v, cu, S0 = device_args(x)
    g, beta = gpu_gate(lib, x)
    o, Sf, ckpt = lib.prefill_checkpointed(q, k, v, g, beta, cu_seqlens=cu, scale=0.7,
                                           initial_state=S0, o_dtype=o_dtype)
    o_ref, Sf_ref = lib.prefill(q, k, v, g, beta, cu_seqlens=cu, scale=0.7, initial_state=S0,
                                o_dtype=o_dtype)
    assert lib.kda_get_last_device_error() == 0
    assert torch.equal(o, o_ref)
    assert torch.equal(Sf, Sf_ref)
    assert ckpt.numel() == lib.kda_chunk_checkpoints_size(x.N, x.B, H)
    flags, states = unpack(ckpt, x.B, H)
    assert int(flags.abs().sum()) == 0
    # every chunk start of every sequence against the fp64 recurrence over the
    # tokens before it (chunk c of sequence b sits in slot cu[b] / 64 + b + c)
    g_ref, b_ref = oracle_gate(x)
    cu_np = [0, x.N] if x.cu_seqlens is None else [int(c) for c in x.cu_seqlens]
    qf, kf, vf = f64(x.q), f64(x.k), f64(x.v)
    gf, bf = np.asarray(g_ref, np.float64), np.asarray(b_ref, np.float64)
    for b in range(x.B):
        t0, t1 = cu_np[b], cu_np[b + 1]
        S = f64(x.initial_state)[b:b + 1]
        for c, tc in enumerate(range(t0, t1, 64)):
            got = f64(states[t0 // 64 + b + c])
            err = rel_l2(got, S[0]) if np.linalg.norm(S) > 0 else float(np.abs(got).max())
            assert err <= STATE_TOL, f"sequence {b} chunk {c}: rel L2 {err:.3e}"
            te = min(tc + 64, t1)
            _, S = oracle.recurrent(qf[tc:te], kf[tc:te], vf[tc:te], gf[tc:te], bf[tc:te],
                                    scale=0.7, initial_state=S, nthreads=4)


@pytest.mark.parametrize("lens,do_dtype,scale", [
    ([0, 1, 17, 130, 64, 33, 0, 5], torch.bfloat16, 128 ** -0.5),
    ([300, 1, 64, 127], torch.float32, 0.8),
])
def test_backward_checkpointed_matches_backward_and_the_oracle(lib, lens, do_dtype, scale):
    x, dO, dSf = make_case(lens=lens, H=2, seed=3)
    dO = dO.to(do_dtype)
    q, k, v, cu, S0 = device_args(x)
    g, beta = gpu_gate(lib, x)
    _, _, ckpt = lib.prefill_checkpointed(q, k, v, g, beta, cu_seqlens=cu, scale=scale,
                                          initial_state=S0)
    a = lib.backward_from_checkpoints(q, k, v, g, beta, dO.to(DEV), ckpt, cu_seqlens=cu,
                                      scale=scale, dS_final=dSf.to(DEV))
    ref = lib.backward_chunked(q, k, v, g, beta, dO.to(DEV), cu_seqlens=cu, scale=scale,
                               initial_state=S0, dS_final=dSf.to(DEV))
    assert lib.kda_get_last_device_error() == 0
    for name, ga, gr in zip(NAMES, a, ref):
        assert torch.equal(ga, gr), name
    g_ref, b_ref = oracle_gate(x)
    exact = oracle.recurrent_backward(f64(x.q), f64(x.k), f64(x.v), np.asarray(g_ref, np.float64),
                                      np.asarray(b_ref, np.float64), f64(dO),
                                      cu_seqlens=x.cu_seqlens.numpy(), scale=scale,
                                      initial_state=f64(x.initial_state), dS_final=f64(dSf),
                                      nthreads=8)
    for name, ga, r in zip(NAMES, a, exact):
        err = rel_l2(f64(ga), r)
        assert err <= GRAD_TOL, f"{name}: rel L2 {err:.3e}"


def test_checkpoints_serve_several_backward_calls_at_t4096(lib):
    """T = 4096, H = 96: the checkpoints are only read, so two backward calls
    on them (with different dO) each equal the self-contained backward."""
    x, dO, dSf = make_case(N=4096, H=96, seed=5)
    q, k, v, cu, S0 = device_args(x)
    g, beta = gpu_gate(lib, x)
    _, _, ckpt = lib.prefill_checkpointed(q, k, v, g, beta, initial_state=S0)
    for dO_i in (dO.to(DEV), (dO.float() * -0.5).to(DEV)):
        a = lib.backward_from_checkpoints(q, k, v, g, beta, dO_i, ckpt, dS_final=dSf.to(DEV))
        ref = lib.backward_chunked(q, k, v, g, beta, dO_i, initial_state=S0,
                                   dS_final=dSf.to(DEV))
        assert lib.kda_get_last_device_error() == 0
        for name, ga, gr in zip(NAMES, a, ref):
            assert torch.equal(ga, gr), name
        del a, ref


def test_shortened_chunk_is_flagged_and_reported(lib):
    """Head 1 decays by 5 per token (320 per 64-token chunk, above the 160 one
    chunk represents): its chunks are shortened, the flag is set, and the
    backward reports KDA_ERR_DECAY_RANGE with zero gradients for it while
    head 0 equals the self-contained backward."""
    x, dO, dSf = make_case(N=130, H=2, seed=7)
    q, k, v, cu, S0 = device_args(x)
    g, beta = gpu_gate(lib, x)
    g[:, 1] = -5.0
    _, _, ckpt = lib.prefill_checkpointed(q, k, v, g, beta, initial_state=S0)
    assert lib.kda_get_last_device_error() == 0
    flags, _ = unpack(ckpt, 1, 2)
    assert flags.tolist() == [[0, 1]]
    a = lib.backward_from_checkpoints(q, k, v, g, beta, dO.to(DEV), ckpt, dS_final=dSf.to(DEV))
    assert lib.kda_get_last_device_error() == 11   # KDA_ERR_DECAY_RANGE
    ref = lib.backward_chunked(q, k, v, g, beta, dO.to(DEV), initial_state=S0,
                               dS_final=dSf.to(DEV))
    assert lib.kda_get_last_device_error() == 11
    for name, ga, gr in zip(NAMES, a, ref):
        assert float(ga[:, 1].abs().max()) == 0.0, name
        assert torch.equal(ga[:, 0], gr[:, 0]), name


def test_all_sequences_empty(lib):
    """A batch whose sequences are all empty (N = 0): the prefills pass the
    initial states through, and the backward passes dS_final through to dS0."""
    x, dO, dSf = make_case(lens=[0, 0], H=2, seed=13)
    q, k, v, cu, S0 = device_args(x)
    g, beta = gpu_gate(lib, x)
    o, Sf = lib.prefill(q, k, v, g, beta, cu_seqlens=cu, initial_state=S0)
    o2, Sf2, ckpt = lib.prefill_checkpointed(q, k, v, g, beta, cu_seqlens=cu, initial_state=S0)
    og, Sfg = lib.prefill_gated(q, k, v, x.f.to(DEV), x.b.to(DEV), x.A_log.to(DEV),
                                x.dt_bias.to(DEV), x.alog_mode, cu, 1.0, S0)
    assert lib.kda_get_last_device_error() == 0
    assert o.numel() == o2.numel() == og.numel() == 0
    for S in (Sf, Sf2, Sfg):
        assert torch.equal(S, S0)
    a = lib.backward_from_checkpoints(q, k, v, g, beta, dO.to(DEV), ckpt, cu_seqlens=cu,
                                      dS_final=dSf.to(DEV))
    b = lib.backward_chunked(q, k, v, g, beta, dO.to(DEV), cu_seqlens=cu, initial_state=S0,
                             dS_final=dSf.to(DEV))
    assert lib.kda_get_last_device_error() == 0
    for grads in (a, b):
        assert all(t.numel() == 0 for t in grads[:5])
        assert torch.equal(grads[5], dSf.to(DEV))

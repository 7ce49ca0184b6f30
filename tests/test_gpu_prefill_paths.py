"""The two algorithms behind kda_chunk_prefill and kda_chunk_prefill_gated.

Given kda_chunk_prefill_workspace_size() bytes of workspace the entry points
run the two-phase path (chunk-parallel intra-chunk kernel + per-head state
pass); given only KDA_PREFILL_MIN_WORKSPACE (256) bytes they run the one-kernel
path.  Both must meet the parity tolerances against the fp64 oracle, and they
perform the same roundings in the same order, so they must agree with each
other to 1e-6 relative L2."""
import numpy as np
import pytest
import torch

from gated_delta_rule_33_gb300 import synth
from parity_utils import (DEV, O_TOL, STATE_TOL, f64, gpu_gate, oracle_gate, oracle_prefill,
                          rel_l2)

pytestmark = pytest.mark.gpu
PATH_TOL = 1e-6
MIN_WS = 256


def run_paths(lib, x, scale, o_dtype, gated):
    N, H = x.N, x.H
    B = x.B
    cu = None if x.cu_seqlens is None else x.cu_seqlens.to(DEV)
    S0 = None if x.initial_state is None else x.initial_state.to(DEV)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    big = lib.kda_chunk_prefill_workspace_size(N, B, H)
    outs = []
    g, beta = gpu_gate(lib, x)
    for ws_bytes in (big, MIN_WS):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
        o = torch.full((N, H, 128), float("nan"), dtype=o_dtype, device=DEV)
        Sf = torch.full((B, H, 128, 128), float("nan"), device=DEV)
        if gated:
            lib.kda_chunk_prefill_gated(q, k, v, x.f.to(DEV), x.b.to(DEV), x.A_log.to(DEV),
                                        x.alog_mode, x.dt_bias.to(DEV), cu, scale, S0, Sf, o, ws)
        else:
            lib.kda_chunk_prefill(q, k, v, g, beta, cu, scale, S0, Sf, o, ws)
        assert lib.kda_get_last_device_error() == 0
        outs.append((f64(o), f64(Sf)))
    g_ref, beta_ref = oracle_gate(x)
    o_ref, S_ref = oracle_prefill(x, g_ref, beta_ref, scale=scale)
    for o, S in outs:
        assert np.isfinite(o).all() and np.isfinite(S).all()
        assert rel_l2(o, o_ref) <= O_TOL
        assert rel_l2(S, S_ref) <= STATE_TOL
    (o1, S1), (o2, S2) = outs
    assert rel_l2(o1, o2) <= PATH_TOL, rel_l2(o1, o2)
    assert rel_l2(S1, S2) <= PATH_TOL, rel_l2(S1, S2)


@pytest.mark.parametrize("gated", [False, True])
def test_varlen_edges_both_paths(lib, gated):
    x = synth.make_inputs(lengths=[0, 1, 63, 64, 65, 300, 0, 129], H=4, D=128, seed=21,
                          s0_std=0.05)
    run_paths(lib, x, 0.9, torch.float32, gated)


@pytest.mark.parametrize("gated", [False, True])
def test_single_sequence_both_paths(lib, gated):
    x = synth.make_inputs(1000, H=3, D=128, seed=22)
    run_paths(lib, x, 1.0, torch.bfloat16, gated)


def test_many_short_sequences_both_paths(lib):
    """More chains than SMs, many record slots left empty."""
    lens = synth.varlen_lengths(200, 1, 40, seed=5)
    x = synth.make_inputs(lengths=lens, H=2, D=128, seed=23, s0_std=0.05)
    run_paths(lib, x, 1.0, torch.float32, False)

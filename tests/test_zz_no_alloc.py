"""The prefill entry point that allocates nothing (kda_chunk_prefill_noalloc).

Some callers cannot allocate device memory for a workspace: a plugin
interface that passes the library only its inputs and outputs, or a server
that reserved all device memory at start-up.  For them the library offers a
variant of kda_chunk_prefill that takes its scratch from a device array built
into the library.  This test calls it through the C ABI twice in a row (the
array keeps the previous call's contents, so the second call checks that the
scratch is cleared where it must be) and compares each result with the
workspace entry point's, within the parity tolerances used everywhere else.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_33_gb300 import synth
from parity_utils import DEV, O_TOL, STATE_TOL, f64, gpu_gate, rel_l2

pytestmark = pytest.mark.gpu


def test_noalloc_prefill_matches_workspace_entry_point(lib):
    x = synth.make_inputs(lengths=[300, 77, 0, 129], H=8, D=128, seed=31, s0_std=0.05)
    g, beta = gpu_gate(lib, x)
    q, k, v = x.q.to(DEV), x.k.to(DEV), x.v.to(DEV)
    cu = x.cu_seqlens.to(DEV)
    S0 = x.initial_state.to(DEV)
    o_ref, S_ref = lib.prefill(q, k, v, g, beta, cu, 0.75, S0, o_dtype=torch.float32)
    assert lib.kda_get_last_device_error() == 0
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        Sf = torch.full_like(S_ref, float("nan"))
        lib.kda_chunk_prefill_noalloc(q, k, v, g, beta, cu, 0.75, S0, Sf, o)
        assert lib.kda_get_last_device_error() == 0
        assert np.isfinite(f64(o)).all() and np.isfinite(f64(Sf)).all()
        assert rel_l2(f64(o), f64(o_ref)) <= O_TOL
        assert rel_l2(f64(Sf), f64(S_ref)) <= STATE_TOL

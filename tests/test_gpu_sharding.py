"""The placement of gated_delta_rule_33_gb300/sharding.py on the real kernels:
a batch split by heads, or a packed batch split by sequences, and run shard by
shard (as separate ranks would) gives exactly the full run's outputs and final
states.  Every (sequence, head) chain is computed on its own, so the split
must not change a single bit."""
import pytest
import torch

from gated_delta_rule_33_gb300 import synth
from gated_delta_rule_33_gb300.sharding import head_shard, sequence_shard
from parity_utils import DEV

pytestmark = pytest.mark.gpu


def _run(lib, x, cu=None, heads=None, tokens=None, seqs=None):
    h = slice(None) if heads is None else slice(*heads)
    t = slice(None) if tokens is None else slice(*tokens)
    s = slice(None) if seqs is None else slice(*seqs)

    def dev(a):
        return a.contiguous().to(DEV)

    S0 = None if x.initial_state is None else dev(x.initial_state[s, h])
    return lib.prefill_gated(dev(x.q[t, h]), dev(x.k[t, h]), dev(x.v[t, h]), dev(x.f[t, h]),
                             dev(x.b[t, h]), x.A_log.to(DEV), dev(x.dt_bias[h]), x.alog_mode,
                             cu_seqlens=None if cu is None else cu.to(DEV), initial_state=S0)


@pytest.mark.parametrize("world", [2, 3])
def test_head_shards_reproduce_the_full_prefill(lib, world):
    lengths = [120, 0, 180, 64]
    x = synth.make_inputs(sum(lengths), H=7, D=128, seed=11, lengths=lengths, s0_std=0.05)
    full_o, full_S = _run(lib, x, cu=x.cu_seqlens)
    for rank in range(world):
        h0, h1 = head_shard(7, rank, world)
        o, S = _run(lib, x, cu=x.cu_seqlens, heads=(h0, h1))
        assert torch.equal(o, full_o[:, h0:h1])
        assert torch.equal(S, full_S[:, h0:h1])


@pytest.mark.parametrize("world", [2, 3, 4])
def test_sequence_shards_reproduce_the_full_prefill(lib, world):
    lengths = [100, 0, 64, 250, 17, 130]
    x = synth.make_inputs(sum(lengths), H=3, D=128, seed=12, lengths=lengths, s0_std=0.05)
    cu = x.cu_seqlens.tolist()
    full_o, full_S = _run(lib, x, cu=x.cu_seqlens)
    covered = 0
    for rank in range(world):
        s0, s1 = sequence_shard(cu, rank, world)
        if s1 == s0:
            continue
        t0, t1 = cu[s0], cu[s1]
        sub = torch.tensor([c - t0 for c in cu[s0:s1 + 1]], dtype=torch.int32)
        o, S = _run(lib, x, cu=sub, tokens=(t0, t1), seqs=(s0, s1))
        assert torch.equal(o, full_o[t0:t1])
        assert torch.equal(S, full_S[s0:s1])
        covered += s1 - s0
    assert covered == len(lengths)

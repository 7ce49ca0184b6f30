"""The multi-rank path on CPU: the head and sequence splits of
gated_delta_rule_33_gb300/sharding.py, and two gloo ranks that each run the
fp64 oracle on their own shard and gather, which must give exactly the
single-process result (every (sequence, head) chain is independent, so a
split changes no arithmetic), plus the max over ranks that bench.py times
with.  No GPU: the ranks are CPU processes on 127.0.0.1."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from gated_delta_rule_33_gb300 import synth
from gated_delta_rule_33_gb300.sharding import head_shard, max_over_ranks, sequence_shard


@pytest.mark.parametrize("H", [0, 1, 2, 3, 7, 96])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_head_shard_is_a_balanced_partition(H, world):
    spans = [head_shard(H, r, world) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == H
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    sizes = [h1 - h0 for h0, h1 in spans]
    assert min(sizes) >= 0 and max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_sequence_shard_is_a_token_balanced_partition(world):
    r = np.random.default_rng(world)
    for _ in range(50):
        lens = r.integers(0, 300, size=int(r.integers(1, 12)))
        cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
        B, N = len(lens), cu[-1]
        spans = [sequence_shard(cu, rk, world) for rk in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == B
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        longest = int(lens.max()) if B else 0
        for s0, s1 in spans:
            tokens = cu[s1] - cu[s0]
            assert abs(tokens - N / world) <= longest + 1e-9


def test_splits_reject_bad_arguments():
    with pytest.raises(ValueError):
        head_shard(4, 2, 2)
    with pytest.raises(ValueError):
        sequence_shard([0, 5, 3], 0, 2)
    with pytest.raises(ValueError):
        sequence_shard([1, 5], 0, 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        H, D = 5, 16
        # one packed batch of four sequences, split by heads
        lengths = [40, 0, 75, 17]
        x = synth.make_inputs(sum(lengths), H=H, D=D, seed=3, lengths=lengths)
        g, beta = oracle.gate(x.f.float().numpy(), x.b.numpy(), x.A_log.numpy(),
                              x.dt_bias.numpy(), x.alog_mode)
        h0, h1 = head_shard(H, rank, world)
        sel = slice(h0, h1)
        o, S = oracle.recurrent(x.q[:, sel].double().numpy(), x.k[:, sel].double().numpy(),
                                x.v[:, sel].double().numpy(), g[:, sel], beta[:, sel],
                                cu_seqlens=x.cu_seqlens.numpy(), nthreads=1)
        parts_o = [None] * world
        parts_S = [None] * world
        dist.all_gather_object(parts_o, (h0, h1, o))
        dist.all_gather_object(parts_S, (h0, h1, S))
        # the same batch split by sequences
        cu = x.cu_seqlens.tolist()
        s0, s1 = sequence_shard(cu, rank, world)
        t0, t1 = cu[s0], cu[s1]
        sub_cu = np.array([c - t0 for c in cu[s0:s1 + 1]], dtype=np.int32)
        if s1 > s0:
            so, sS = oracle.recurrent(x.q[t0:t1].double().numpy(), x.k[t0:t1].double().numpy(),
                                      x.v[t0:t1].double().numpy(), g[t0:t1], beta[t0:t1],
                                      cu_seqlens=sub_cu, nthreads=1)
        else:
            so, sS = np.zeros((0, H, D)), np.zeros((0, H, D, D))
        seq_parts = [None] * world
        dist.all_gather_object(seq_parts, (s0, s1, t0, t1, so, sS))
        slowest = max_over_ranks(10.0 + rank, world)
        if rank == 0:
            np.savez(os.path.join(out_dir, "gathered.npz"),
                     o=np.concatenate([p[2] for p in sorted(parts_o, key=lambda p: p[0])], axis=1),
                     S=np.concatenate([p[2] for p in sorted(parts_S, key=lambda p: p[0])], axis=1),
                     so=np.concatenate([p[4] for p in seq_parts], axis=0),
                     sS=np.concatenate([p[5] for p in seq_parts], axis=0),
                     spans=np.array([[p[0], p[1], p[2], p[3]] for p in seq_parts]),
                     slowest=np.array([slowest]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_reproduce_the_single_process_result(tmp_path, world):
    oracle.build()
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = np.load(tmp_path / "gathered.npz")
    H, D = 5, 16
    lengths = [40, 0, 75, 17]
    x = synth.make_inputs(sum(lengths), H=H, D=D, seed=3, lengths=lengths)
    g, beta = oracle.gate(x.f.float().numpy(), x.b.numpy(), x.A_log.numpy(), x.dt_bias.numpy(),
                          x.alog_mode)
    o, S = oracle.recurrent(x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy(), g,
                            beta, cu_seqlens=x.cu_seqlens.numpy(), nthreads=1)
    # head split: each chain computed by exactly one rank, bit for bit
    np.testing.assert_array_equal(got["o"], o)
    np.testing.assert_array_equal(got["S"], S)
    # sequence split: outputs in token order, final states in sequence order
    np.testing.assert_array_equal(got["so"], o)
    np.testing.assert_array_equal(got["sS"], S)
    spans = got["spans"]
    assert spans[0][0] == 0 and spans[-1][1] == len(lengths)
    assert float(got["slowest"][0]) == 10.0 + world - 1

"""Placement of independent KDA work across ranks (one process per GPU).

Every (sequence, head) chain of the recurrence is independent of every other:
the state of one head of one sequence never meets another's (the recurrence
S_t = (I - beta k k^T) Diag(e^g) S_{t-1} + beta k v^T runs per head, and a
sequence starts from its own initial state).  A batch therefore splits across
ranks with no data-path exchange, either by whole sequences (weak scaling:
each rank owns its own sequences) or by heads of the same sequences.  Only
the timing and the checks use a collective (a max, or a gather in tests).

Host logic only: nothing here launches a kernel.
"""
from __future__ import annotations

import os
from typing import Sequence, Tuple


def dist_setup() -> Tuple[int, int, int]:
    """(rank, world, local_rank) from the torchrun environment; initialises the
    process group (NCCL with a GPU, gloo without) when WORLD_SIZE > 1."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (the job's time is the slowest rank's)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def head_shard(H: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous heads [h0, h1) of this rank; shard sizes differ by at most one
    and every head belongs to exactly one rank."""
    if H < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad split: H={H} rank={rank} world={world}")
    base, extra = divmod(H, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def sequence_shard(cu_seqlens: Sequence[int], rank: int, world: int) -> Tuple[int, int]:
    """Contiguous sequences [s0, s1) of this rank for a packed batch given by
    its cu_seqlens (B + 1 offsets): rank r takes the sequences whose first
    token lies in [r N / world, (r + 1) N / world), so shards hold about N /
    world tokens each (off by less than one sequence's length) and every
    sequence, empty ones included, belongs to exactly one rank."""
    cu = [int(c) for c in cu_seqlens]
    B = len(cu) - 1
    if B < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad split: B={B} rank={rank} world={world}")
    if cu and (cu[0] != 0 or any(a > b for a, b in zip(cu, cu[1:]))):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    N = cu[-1] if cu else 0

    def first_owned(r: int) -> int:
        # the first sequence whose start is at or past r * N / world (integer form)
        if r >= world:
            return B
        s = 0
        while s < B and cu[s] * world < r * N:
            s += 1
        return s

    return first_owned(rank), first_owned(rank + 1)

"""Host-side partitioning of decode work across GPUs (one process per GPU).

Sequences, layers and rows of the quantized cache are independent, so N GPUs run N
disjoint shards with no collective on the data path; the only communication is the
timing reduction of a benchmark.  A ragged batch is split by longest-processing-time
greedy assignment on the per-sequence row counts, which keeps the busiest rank within
max(L_i) rows of the mean.
"""
from __future__ import annotations

from typing import Sequence


def shard_sequences(seq_len: Sequence[int], world: int, rank: int) -> list[int]:
    """Indices of the sequences rank `rank` of `world` owns (sorted)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    order = sorted(range(len(seq_len)), key=lambda i: (-int(seq_len[i]), i))
    load = [0] * world
    owner = [0] * len(seq_len)
    for i in order:
        r = min(range(world), key=lambda k: (load[k], k))
        owner[i] = r
        load[r] += int(seq_len[i])
    return [i for i in range(len(seq_len)) if owner[i] == rank]


def shard_range(n: int, world: int, rank: int) -> range:
    """Contiguous block of n units (layers, rows) for `rank`."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    lo = n * rank // world
    hi = n * (rank + 1) // world
    return range(lo, hi)


def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())

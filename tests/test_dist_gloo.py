"""The N>1 host path on CPU: world_size-2 gloo ranks shard a ragged batch and the
benchmark's time reduction, with no GPU."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from quantized_kv_cache_fp8_gb300.sharding import max_over_ranks, shard_range, shard_sequences


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, seq_len, out_q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = shard_sequences(seq_len, world, rank)
    layers = list(shard_range(32, world, rank))
    # each rank "times" its shard by its row count; the job time is the slowest rank's
    t = float(sum(seq_len[i] for i in mine))
    tmax = max_over_ranks(t)
    out_q.put((rank, mine, layers, t, tmax))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_sharding_and_timing():
    # the ragged workload's length draw: 32 lengths uniform in [1024, 65536]
    seq_len = [int(x) for x in np.random.default_rng(0).integers(1024, 65537, 32)]
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, seq_len, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    owned = sorted(i for r in res for i in r[1])
    assert owned == list(range(32))                      # every sequence exactly once
    layers = sorted(l for r in res for l in r[2])
    assert layers == list(range(32))
    loads = [r[3] for r in res]
    assert max(loads) - min(loads) <= max(seq_len)       # LPT balance bound
    assert all(r[4] == max(loads) for r in res)          # max over ranks seen by all


def test_shard_edge_cases():
    assert shard_sequences([], 2, 0) == []
    assert shard_sequences([5], 3, 2) == []
    assert shard_sequences([5], 3, 0) == [0]
    assert list(shard_range(3, 4, 3)) == [2]
    with pytest.raises(ValueError):
        shard_range(3, 0, 0)
    assert max_over_ranks(1.5) == 1.5

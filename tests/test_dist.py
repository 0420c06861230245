"""Multi-rank host logic on CPU (gloo, world size 2): request sharding,
per-rank seeds and the max-time / summed-work reduction the benchmark uses."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_decode_bind_gb300 import dist as D


def test_shard_range_partitions():
    for n in (0, 1, 5, 16, 17):
        for world in (1, 2, 3, 8):
            parts = [D.shard_range(n, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            for (a, b), (c, d) in zip(parts, parts[1:]):
                assert b == c
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        D.shard_range(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t, w = D.reduce_time_and_work(0.5 + rank, 10.0 * (rank + 1))
        lo, hi = D.shard_range(16, rank, world)
        q.put((rank, t, w, lo, hi, D.rank_seed(7, rank)))
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for rank, t, w, lo, hi, seed in res:
        assert t == 1.5 and w == 30.0
    assert [(r[3], r[4]) for r in res] == [(0, 8), (8, 16)]
    assert res[0][5] != res[1][5]


def test_single_process_identity():
    assert D.reduce_time_and_work(2.0, 3.0) == (2.0, 3.0)

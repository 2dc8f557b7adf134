"""Multi-rank plumbing of bench.py on CPU: two gloo ranks, no GPU.

The path shards with no exchange (independent sequences / heads), so ranks
meet only in the barrier and the max / sum over ranks of the timing.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

from kda_delta_rule_gb300 import dist as D


def test_shard_partitions_exactly():
    for n in (0, 1, 7, 32, 1000):
        for world in (1, 2, 3, 8):
            parts = [D.shard(n, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
            sizes = [e - b for b, e in parts]
            assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, _ = D.init(backend="gloo")
    D.barrier()
    mx = D.max_over_ranks(10.0 + r)
    sm = D.sum_over_ranks(1.0)
    b, e = D.shard(32, r, w)
    q.put((r, mx, sm, b, e))
    D.finalize()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [x[1] for x in res] == [11.0, 11.0]
    assert [x[2] for x in res] == [2.0, 2.0]
    assert [(x[3], x[4]) for x in res] == [(0, 16), (16, 32)]

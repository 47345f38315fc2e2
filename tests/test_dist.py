"""The benchmark's multi-process logic without a GPU: world_size 2 over gloo on
127.0.0.1.  Each rank is a replica; the timing that counts is the maximum over
ranks, taken with an all-reduce after a barrier."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup("gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + rank, w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, got))


@pytest.mark.timeout(120)
def test_max_over_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=90) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert res == {0: 11.0, 1: 11.0}


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5

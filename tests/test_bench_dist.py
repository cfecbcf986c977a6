"""Multi-rank bench aggregation on CPU (gloo, world size 2): the job's value
is every rank's units over the slowest rank's time."""
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
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 20.0][rank]
    local_units = [7936 * 5, 7936 * 5 + 32][rank]
    q.put((rank, bench.reduce_over_ranks(local_ms, local_units, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_is_max_time_and_total_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        ms, units = res[r]
        assert ms == 20.0
        assert units == 2 * 7936 * 5 + 32


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.0, 17, 1) == (3.0, 17)

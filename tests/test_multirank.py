"""bench.py's multi-process path on CPU: ranks are independent replicas; the job's time is the slowest
rank's and its throughput counts every rank's units (gloo, world size 2)."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [0.25, 0.75][rank]
    units = [1000.0, 3000.0][rank]
    t, u = bench.combine_ranks(elapsed, units, dist)
    bench.barrier(dist)
    out[rank] = (t, u)
    dist.destroy_process_group()


def test_combine_ranks_takes_max_time_and_total_units():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        assert res[r] == (0.75, 4000.0)


def test_single_process_is_identity():
    import bench
    assert bench.combine_ranks(1.5, 10.0, None) == (1.5, 10.0)

"""The bench's multi-process path (replicas only: no data exchange) on CPU:
world size 2 over gloo, the barrier and the max-over-ranks time."""

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
    bench.barrier(world)
    t = bench.max_over_ranks(10.0 + rank * 5.0, world)
    out[rank] = t
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_process_needs_no_group():
    import bench
    bench.barrier(1)
    assert bench.max_over_ranks(3.5, 1) == 3.5

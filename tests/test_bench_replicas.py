"""Host-side logic of the multi-replica benchmark on CPU (gloo, world size 2):
the job time is the slowest rank's, and the throughput counts every rank's units."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 150.0][rank]
    t = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
    dist.barrier()
    q.put((rank, t, bench.aggregate_rate(4096, world, 10, t)))
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_rate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for _, t, rate in res:
        assert t == 150.0
        assert rate == pytest.approx(4096 * 2 * 10 / 0.150)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate_rate(100, 1, 4, 2000.0) == pytest.approx(200.0)

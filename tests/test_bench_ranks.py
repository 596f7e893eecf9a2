"""The multi-rank arithmetic of bench.py, run as two gloo ranks on the CPU:
each rank's time becomes the slowest rank's, and the whole-job value counts
the units of every rank (replicas, weak scaling)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        cpu = torch.device("cpu")
        ms = bench.rank_max(10.0 + 5.0 * rank, cpu, world)  # rank 1 is slower
        dist.barrier()
        q.put((rank, ms, bench.job_value(world, 40, ms)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_every_rank_counts():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in range(world))
    finally:
        for p in procs:
            p.join(60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, value in res:
        assert ms == 15.0
        assert value == pytest.approx(2 * 40 / 15e-3)


def test_one_rank_needs_no_process_group():
    import bench
    assert not dist.is_initialized()
    assert bench.rank_max(12.5, torch.device("cpu"), 1) == 12.5
    assert bench.job_value(1, 40, 12.5) == pytest.approx(40 / 12.5e-3)

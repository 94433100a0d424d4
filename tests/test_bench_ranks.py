"""bench.py's multi-rank arithmetic on CPU with two gloo ranks: every rank gets
the max step time over ranks, and the whole-job value aggregates all replicas."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(0.05 + 0.01 * rank)
    val = bench.whole_job_gbs(285212672, ms, world)
    dist.barrier()
    q.put((rank, ms, val))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, val in res:
        assert ms == pytest.approx(0.06)
        assert val == pytest.approx(2 * 285212672 / 0.06e-3 / 1e9)


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.whole_job_gbs(10**9, 1.0, 1) == pytest.approx(1000.0)

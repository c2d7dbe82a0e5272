"""Multi-process (gloo, world size 2, CPU) checks of the bench's multi-GPU
harness: every rank runs an independent replica, the timed region is the max
over ranks, and the reported value aggregates the units of all ranks."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [12.5, 30.0][rank]
    got = bench.max_over_ranks(elapsed, world, None)
    bench.barrier(world)
    # whole-job throughput: units of all ranks over the slowest rank's time
    units = 1e9
    value = world * units / (got * 1e-3)
    q.put((rank, got, value))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert [r[1] for r in res] == [30.0, 30.0]
    assert res[0][2] == pytest.approx(2 * 1e9 / 0.030)


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)

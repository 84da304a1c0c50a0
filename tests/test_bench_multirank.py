"""The N>1 host logic of bench.py on CPU: two gloo ranks agree on the slowest rank's
time, and the whole-job throughput counts every rank's work (replicas, weak scaling)."""

import os
import socket

import pytest
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
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_max(1.0 + rank * 0.5, "cpu")
        q.put((rank, ms, bench.job_throughput(1e12, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
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
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [1.5, 1.5]
    # 2 ranks x 1 TFLOP in 1.5 ms each
    assert res[0][2] == pytest.approx(2 * 1e12 / 1.5e-3 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.25, "cpu") == 3.25
    assert bench.job_throughput(2e12, 1, 1.0) == pytest.approx(2000.0)

"""The benchmark's multi-rank host logic on CPU with the gloo backend (world size 2).

Each rank runs the same per-GPU workload (heads and sequences are independent,
so there is no data-path collective); the only exchange is the max over ranks
of the timed region, and the job's throughput is all ranks' FLOPs divided by
that slowest time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = bench.slowest_rank_ms(times[rank], world)
        out.put((rank, ms, bench.job_throughput(1e12, world, ms)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_and_weak_scaling_value():
    world = 2
    times = [12.5, 20.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tflops in res:
        assert ms == 20.0
        assert tflops == pytest.approx(2 * 1e12 / 0.020 / 1e12)



def test_single_rank_needs_no_process_group():
    import bench

    assert bench.slowest_rank_ms(7.0, 1) == 7.0
    assert bench.job_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)

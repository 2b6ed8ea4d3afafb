"""The N>1 path of bench.py on the CPU: replicas with a barrier and max-over-ranks timing.

The method has no exchange between GPUs inside one call, so ranks run independent
replicas; the only cross-rank step is the timing reduction, tested here with two gloo
ranks (127.0.0.1) on the CPU.
"""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 10.0 + 5.0 * rank          # rank 1 is the slow one
        dist.barrier()
        worst = bench.max_over_ranks(elapsed, world, torch.device("cpu"))
        q.put((rank, worst, bench.job_throughput(8, 100, worst, world)))
    finally:
        dist.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    # 2 ranks x 8 tokens x 100 steps in 15 ms
    assert abs(res[0][2] - 2 * 8 * 100 / 0.015) < 1e-6


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_throughput(8, 10, 2.0, 1) == 8 * 10 / 0.002

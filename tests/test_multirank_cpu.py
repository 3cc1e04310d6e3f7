"""The N-GPU path of bench.py (independent replicas) on two gloo ranks on the CPU.

Each rank reports its own step time; the job's time is the slowest rank's
and the job's throughput is N times one rank's throughput at that time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [4.0, 5.0][rank]                       # rank 1 is the slow one
        slowest = bench.reduce_max(ms, world, torch.device("cpu"))
        out[rank] = (slowest, bench.whole_job_value(1e3 / slowest, world))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (5.0, 400.0)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1, None) == 3.5
    assert bench.whole_job_value(10.0, 1) == 10.0

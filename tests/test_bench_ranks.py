"""The replicas' path of bench.py (one process per GPU under torchrun), on CPU
with two gloo ranks: the job's time is the slowest rank's, every rank sees
it, the rate counts every rank's steps, and only rank 0 runs the reference
arm.  The GPU work of each rank is not exercised here."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        mine = 10.0 + 5.0 * rank          # rank 1 is the slow replica
        slowest = bench.slowest_rank_ms(mine, dist, "cpu")
        rate = bench.job_rate(1000, world, slowest)
        ref = bench.run_reference(None, rank, world) if rank != 0 else "rank0"
        results[rank] = (slowest, rate, ref)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this multi-threaded process
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1000 / 0.015)
    assert res[1][2] is None  # the reference arm runs on rank 0 only


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(12.5, None, "cpu") == 12.5
    assert bench.job_rate(200, 1, 10.0) == pytest.approx(20000.0)

"""The multi-rank timing of bench.py on CPU: two gloo ranks with different elapsed times.

Each rank of a weak-scaled run links its own workload; the whole job's time is the slowest
rank's, and its throughput is all ranks' units over that time. Runs on CPU (gloo, world size 2,
127.0.0.1 rendezvous), with no GPU and no data-path collective beyond the timing reduction.
"""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [12.5, 20.0][rank]                      # rank 1 is the slow one
        slow = bench.slowest_rank(ms, world, device="cpu")
        out[rank] = (slow, bench.job_throughput(1000.0, world, slow / 1e3))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0] == res[1]                           # every rank reports the same job figures
    slow, value = res[0]
    assert slow == pytest.approx(20.0)
    assert value == pytest.approx(2 * 1000.0 / 0.020)


def test_single_rank_is_identity():
    import bench
    assert bench.slowest_rank(7.0, 1) == 7.0
    assert bench.job_throughput(5.0, 1, 0.5) == pytest.approx(10.0)

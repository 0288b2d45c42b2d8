"""The multi-GPU host logic of bench.py on CPU ranks (gloo, world size 2):
every rank runs its own replica, the reported time is the slowest rank's,
and the value counts all ranks' work.  No data-path collective exists."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        slow = bench.slowest_rank(ms, dist, torch.device("cpu"))
        out[rank] = (r, w, local, slow, bench.whole_job_tflops(w, 2e12, slow))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time_and_all_work():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert sorted(out.keys()) == [0, 1]
    for rank in (0, 1):
        r, w, local, slow, tflops = out[rank]
        assert (r, w, local) == (rank, 2, rank)
        assert slow == pytest.approx(15.0)
        # two replicas of 2 TFLOP each in 15 ms
        assert tflops == pytest.approx(2 * 2e12 / 15e-3 / 1e12)


def test_single_process_needs_no_process_group():
    assert bench.slowest_rank(3.5, None, None) == 3.5
    assert bench.whole_job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)

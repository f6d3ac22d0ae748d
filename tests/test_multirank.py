"""The N > 1 bench path on CPU: two gloo ranks exercise the replica
bookkeeping that bench.py runs over NCCL on GPUs (max over ranks, whole-job
rate, per-rank seeds, the reference arm printing on rank 0 only)."""

import io
import contextlib
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        my_ms = 100.0 + 50.0 * rank
        slowest = bench.max_over_ranks(my_ms, world, torch.device("cpu"))
        rate = bench.job_rate(1e15, 3, world, slowest)
        seed = bench.replica_seed(3, rank)
        seeds = [None] * world
        dist.all_gather_object(seeds, seed)
        buf = io.StringIO()

        class _A:
            workload, steps, warmup, gpus = "tiny", 0, 0, world
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(_A, rank, world)
        out[rank] = (slowest, rate, seeds, buf.getvalue())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        slowest, rate, seeds, printed = res[rank]
        assert slowest == 150.0                       # both ranks see the max
        assert rate == pytest.approx(1e15 * 3 * 2 / 0.150 / 1e12)
        assert len(set(seeds)) == world               # independent replica inputs
    assert res[1][3] == ""                            # the reference arm prints on rank 0 only


def test_single_rank_helpers_are_identity():
    import bench
    assert bench.max_over_ranks(12.5, 1, torch.device("cpu")) == 12.5
    assert bench.job_rate(2e12, 2, 1, 1000.0) == pytest.approx(4.0)
    assert bench.replica_seed(5, 0) == 5

"""The multi-rank logic of bench.py on CPU: two gloo ranks in separate processes.

Under torchrun every rank times its own independent 4096³ problem (output tiles
need no exchange, so there is no collective on the data path); the ranks agree
on the slowest rank's time with one MAX all-reduce, and rank 0 reports the
whole job's throughput. The reference arm runs on rank 0 only.
"""
from __future__ import annotations

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _rank_main(rank, world, store_path, times, out):
    # a file store: no TCP port to pick (a port found free can be taken before the ranks bind it)
    dist.init_process_group("gloo", init_method=f"file://{store_path}", rank=rank, world_size=world)
    try:
        ms_max = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        out[rank] = (ms_max, bench.job_value(bench.FLOPS, world, 100, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    world = 2
    times = [80.0, 95.5]   # rank 1 is the slower one
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, str(tmp_path / "store"), times, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0][0] == out[1][0] == 95.5
    # whole-job value: both ranks' flops over the slowest rank's time
    assert out[0][1] == pytest.approx(bench.FLOPS * 2 * 100 / 95.5e-3 / 1e12)


def test_job_value_single_rank():
    assert bench.job_value(2.0e12, 1, 10, 1000.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        steps, warmup = 1, 0
    bench.run_reference(Args(), rank=1, world=2)   # returns at once, prints nothing
    assert capsys.readouterr().out == ""

"""Multi-rank host logic of the benchmark on CPU: two gloo ranks.

The layer is data parallel with no exchange step: each rank routes and computes its
own batch of tokens against a full replica of the weights, so the only cross-rank
operations are the barrier around the timed region and the maximum of the ranks'
elapsed times, from which the whole-job throughput is formed.  These tests run that
logic with world size 2 on the gloo backend.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, totals, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    got = bench.max_over_ranks(totals[rank], torch.device("cpu"), world)
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    totals = {0: [12.5, 30.0], 1: [14.0, 29.0]}   # rank 1 slower on the device, rank 0 on e2e
    mp.start_processes(_rank_main, args=(2, _free_port(), totals, out), nprocs=2,
                       join=True, start_method="spawn")
    assert out[0] == [14.0, 30.0]
    assert out[1] == [14.0, 30.0]


def test_job_throughput_counts_all_ranks_over_slowest_time():
    sys.path.insert(0, ROOT)
    import bench
    # two ranks x 8192 tokens x 10 steps in 20 ms -> 8.192e6 tokens/s
    assert bench.job_tokens_per_s(2, 8192, 10, 20.0) == pytest.approx(8.192e6)
    # one rank: the per-rank figure
    assert bench.job_tokens_per_s(1, 8192, 10, 20.0) == pytest.approx(4.096e6)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks([3.0, 4.0], torch.device("cpu"), 1) == [3.0, 4.0]


def test_clock_summary_keeps_only_the_timed_window():
    sys.path.insert(0, ROOT)
    import bench
    rows = [
        ["2026/01/01 00:00:00.000", "0", "1000", "2070", "300", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
        ["2026/01/01 00:00:01.000", "0", "2070", "2070", "900", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["2026/01/01 00:00:01.100", "0", "2040", "2070", "950", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["2026/01/01 00:00:03.000", "0", "800", "2070", "200", "0x1", "Active", "Not Active", "Not Active", "Not Active"],
    ]
    t0 = bench._stamp("2026/01/01 00:00:00.900")
    t1 = bench._stamp("2026/01/01 00:00:01.200")
    c = bench.summarize_clocks(rows, t0, t1)
    assert c["samples"] == 2 and c["window"] == "timed region"
    assert c["sm_mhz"] == pytest.approx(2055.0)
    assert c["reasons"] == ["sw_power_cap"]          # the idle sample's hw_slowdown is outside
    assert c["power_w"] == pytest.approx(925.0) and c["power_instant_w"] is None
    # with the instantaneous power column
    rows11 = [r + [p] for r, p in zip(rows, ["310", "1180", "1240", "205"])]
    c = bench.summarize_clocks(rows11, t0, t1)
    assert c["power_instant_w"] == pytest.approx(1210.0) and c["power_instant_max_w"] == 1240.0
    # a window shorter than the sampling interval falls back to the nearest samples
    t0 = bench._stamp("2026/01/01 00:00:02.000")
    c = bench.summarize_clocks(rows, t0, t0 + 0.01)
    assert c["samples"] == 2 and c["window"].startswith("nearest")

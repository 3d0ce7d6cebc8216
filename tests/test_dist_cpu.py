"""Multi-rank host logic of the benchmark, on CPU with the gloo backend (world size 2).

Rows are independent, so each rank runs its own replica (its own shard of routed
rows) with no data exchange; the only cross-rank steps are the barrier and the
max-over-ranks of the timed region.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        slowest = bench.max_over_ranks(10.0 + rank, w, torch.device("cpu"))
        rate = bench.whole_job_rate(1_600_000, w, 20, slowest)
        q.put((r, w, local, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, local, slowest, rate) in enumerate(res):
        assert (r, w, local) == (rank, world, rank)
        assert slowest == 11.0                     # the slowest rank's time, on every rank
        assert rate == 1_600_000 * 2 * 20 / 11.0   # units of all ranks / slowest time


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_clock_parsing():
    lines = [
        "0, 1965, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "0, 1980, 2070, 1100.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, 1990, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "garbage\n",
    ]
    c = bench.parse_clock_lines(lines)
    assert c["sm_mhz"] == 1980 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_lines([])["samples"] == 0

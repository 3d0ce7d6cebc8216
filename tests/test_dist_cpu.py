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


def test_reference_arm_line_keeps_the_contract(monkeypatch, capsys):
    """--impl reference on rank 0 prints one JSON line with the contract's keys: the oracle timed
    on the host cores on a bounded sample, its own cpu_baseline and a host-only e2e."""
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1", "--rows", "512"]) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 1
    assert line["config"]["workload"] == bench.WORKLOAD
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]


def test_host_numa_report_finds_the_buffer():
    h = torch.empty(1 << 22, dtype=torch.uint8)
    h.zero_()
    rep = bench.host_numa_report(h)
    if rep is not None:                         # /proc and /sys present (Linux)
        assert sum(rep["pages_by_node"].values()) > 0 and rep["node_free_GiB"]

"""Benchmark: SiTU-GLU forward + fused backward/router-gradient at the pages' scale.

One step = one pass of the whole hot path over one batch of routed rows:
    situ_glu_fwd(x) -> out        then        situ_glu_bwd_router(x, g, p) -> dx, dp
on R = 1,600,000 rows (100k tokens x 16 experts), H = 3072, inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints ONE JSON line (rank 0). ``value`` is whole-job rows/s (all ranks); the
roofline object reports the dominant kernel (the backward) against the measured
HBM copy bandwidth. ``--impl reference`` times the fp64 CPU oracle on the host
cores instead (bounded sample of the same workload), for the driver's ratio.

Multi-GPU: rows shard with no exchange, so each rank runs its own replica of
the workload on its own GPU (weak scaling); only the timing is reduced (max).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SiTU-GLU fwd+bwd rows/s and HBM GB/s (% of GB300 roofline) at R=1.6M,H=3072"
WORKLOAD = "pages_scale_r1600000_h3072"
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic of the backward kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), per row, and the hash of the kernel source it was taken on.
# Reported only while the source is unchanged; otherwise null.
NCU_TRAFFIC = {
    "source_sha256": "fa1328fb9fc97cf3f5b90d940a718f95065ef6fb516ba234eb3595fb94041587",
    "bwd_bytes_per_row": (1.208397e9 + 0.767695104e9) / 65536,
    "fwd_bytes_per_row": (0.805462e9 + 0.3650048e9) / 65536,
    "capture": "ncu --set full capture, backward kernel, R=65536, H=3072: dram__bytes_read.sum + "
               "dram__bytes_write.sum per row, times R; valid for kernel sources of sha256 {sha:.12}",
}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in ("bwd_situ_glu_gb300/csrc/situ_glu.cu", "bwd_situ_glu_gb300/csrc/situ_math.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-host", default="mapped", choices=["mapped", "cuda"],
                    help="host buffers of the e2e leg: page-aligned mappings registered with cudaHostRegister "
                         "(mapped) or page-locked memory from cudaHostAlloc (cuda)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 saved-x variant's timing")
    ap.add_argument("--no-dgrad", action="store_true", help="skip the fused dgrad GEMM's timing")
    ap.add_argument("--no-gateup", action="store_true", help="skip the fused gate/up GEMM's timing")
    ap.add_argument("--no-adam", action="store_true", help="skip the streamed host Adam step's timing")
    ap.add_argument("--only-dgrad", action="store_true", help="time only the fused dgrad GEMM (profiling runs)")
    ap.add_argument("--only-gateup", action="store_true", help="time only the fused gate/up GEMM (profiling runs)")
    ap.add_argument("--only-adam", action="store_true", help="time only the streamed host Adam step")
    ap.add_argument("--unfused", action="store_true",
                    help="with --only-dgrad / --only-gateup: also time the unfused route (library GEMM, then the "
                         "elementwise kernel)")
    ap.add_argument("--adam-params", type=int, default=1 << 28, help="parameters of the Adam leg")
    ap.add_argument("--gemm-rows", type=int, default=None, help="rows split evenly over --gemm-experts")
    ap.add_argument("--gemm-experts", type=int, default=None)
    ap.add_argument("--rows", type=int, default=None, help="override R (for small profiling runs)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank: int, world: int, steps: int, max_seconds: float) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return units_per_rank * world * steps / max_seconds


# ---------------------------------------------------------------- peaks, clocks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_clock_lines(lines):
    """nvidia-smi csv,noheader,nounits lines -> {"sm_mhz", "sm_max_mhz", "reasons", "samples"}."""
    sm, smax, reasons = [], [], set()
    for ln in lines:
        parts = [t.strip() for t in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        for name, flag in zip(REASON_NAMES, parts[5:9]):
            if flag.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


class ClockSampler:
    """Runs nvidia-smi in the background while the timed region runs."""

    def __init__(self, gpu_uuid=None, period_ms=100):
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                    f"-lms", str(period_ms)]
        if gpu_uuid:
            self.cmd += ["-i", gpu_uuid]
        self.lines = []
        self.proc = None
        self.thread = None
        self.first = threading.Event()

    def _reader(self):
        for ln in self.proc.stdout:
            self.lines.append(ln)
            self.first.set()

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        self.first.wait(timeout=5.0)
        self.lines.clear()

    def stop(self):
        if self.proc is None:
            return parse_clock_lines([])
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        return parse_clock_lines(self.lines)


# ---------------------------------------------------------------- CPU oracle timing

def oracle_rows_per_s(x_cpu, g_cpu, p_cpu, nthreads=0):
    """Time the fp64 oracle on one block of rows (fwd then bwd+router), return (rows/s, seconds)."""
    import numpy as np
    import torch

    import oracle
    xb = x_cpu.view(torch.int16).numpy().view(np.uint16)
    gb = g_cpu.view(torch.int16).numpy().view(np.uint16)
    pn = p_cpu.numpy()
    t0 = time.perf_counter()
    oracle.fwd_bf16(xb, nthreads=nthreads)
    oracle.bwd_router_bf16(xb, gb, pn, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return x_cpu.shape[0] / dt, dt


def cpu_baseline(get_rows, R, target_s):
    """Oracle rows/s on a bounded prefix of the workload, sized to ~target_s of CPU time."""
    import oracle
    cores = oracle.default_threads()
    n0 = min(R, 1024)
    x, g, p = get_rows(n0)
    rate0, dt0 = oracle_rows_per_s(x, g, p)
    n = int(min(R, max(n0, rate0 * target_s)))
    n -= n % 16
    n = max(n, 16)
    x, g, p = get_rows(n)
    rate, dt = oracle_rows_per_s(x, g, p)
    # and on one core, over a sample sized to ~target_s / 4
    n1 = int(min(n, max(16, rate / cores * target_s / 4)))
    n1 -= n1 % 16
    n1 = max(n1, 16)
    rate1, dt1 = oracle_rows_per_s(x[:n1], g[:n1], p[:n1], nthreads=1)
    return {"value": rate, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {R} rows (fwd then bwd+router grad, fp64, {cores} threads), {dt:.1f} s",
            "single_core": {"value": rate1, "unit": "rows/s", "cores": 1,
                            "sample": f"first {n1} rows on one thread, {dt1:.1f} s"}}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import situ_inputs as si
    w = si.get(WORKLOAD)
    R = args.rows or w.R
    import oracle
    oracle.build()
    cores = oracle.default_threads()

    # each step: a bounded sample of the same workload (same distributions and seed), on the host
    def sample(n):
        ws = si.Workload(w.name, n, w.H, w.x_kind, w.x_std, w.g_std, w.p_kind, w.order, w.seed)
        return si.generate(ws, device="cpu")

    x, g, p = sample(512)
    rate0, _ = oracle_rows_per_s(x, g, p)
    budget_steps = max(1, args.steps + args.warmup)
    n = int(max(256, min(R, rate0 * 150.0 / budget_steps)))   # whole run ~ 2.5 minutes at most
    n -= n % 16
    x, g, p = sample(n)
    for _ in range(args.warmup):
        oracle_rows_per_s(x, g, p)
    total = 0.0
    for _ in range(args.steps):
        _, dt = oracle_rows_per_s(x, g, p)
        total += dt
    rate = n * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "R": R, "H": w.H, "beta": 4.0, "lbeta": 25.0,
                   "step_sample_rows": n},
        "cpu_baseline": {"value": rate, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} rows of the workload per step (fwd then bwd+router grad, fp64)"},
        "e2e": {"value": rate, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- native arm

def run_gemm_only(args):
    """Time only the fused tensor-core kernels (profiling runs)."""
    import torch

    import bwd_situ_glu_gb300 as sg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sg.build()
    sg.load()
    peak, _ = load_peaks()
    line, ok = {}, True
    if args.only_dgrad:
        line["dgrad_fused"] = time_dgrad(sg, dev, args.steps, args.warmup, peak, rows=args.gemm_rows,
                                         experts=args.gemm_experts, unfused=args.unfused)
        ok &= line["dgrad_fused"]["status"] == 0
    if args.only_gateup:
        line["gateup_fused"] = time_gateup(sg, dev, args.steps, args.warmup, peak, rows=args.gemm_rows,
                                           experts=args.gemm_experts, unfused=args.unfused)
        ok &= line["gateup_fused"]["status"] == 0
    if args.only_adam:
        line["adam_stream"] = time_adam(sg, dev, args.steps, n=args.adam_params)
    print(json.dumps(line), flush=True)
    return 0 if ok else 1


def run_native(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import bwd_situ_glu_gb300 as sg
    import situ_inputs as si
    sg.build()
    sg.load()

    w = si.get(WORKLOAD)
    R = args.rows or w.R
    H = w.H
    # each rank draws its own shard of routed rows (different seed per rank)
    ws = si.Workload(w.name, R, H, w.x_kind, w.x_std, w.g_std, w.p_kind, w.order, w.seed + 1000 * rank)
    x, g, p = si.generate(ws, device=dev)
    out = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((R, 2 * H), dtype=torch.bfloat16, device=dev)
    dp = torch.empty((R,), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)

    def step():
        sg.situ_glu_fwd_ptr(x.data_ptr(), out.data_ptr(), R, H, 4.0, 25.0, sh)
        sg.situ_glu_bwd_router_ptr(x.data_ptr(), g.data_ptr(), p.data_ptr(), dx.data_ptr(), dp.data_ptr(),
                                   R, H, 4.0, 25.0, sh)

    torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    torch.cuda.nvtx.range_push("timed")
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        sg.situ_glu_fwd_ptr(x.data_ptr(), out.data_ptr(), R, H, 4.0, 25.0, sh)
        ev[i][1].record(stream)
        sg.situ_glu_bwd_router_ptr(x.data_ptr(), g.data_ptr(), p.data_ptr(), dx.data_ptr(), dp.data_ptr(),
                                   R, H, 4.0, 25.0, sh)
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(world)
    elapsed_ms = start.elapsed_time(end)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    max_ms = max_over_ranks(elapsed_ms, world, dev)

    fwd_bytes = 6 * H * R
    bwd_bytes = (10 * H + 8) * R
    peak, peak_src = load_peaks()
    fwd_avg, bwd_avg = sum(fwd_ms) / K, sum(bwd_ms) / K
    fwd_gbs = fwd_bytes / (fwd_avg * 1e-3) / 1e9
    bwd_gbs = bwd_bytes / (bwd_avg * 1e-3) / 1e9
    step_gbs = (fwd_bytes + bwd_bytes) / (elapsed_ms / K * 1e-3) / 1e9

    fp8 = None if args.no_fp8 else time_fp8(sg, x, g, p, out, dx, dp, R, H, stream, dev, K, args.warmup, peak)
    dgrad = None if args.no_dgrad else time_dgrad(sg, dev, max(3, min(K, 20)), args.warmup, peak, unfused=True)
    gateup = None if args.no_gateup else time_gateup(sg, dev, max(3, min(K, 20)), args.warmup, peak, unfused=True)
    # the same kernels on few large experts (32 x 8192 rows: the tensor-bound regime)
    dgrad_large = None if args.no_dgrad else time_dgrad(sg, dev, max(3, min(K, 20)), args.warmup, peak,
                                                        rows=1 << 18, experts=32)
    gateup_large = None if args.no_gateup else time_gateup(sg, dev, max(3, min(K, 20)), args.warmup, peak,
                                                           rows=1 << 18, experts=32)
    adam = None if args.no_adam else time_adam(sg, dev, 3, n=args.adam_params)

    traffic = None
    if NCU_TRAFFIC["source_sha256"] == kernel_source_hash() and NCU_TRAFFIC["bwd_bytes_per_row"]:
        traffic = NCU_TRAFFIC["bwd_bytes_per_row"] * R

    # ---------------- end to end through the public API: pinned host in, pinned host out
    e2e = None
    if not args.no_e2e:
        e2e = time_e2e(sg, x, g, p, out, dx, dp, R, H, stream, dev, args.e2e_steps, world, host=args.e2e_host)

    # ---------------- CPU baseline: the oracle on a bounded sample (rank 0 at N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        def rows(n):
            return x[:n].cpu(), g[:n].cpu(), p[:n].cpu()
        cpu = cpu_baseline(rows, R, args.cpu_seconds)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC,
        "value": whole_job_rate(R, world, K, max_ms * 1e-3),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": max_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "R": R, "H": H, "io_dtype": "bf16", "beta": 4.0, "lbeta": 25.0,
                   "parallelism": f"replicas x{world} (rows shard, no collective)",
                   "l2": "inputs larger than L2 (x alone is %.2f GB vs 129 MB L2); no flush" % (4 * H * R / 1e9)},
        "passes": {
            "fwd": {"ms": fwd_avg, "ms_median": statistics.median(fwd_ms), "ms_min": min(fwd_ms),
                    "GB_s": fwd_gbs, "frac_of_peak": fwd_gbs / peak,
                    "rows_per_s": R / (fwd_avg * 1e-3), "bytes": fwd_bytes},
            "bwd_router": {"ms": bwd_avg, "ms_median": statistics.median(bwd_ms), "ms_min": min(bwd_ms),
                           "GB_s": bwd_gbs, "frac_of_peak": bwd_gbs / peak,
                           "rows_per_s": R / (bwd_avg * 1e-3), "bytes": bwd_bytes},
            "step_GB_s": step_gbs,
        },
        "roofline": {"bound": "hbm", "kernel": "bwd_vec_kernel (situ_glu_bwd_router)",
                     "achieved": bwd_gbs, "peak": peak, "unit": "GB/s", "frac": bwd_gbs / peak,
                     "peak_source": f"{peak_src} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": bwd_bytes, "traffic": traffic,
                     "traffic_source": NCU_TRAFFIC["capture"].format(sha=NCU_TRAFFIC["source_sha256"])
                     if traffic is not None else None},
        "clocks": clocks,
        "gpu_launches": 2 * K,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "fp8_saved_x": fp8,
        "dgrad_fused": dgrad,
        "gateup_fused": gateup,
        "dgrad_fused_large_experts": dgrad_large,
        "gateup_fused_large_experts": gateup_large,
        "adam_stream": adam,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def time_fp8(sg, x, g, p, out, dx, dp, R, H, stream, dev, steps, warmup, peak):
    """The block-wise FP8 saved-x variant on the same workload: forward that also writes the
    E4M3 codes and block scales of x, backward + router gradient from them."""
    import torch
    nb = sg.fp8_scale_blocks(H)
    xq = torch.empty((R, 2 * H), dtype=torch.uint8, device=dev)
    xs = torch.empty((R, 2 * nb), dtype=torch.float32, device=dev)
    sh = int(stream.cuda_stream)
    lib = sg.load()

    def fwd():
        sg._check(lib.situ_glu_fwd_save_fp8(x.data_ptr(), out.data_ptr(), xq.data_ptr(), xs.data_ptr(), R, H,
                                            4.0, 25.0, sh))

    def bwd():
        sg._check(lib.situ_glu_bwd_router_fp8(xq.data_ptr(), xs.data_ptr(), g.data_ptr(), p.data_ptr(),
                                              dx.data_ptr(), dp.data_ptr(), R, H, 4.0, 25.0, sh))

    for _ in range(max(1, warmup)):
        fwd()
        bwd()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    f_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    b_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    fb = (8 * H + 8 * nb) * R
    bb = (8 * H + 8 * nb + 8) * R
    del xq, xs
    return {"fwd_save_fp8": {"ms": f_ms, "GB_s": fb / f_ms / 1e6, "frac_of_peak": fb / f_ms / 1e6 / peak, "bytes": fb},
            "bwd_router_fp8": {"ms": b_ms, "GB_s": bb / b_ms / 1e6, "frac_of_peak": bb / b_ms / 1e6 / peak, "bytes": bb},
            "rows_per_s": R / ((f_ms + b_ms) * 1e-3),
            "saved_bytes_per_row": {"bf16_x": 4 * H, "fp8_x": 2 * H + 8 * nb},
            "gpu_launches": 2 * steps}


def grouped_workload(seed, rows=None, experts=None):
    """Expert-grouped routed rows: 16384 tokens x top-16 of 896 experts, rows sorted by expert
    (H = 3072), or with rows and experts given, that many rows split evenly over that many
    experts. Returns (counts per expert, router weights p [R] on the CPU, workload name, H)."""
    import numpy as np
    import torch

    import situ_inputs as si
    w = si.get("expert_grouped_r262144_h3072")
    if rows and experts:
        counts = np.full(experts, rows // experts, dtype=np.int64)
        counts[: rows % experts] += 1
        p = torch.rand(rows, generator=torch.Generator().manual_seed(seed))
        return counts, p, f"uniform_r{rows}_e{experts}_h{w.H}", w.H, w.x_std
    p, experts_of_row, _ = si.router_rows(w.tokens, w.seed, order="expert")
    counts = np.bincount(experts_of_row.numpy(), minlength=si.N_EXPERTS)
    return counts, p, f"expert_grouped_r{w.R}_h{w.H}, {si.N_EXPERTS} experts", w.H, w.x_std


def bf16_tflops_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def randn_bf16(shape, gen, dev, scale=1.0, chunk=1 << 27):
    """Seeded N(0, scale²) bf16 tensor, generated on the device in chunks of `chunk` elements."""
    import torch
    t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    flat = t.view(-1)
    for a in range(0, flat.numel(), chunk):
        b = min(flat.numel(), a + chunk)
        flat[a:b] = (torch.randn(b - a, generator=gen, device=dev) * scale).to(torch.bfloat16)
    return t


def time_launches(fn, stream, steps, warmup):
    """Average ms per launch of fn over `steps` back-to-back launches on `stream` (CUDA events),
    after `warmup` untimed ones."""
    import torch
    for _ in range(max(1, warmup)):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def gemm_result(workload, ms, flops, nbytes, hbm_peak, steps, status):
    tf_peak, tf_src = bf16_tflops_peak()
    t_flop = flops / (tf_peak * 1e12) * 1e3
    t_byte = nbytes / (hbm_peak * 1e9) * 1e3
    return {"workload": workload,
            "ms": ms, "TFLOP_s": flops / ms / 1e9, "frac_of_bf16_peak": flops / ms / 1e9 / tf_peak,
            "bf16_peak": tf_peak, "bf16_peak_source": tf_src,
            "GB_s": nbytes / ms / 1e6, "frac_of_hbm_peak": nbytes / ms / 1e6 / hbm_peak,
            "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
            "bound": "tensor" if t_flop >= t_byte else "hbm",
            "roofline_frac": max(t_flop, t_byte) / ms, "status": status, "gpu_launches": steps}


def library_grouped_gemm(a, b_kn, off_cpu, out):
    """The route a fusion replaces starts with a plain library grouped GEMM: out rows of expert e
    = a[rows of e] @ b_kn[e] in bf16 (fp32 accumulation), b_kn [E, K, N] (a transposed view of the
    K-major weights): cuBLAS per expert (torch.mm into row slices of out), captured once into a
    CUDA graph and replayed, so that launch overhead does not count against it. Returns fn() -> out.
    (torch's one-launch grouped GEMM is not used: on this GPU it faulted on row counts that are not
    multiples of 16.)"""
    import torch
    E = b_kn.shape[0]

    def per_expert():
        for e in range(E):
            r0, r1 = int(off_cpu[e]), int(off_cpu[e + 1])
            if r1 > r0:
                torch.mm(a[r0:r1], b_kn[e], out=out[r0:r1])

    side = torch.cuda.Stream(a.device)
    side.wait_stream(torch.cuda.current_stream(a.device))
    with torch.cuda.stream(side):
        per_expert()                                  # cuBLAS handles and workspaces before capture
    torch.cuda.current_stream(a.device).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        per_expert()

    def replay():
        graph.replay()
        return out
    return replay


def time_dgrad(sg, dev, steps, warmup, hbm_peak, seed=5, D=3584, rows=None, experts=None, unfused=False):
    """Fused down-projection dgrad (tcgen05 grouped GEMM) + backward + router gradient on the
    expert-grouped workload, D = 3584 (the expert output width), synthetic N(0, 1/D) weights.
    unfused: also time, on the same tensors, the route the fusion replaces (a library grouped
    GEMM writing g in bf16, then situ_glu_bwd_router reading it back)."""
    import numpy as np
    import torch
    counts, p, workload, H, x_std = grouped_workload(seed, rows, experts)
    R, E = int(counts.sum()), len(counts)
    gen = torch.Generator(device=dev).manual_seed(seed)
    x = randn_bf16((R, 2 * H), gen, dev, x_std)
    dy = randn_bf16((R, D), gen, dev)
    wt = randn_bf16((E, H, D), gen, dev, 1.0 / D ** 0.5)
    off_cpu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    off = torch.from_numpy(off_cpu).to(dev)
    p = p.to(dev)
    dx = torch.empty(R, 2 * H, dtype=torch.bfloat16, device=dev)
    dp = torch.empty(R, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ms = time_launches(lambda: sg.situ_glu_bwd_router_dgrad(x, dy, wt, off, p, dx, dp, status=status),
                       stream, steps, warmup)
    nbytes = R * D * 2 + E * H * D * 2 + R * 4 * H + R * 4 * H + R * 8 + (E + 1) * 8
    res = gemm_result(f"{workload} x D={D}", ms, 2.0 * R * D * H, nbytes, hbm_peak, steps, int(status.item()))
    if unfused:
        g = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
        gemm = library_grouped_gemm(dy, wt.transpose(1, 2), off_cpu, g)
        route = "cuBLAS per expert (torch.mm), one CUDA graph"
        dx2 = torch.empty_like(dx)
        dp2 = torch.empty_like(dp)

        def unfused_step():
            sg.situ_glu_bwd_router(x, gemm(), p, dx2, dp2)
        ms_u = time_launches(unfused_step, stream, steps, warmup)
        rel = ((dp2 - dp).abs() / dp.abs().clamp_min(1e-30)).median().item()
        res["unfused"] = {"ms": ms_u, "route": route + ", then situ_glu_bwd_router",
                          "bytes": nbytes + R * H * 2 * 2, "fused_speedup": ms_u / ms,
                          "dp_median_rel_diff_vs_fused": rel,
                          "what": "g = dY·W_down,e written to HBM in bf16 and read back by the backward"}
        del dx2, dp2, g, gemm
    del x, dy, wt, dx, dp
    torch.cuda.empty_cache()
    return res


def time_gateup(sg, dev, steps, warmup, hbm_peak, seed=6, D=3584, rows=None, experts=None, unfused=False):
    """Fused gate/up projection (tcgen05 grouped GEMM, N = 2H) + SiTU-GLU forward on the
    expert-grouped workload: h [R, D] ~ N(0, 1), [W_gate; W_up] ~ N(0, x_std²/D) per expert.
    unfused: also time, on the same tensors, the route the fusion replaces (a library grouped
    GEMM writing x in bf16, then situ_glu_fwd reading it back)."""
    import numpy as np
    import torch
    counts, _, workload, H, x_std = grouped_workload(seed, rows, experts)
    R, E = int(counts.sum()), len(counts)
    gen = torch.Generator(device=dev).manual_seed(seed)
    h = randn_bf16((R, D), gen, dev)
    w = randn_bf16((E, 2 * H, D), gen, dev, x_std / D ** 0.5)
    off_cpu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    off = torch.from_numpy(off_cpu).to(dev)
    x = torch.empty(R, 2 * H, dtype=torch.bfloat16, device=dev)
    out = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ms = time_launches(lambda: sg.situ_glu_fwd_gateup(h, w, off, x, out, status=status), stream, steps, warmup)
    nbytes = R * D * 2 + E * 2 * H * D * 2 + R * 4 * H + R * 2 * H + (E + 1) * 8
    res = gemm_result(f"{workload} x D={D}", ms, 2.0 * R * D * 2 * H, nbytes, hbm_peak, steps, int(status.item()))
    if unfused:
        xu = torch.empty(R, 2 * H, dtype=torch.bfloat16, device=dev)
        gemm = library_grouped_gemm(h, w.transpose(1, 2), off_cpu, xu)
        route = "cuBLAS per expert (torch.mm), one CUDA graph"
        out2 = torch.empty_like(out)

        def unfused_step():
            sg.situ_glu_fwd(gemm(), out2)
        ms_u = time_launches(unfused_step, stream, steps, warmup)
        same = (out2.view(torch.int16) == out.view(torch.int16)).float().mean().item()
        res["unfused"] = {"ms": ms_u, "route": route + ", then situ_glu_fwd",
                          "bytes": nbytes + R * 2 * H * 2, "fused_speedup": ms_u / ms,
                          "out_bitwise_equal_fraction_vs_fused": same,
                          "what": "the projection x written to HBM in bf16 and read back by the forward"}
        del out2, xu, gemm
    del h, w, x, out
    torch.cuda.empty_cache()
    return res


def time_adam(sg, dev, steps, n=1 << 28, chunk=1 << 24, nslots=2, seed=7):
    """Adam on host-resident state, streamed (the streaming-gradients design) against the one-big-
    transfer baseline it replaces, on n parameters: device fp32 gradients, host fp32 master + bf16
    moments, device bf16 working weights. Also times each leg alone (gradient D2H, weight H2D, the
    host update on resident data) to give the overlap roofline: a perfectly overlapped step takes
    max(D2H + H2D on the one copy stream, host update)."""
    import time

    import numpy as np
    import torch
    gen = torch.Generator(device=dev).manual_seed(seed)
    grad = torch.randn(n, generator=gen, device=dev) * 1e-3
    weight = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    master = torch.zeros(n, dtype=torch.float32).normal_(0, 0.02)
    m = torch.zeros(n, dtype=torch.bfloat16)
    v = torch.zeros(n, dtype=torch.bfloat16)
    staging = pinned_like(torch.empty(sg.adam_staging_bytes(chunk, nslots), dtype=torch.uint8))
    stream = torch.cuda.current_stream(dev)
    threads = len(os.sched_getaffinity(0))

    def streamed(step):
        sg.situ_adam_stream_step(grad, weight, master, m, v, sg.adam_params(step=step), staging, chunk, nslots,
                                 threads, stream)

    for i in range(2):                                    # warm-up (page faults, thread start)
        streamed(i + 1)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(steps):
        streamed(i + 3)
    t_stream = (time.perf_counter() - t0) / steps

    # the baseline: one parameter-sized fp32 host gradient buffer, one transfer each way
    gbuf = pinned_like(torch.empty(n, dtype=torch.float32))
    wbuf = pinned_like(torch.empty(n, dtype=torch.bfloat16))

    def one_big(step):
        gbuf.copy_(grad, non_blocking=True)
        torch.cuda.synchronize(dev)
        sg.situ_adam_update_host(master, m, v, gbuf, wbuf, sg.adam_params(step=step), threads)
        weight.copy_(wbuf, non_blocking=True)
        torch.cuda.synchronize(dev)

    one_big(1)
    t0 = time.perf_counter()
    for i in range(steps):
        one_big(i + 2)
    t_big = (time.perf_counter() - t0) / steps

    # legs alone
    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / reps
    t_d2h = timed(lambda: gbuf.copy_(grad, non_blocking=True))
    t_h2d = timed(lambda: weight.copy_(wbuf, non_blocking=True))
    t_upd = timed(lambda: sg.situ_adam_update_host(master, m, v, gbuf, wbuf, sg.adam_params(step=9), threads))
    ideal = max(t_d2h + t_h2d, t_upd)
    # host memory: a multi-threaded copy of 1 GiB (read + write bytes), the denominator of the
    # host-memory roofline; the streamed step moves 28 B per parameter through host memory
    # (update: read g 4, master 4, m 2, v 2; write master 4, m 2, v 2, weight slot 2; DMA: the
    # gradient slot written 4, the weight slot read 2)
    torch.set_num_threads(threads)
    src = torch.empty(1 << 28, dtype=torch.float32).fill_(1.0)
    dst = torch.empty_like(src)
    t_copy = timed(lambda: dst.copy_(src), reps=5)
    host_peak = 2 * src.numel() * 4 / t_copy / 1e9
    del src, dst
    host_gbs = 28 * n / t_stream / 1e9
    for t in (staging, gbuf, wbuf):
        torch.cuda.cudart().cudaHostUnregister(t.data_ptr())
    del grad, weight
    torch.cuda.empty_cache()
    return {"params": n, "chunk": chunk, "nslots": nslots, "host_threads": threads,
            "ms": t_stream * 1e3, "params_per_s": n / t_stream,
            "one_big_transfer_ms": t_big * 1e3, "one_big_transfer_params_per_s": n / t_big,
            "host_bytes_per_param": {"streamed": 8 + sg.adam_staging_bytes(chunk, nslots) / n, "one_big_transfer": 12},
            "legs_ms": {"grad_d2h": t_d2h * 1e3, "weight_h2d": t_h2d * 1e3, "host_update": t_upd * 1e3},
            "link_GB_s": {"d2h": 4 * n / t_d2h / 1e9, "h2d": 2 * n / t_h2d / 1e9},
            "host_update_params_per_s": n / t_upd,
            "roofline": {"bound": "host_memory", "achieved": host_gbs, "peak": host_peak, "unit": "GB/s",
                         "frac": host_gbs / host_peak, "bytes_per_param": 28,
                         "peak_source": "measured here: multi-threaded host copy of 1 GiB, read + write bytes"},
            "overlap": {"slowest_leg": "host_update" if t_upd >= t_d2h + t_h2d else "host_link",
                        "ideal_ms": ideal * 1e3, "frac": ideal / t_stream},
            "timing": "host wall clock per step (the step returns when every chunk's weights are on the device)"}


def host_numa_report(h):
    """Where the pages of host tensor h live (NUMA node -> pages, from /proc/self/numa_maps) and
    each node's free memory: a slow host link on some boxes goes with buffers placed away from
    the GPU's node. Best effort (None where the files are missing)."""
    try:
        a0, a1 = h.data_ptr(), h.data_ptr() + h.numel() * h.element_size()
        starts = set()
        with open("/proc/self/maps") as f:                 # the mappings that overlap h
            for line in f:
                lo, hi = (int(v, 16) for v in line.split()[0].split("-"))
                if lo < a1 and hi > a0:
                    starts.add(lo)
        pages = {}
        with open("/proc/self/numa_maps") as f:
            for line in f:
                if int(line.split()[0], 16) in starts:
                    for w in line.split():
                        if w.startswith("N") and "=" in w:
                            k, v = w[1:].split("=")
                            pages[k] = pages.get(k, 0) + int(v)
        free = {}
        import glob
        for d in sorted(glob.glob("/sys/devices/system/node/node*")):
            for line in open(d + "/meminfo"):
                if "MemFree" in line:
                    free[d.rsplit("node", 1)[1]] = int(line.split()[3]) // (1 << 20)
        return {"pages_by_node": pages, "node_free_GiB": free}
    except (OSError, ValueError):
        return None


def pinned_like(t):
    """Host tensor of t's shape and dtype in its own page-aligned anonymous mapping, touched and
    page-locked with cudaHostRegister (exact size).

    Registered portable | mapped (flags 3): on this platform device->host copies into memory
    registered with flags 0 ran at ~31 GB/s against ~190 GB/s with these flags. A mapping of its
    own rather than torch's (malloc'd) host storage: on some boxes of the pool, host->device
    copies from registered 16 GB malloc'd buffers ran at ~18 GB/s against ~140 GB/s from
    registered page-aligned mappings of the same size (measured back to back on one box, after
    a host-memory-heavy run), and with MADV_HUGEPAGE on the mapping ~190-210 GB/s."""
    import ctypes
    import mmap

    import numpy as np
    import torch
    nbytes = t.numel() * t.element_size()
    buf = np.frombuffer(mmap.mmap(-1, max(nbytes, 1)), dtype=np.uint8, count=nbytes)
    if nbytes:                                      # transparent huge pages where the kernel has them
        ctypes.CDLL(None).madvise(ctypes.c_void_p(buf.ctypes.data), ctypes.c_size_t(nbytes), 14)
    buf[:] = 0                                      # touch every page before registering
    h = torch.from_numpy(buf).view(t.dtype).view(t.shape)   # keeps the mapping alive
    rc = torch.cuda.cudart().cudaHostRegister(h.data_ptr(), nbytes, 3)
    if int(rc) != 0:
        raise RuntimeError(f"cudaHostRegister failed: {rc}")
    return h


def unpin(h):
    import torch
    torch.cuda.cudart().cudaHostUnregister(h.data_ptr())


def pinned_cuda(t):
    """Host tensor of t's shape and dtype in page-locked memory from cudaHostAlloc (torch's pinned
    allocator), zero-filled."""
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.zero_()
    return h


def time_e2e(sg, x, g, p, out, dx, dp, R, H, stream, dev, steps, world, chunk_rows=65536, host="mapped"):
    """The step through the public binding with every input copied in from page-locked host
    memory and every result copied back, inside the timed region.

    Rows are independent, so the step streams over row chunks on three CUDA streams:
    host->device copies of chunk i+1 and device->host copies of chunk i-1 overlap the kernels
    of chunk i. Events order the reuse of each chunk's device rows across steps."""
    import torch
    steps = max(1, steps)
    alloc = pinned_like if host == "mapped" else pinned_cuda
    xh, gh, ph, oh, dxh, dph = (alloc(t) for t in (x, g, p, out, dx, dp))
    xh.copy_(x)
    gh.copy_(g)
    ph.copy_(p)
    h2d = xh.numel() * 2 + gh.numel() * 2 + ph.numel() * 4
    d2h = oh.numel() * 2 + dxh.numel() * 2 + dph.numel() * 4
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), stream, torch.cuda.Stream(dev)
    bounds = [(r0, min(R, r0 + chunk_rows)) for r0 in range(0, R, chunk_rows)]
    n = len(bounds)
    computed = [None] * n   # event: kernels of chunk i done (its x/g/p may be overwritten)
    drained = [None] * n    # event: results of chunk i copied out (its out/dx/dp may be overwritten)
    launches = [0]

    def one_step():
        for i, (a, b) in enumerate(bounds):
            with torch.cuda.stream(s_in):
                if computed[i] is not None:
                    s_in.wait_event(computed[i])
                x[a:b].copy_(xh[a:b], non_blocking=True)
                g[a:b].copy_(gh[a:b], non_blocking=True)
                p[a:b].copy_(ph[a:b], non_blocking=True)
                loaded = torch.cuda.Event()
                loaded.record(s_in)
            s_cmp.wait_event(loaded)
            if drained[i] is not None:
                s_cmp.wait_event(drained[i])
            sg.situ_glu_fwd(x[a:b], out[a:b], stream=s_cmp)
            sg.situ_glu_bwd_router(x[a:b], g[a:b], p[a:b], dx[a:b], dp[a:b], stream=s_cmp)
            launches[0] += 2
            done = torch.cuda.Event()
            done.record(s_cmp)
            computed[i] = done
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                oh[a:b].copy_(out[a:b], non_blocking=True)
                dxh[a:b].copy_(dx[a:b], non_blocking=True)
                dph[a:b].copy_(dp[a:b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_out)
            drained[i] = ev

    one_step()
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    launches[0] = 0
    start.record(s_in)
    s_cmp.wait_event(start)
    s_out.wait_event(start)
    for _ in range(steps):
        one_step()
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    end.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(end), world, dev)

    # the host link of this machine, measured on the same buffers: x alone each way, then both
    # directions at once (x in, dx out on two streams) — the step cannot beat moving its bytes
    def copy_ms(fn, reps=3):
        fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    def both_ways():
        with torch.cuda.stream(s_in):
            x.copy_(xh, non_blocking=True)
        with torch.cuda.stream(s_out):
            dxh.copy_(dx, non_blocking=True)
        torch.cuda.current_stream(dev).wait_stream(s_in)
        torch.cuda.current_stream(dev).wait_stream(s_out)
    nbx = xh.numel() * 2
    t_in = copy_ms(lambda: x.copy_(xh, non_blocking=True))
    t_out = copy_ms(lambda: dxh.copy_(dx, non_blocking=True))
    t_both = copy_ms(both_ways)
    link = {"h2d_GB_s": nbx / t_in / 1e6, "d2h_GB_s": nbx / t_out / 1e6, "both_ways_GB_s": 2 * nbx / t_both / 1e6,
            "host_memory": host_numa_report(xh)}
    link_ms = (h2d + d2h) / (link["both_ways_GB_s"] * 1e6)
    if host == "mapped":
        for t in (xh, gh, ph, oh, dxh, dph):
            unpin(t)
    return {"value": whole_job_rate(R, world, steps, ms * 1e-3), "unit": "rows/s", "steps": steps,
            "ms_per_step": ms / steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "gpu_launches": launches[0],
            "host_link": link, "link_bound_ms_per_step": link_ms, "frac_of_link_bound": link_ms / (ms / steps),
            "host_buffers": "page-aligned mappings + cudaHostRegister" if host == "mapped" else "cudaHostAlloc",
            "how": f"page-locked host x,g,p -> device -> fwd + bwd via the binding -> out,dx,dp -> host, "
                   f"streamed over {n} row chunks of {chunk_rows} on 3 CUDA streams; host_link measured on "
                   f"the same buffers in the same run"}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.only_dgrad or args.only_gateup or args.only_adam:
        return run_gemm_only(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())

"""Element-by-element comparison of the CUDA path with the fp64 oracle.

Acceptance (the stated tolerance of the method's port):
* bf16 outputs (out, dx):  |gpu - ref| <= max(ulp_bf16(ref), 1e-3),
  ulp_bf16(ref) = 2^(floor(log2|ref|) - 7)  (0 for ref == 0, leaving the 1e-3 floor);
* fp32 dp:  |gpu - ref| <= 1e-3·|ref| + 1e-6·Σ_j|g_j·a_j| + 2^-126.
  The second term only matters where the row sum cancels to nearly zero, where a
  purely relative bound is ill-posed; the count of rows that needed it is reported.
  The last is the smallest normal fp32: an fp32 result cannot resolve values below it.
A NaN on one side must be a NaN on the other (non-finite inputs propagate).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle

BF16_ABS_FLOOR = 1e-3
DP_REL = 1e-3
DP_ABS_SCALE = 1e-6
FP32_MIN_NORMAL = 2.0 ** -126


def bits_of(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 numpy array of its storage bits."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return np.left_shift(b, 16, dtype=np.uint32).view(np.float32).astype(np.float64)


def ulp_bf16_reference(ref: np.ndarray) -> np.ndarray:
    """2^(floor(log2|ref|) - 7), 0 for ref == 0: the definition, through frexp (slow)."""
    mag = np.abs(ref)
    _, e = np.frexp(mag)                 # mag = m·2^e, m in [0.5, 1)  ->  floor(log2 mag) = e - 1
    u = np.ldexp(1.0, (e - 8).astype(np.int32))
    return np.where(mag == 0, 0.0, u)


def ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """The same from the float64 exponent field: for a normal double of biased exponent b,
    floor(log2|ref|) = b - 1023, so the ulp is the double with exponent field b - 7 and a zero
    mantissa. Doubles with b < 8 (|ref| < 2^-1016, including 0 and subnormals, all far below
    the 1e-3 floor of the tolerance) give 0; NaN and infinity give 2^-8 as frexp's exponent 0
    does in the definition."""
    ref = np.ascontiguousarray(ref, dtype=np.float64)
    b = (ref.view(np.uint64) >> np.uint64(52)) & np.uint64(0x7FF)
    u = ((np.maximum(b, np.uint64(8)) - np.uint64(7)) << np.uint64(52)).view(np.float64)
    u = np.where(b < 8, 0.0, u)
    return np.where(b == 0x7FF, 2.0 ** -8, u)


@dataclass
class Tally:
    n: int = 0
    bad: int = 0
    worst_ratio: float = 0.0     # max |err| / tol
    worst_abs: float = 0.0
    examples: list = field(default_factory=list)


@dataclass
class DpTally(Tally):
    floor_rows: int = 0          # rows that passed only thanks to the cancellation term
    worst_rel: float = 0.0


class Parity:
    def __init__(self, name: str):
        self.name = name
        self.t = {"out": Tally(), "dx": Tally(), "dp": DpTally()}

    def bf16(self, key: str, gpu_bits: np.ndarray, ref: np.ndarray, row0: int = 0):
        gpu = bf16_bits_to_f64(gpu_bits)
        nan_ref, nan_gpu = np.isnan(ref), np.isnan(gpu)
        tol = np.maximum(ulp_bf16(ref), BF16_ABS_FLOOR)
        with np.errstate(invalid="ignore"):
            err = np.abs(gpu - ref)
            bad = (err > tol) | (nan_ref != nan_gpu)
            bad &= ~(nan_ref & nan_gpu)
            ratio = np.where(nan_ref | nan_gpu, 0.0, err / tol)
        tl = self.t[key]
        tl.n += ref.size
        nb = int(bad.sum())
        tl.bad += nb
        if ref.size:
            tl.worst_ratio = max(tl.worst_ratio, float(np.nanmax(ratio)))
            tl.worst_abs = max(tl.worst_abs, float(np.nanmax(np.where(nan_ref | nan_gpu, 0.0, err))))
        if nb and len(tl.examples) < 5:
            for idx in np.argwhere(bad)[:5 - len(tl.examples)]:
                idx = tuple(int(i) for i in idx)
                tl.examples.append((row0 + idx[0],) + idx[1:] + (float(gpu[idx]), float(ref[idx])))

    def dp(self, gpu: np.ndarray, ref: np.ndarray, ref_abs: np.ndarray, row0: int = 0):
        gpu = gpu.astype(np.float64)
        both_nan = np.isnan(gpu) & np.isnan(ref)
        with np.errstate(invalid="ignore"):
            err = np.where(both_nan, 0.0, np.abs(gpu - ref))
            rel_tol = DP_REL * np.abs(ref)
            tol = np.where(both_nan, 0.0, rel_tol + DP_ABS_SCALE * ref_abs + FP32_MIN_NORMAL)
        bad = ~(err <= tol)
        tl = self.t["dp"]
        tl.n += ref.size
        tl.bad += int(bad.sum())
        with np.errstate(invalid="ignore"):
            tl.floor_rows += int(((err > rel_tol) & ~bad).sum())
        if ref.size:
            tl.worst_ratio = max(tl.worst_ratio, float(np.nanmax(np.where(tol > 0, err / np.maximum(tol, 1e-300), 0))))
            tl.worst_abs = max(tl.worst_abs, float(np.nanmax(err)))
            nz = (np.abs(ref) > 0) & ~both_nan
            if nz.any():
                tl.worst_rel = max(tl.worst_rel, float((err[nz] / np.abs(ref[nz])).max()))
        for i in np.nonzero(bad)[0][:5 - len(tl.examples)]:
            tl.examples.append((row0 + int(i), float(gpu[i]), float(ref[i]), float(ref_abs[i])))

    def summary(self) -> str:
        parts = [self.name]
        for k, tl in self.t.items():
            if tl.n:
                s = f"{k}: n={tl.n} bad={tl.bad} worst_err/tol={tl.worst_ratio:.3g} max_abs={tl.worst_abs:.3g}"
                if k == "dp":
                    s += f" max_rel={tl.worst_rel:.3g} floor_rows={tl.floor_rows}"
                parts.append(s)
        return " | ".join(parts)

    def assert_ok(self):
        print(self.summary())
        for k, tl in self.t.items():
            assert tl.bad == 0, f"{self.name}: {k} has {tl.bad} elements out of tolerance, e.g. {tl.examples}"


def compare_rows(par: Parity, x, g, p, out, dx, dp, beta=4.0, lbeta=25.0, row0=0, nthreads=0):
    """Compare one block of rows (CPU or GPU tensors) against the oracle. Any of out / dx+dp may be None."""
    xb = bits_of(x)
    if out is not None:
        ref = oracle.fwd_bf16(xb, beta, lbeta, nthreads)
        par.bf16("out", bits_of(out), ref, row0)
    if dx is not None:
        dx_ref, dp_ref, dpa = oracle.bwd_router_bf16(xb, bits_of(g), p.detach().cpu().numpy(), beta, lbeta, nthreads)
        par.bf16("dx", bits_of(dx), dx_ref, row0)
        par.dp(dp.detach().cpu().numpy(), dp_ref, dpa, row0)


def compare_full(par: Parity, x, g, p, out, dx, dp, beta=4.0, lbeta=25.0, chunk_rows=8192):
    """Every row, in blocks of chunk_rows (several blocks at once: for_blocks_parallel)."""
    cut = lambda t, r0, r1: None if t is None else t[r0:r1]

    def check(part, r0, r1, nthreads):
        compare_rows(part, x[r0:r1], cut(g, r0, r1), cut(p, r0, r1), cut(out, r0, r1), cut(dx, r0, r1),
                     cut(dp, r0, r1), beta, lbeta, row0=r0, nthreads=nthreads)

    for_blocks_parallel(par, x.shape[0], check, chunk_rows)


def merge(into: Parity, part: Parity):
    """Add the tallies of `part` (a disjoint block of rows) to `into`."""
    for k, a in into.t.items():
        b = part.t[k]
        a.n += b.n
        a.bad += b.bad
        a.worst_ratio = max(a.worst_ratio, b.worst_ratio)
        a.worst_abs = max(a.worst_abs, b.worst_abs)
        a.examples.extend(b.examples[:max(0, 5 - len(a.examples))])
        if k == "dp":
            a.floor_rows += b.floor_rows
            a.worst_rel = max(a.worst_rel, b.worst_rel)


def for_blocks_parallel(par: Parity, R: int, check, chunk_rows=16384, workers=4):
    """Run check(part, r0, r1, nthreads) over the row blocks [r0, r1) of [0, R) with `workers`
    blocks in flight at once (device-to-host copies, the oracle and numpy release the GIL); each
    block has its share of the host's cores for the oracle and its own tallies, merged into par
    in row order. An exception in a block (an assertion) propagates."""
    import concurrent.futures as cf
    nthreads = max(1, oracle.default_threads() // workers)

    def one(r0):
        part = Parity(par.name)
        check(part, r0, min(R, r0 + chunk_rows), nthreads)
        return part

    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        for part in ex.map(one, range(0, R, chunk_rows)):
            merge(par, part)


def compare_full_parallel(par: Parity, x, g, p, out, dx, dp, beta=4.0, lbeta=25.0, chunk_rows=16384,
                          workers=4):
    """compare_full over all rows, several blocks at once (for_blocks_parallel)."""
    def check(part, r0, r1, nthreads):
        compare_rows(part, x[r0:r1], g[r0:r1], p[r0:r1], out[r0:r1], dx[r0:r1], dp[r0:r1], beta, lbeta,
                     row0=r0, nthreads=nthreads)

    for_blocks_parallel(par, x.shape[0], check, chunk_rows, workers)


def expert_groups(offsets, rows_per_group: int = 16384):
    """Split experts 0..E-1 (rows offsets[e]..offsets[e+1]-1, grouped by expert) into runs of
    consecutive experts holding about rows_per_group rows each: a list of (e0, e1), e1 exclusive."""
    offsets = np.asarray(offsets, dtype=np.int64)
    E = len(offsets) - 1
    groups, e0 = [], 0
    for e in range(E):
        if offsets[e + 1] - offsets[e0] >= rows_per_group or e == E - 1:
            groups.append((e0, e + 1))
            e0 = e + 1
    return groups


def for_expert_groups_parallel(par: Parity, offsets, check, rows_per_group: int = 16384, workers: int = 4):
    """Run check(part, e0, e1, nthreads) over runs of consecutive experts (expert_groups) with
    `workers` runs in flight at once, each with its own tallies merged into par in row order;
    returns the list of check's return values. An exception in a run propagates."""
    import concurrent.futures as cf
    nthreads = max(1, oracle.default_threads() // workers)

    def one(g):
        part = Parity(par.name)
        res = check(part, g[0], g[1], nthreads)
        return part, res

    results = []
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        for part, res in ex.map(one, expert_groups(offsets, rows_per_group)):
            merge(par, part)
            results.append(res)
    return results

"""Seeded synthetic inputs for SiTU-GLU (shared by the tests, the benchmark and smoke).

This module holds none of the method's arithmetic: it only draws random
tensors with the shapes, distributions and row structure of the workloads,
so both the CUDA path and the oracle can be fed the same bytes.

Row structure follows the MoE layer the pages describe:

* R = tokens × 16 routed experts, expert intermediate width H = 3072
  ("Frontier-scale RL with Kimi K3", section "Streaming activations").
* The router weight ``p`` of a routed row is the softmax over the top-16 of 896
  router scores of its token ("Inside Kimi K3", section "Idea One", top-k
  routing pseudocode; "Kimi K3 模型结构（9）：显存", the expert equation
  ``y = Σ_{e in top-k} p_e o_e``).

Values are drawn with ``torch.Generator`` seeded per workload. The draw
depends on the device kind (PyTorch's CPU and CUDA generators differ), so a
parity check always hands the very same tensors (copied, never regenerated)
to both sides.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

N_EXPERTS = 896
TOP_K = 16


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    H: int
    x_kind: str          # "normal" | "mixture"
    x_std: float
    g_std: float
    p_kind: str          # "router" | "uniform"
    order: str           # "token" (row = 16·t + k) | "expert" (rows grouped by expert id)
    seed: int

    @property
    def tokens(self) -> int:
        return self.R // TOP_K


# The five workloads. Names say what they are; sizes are in the names.
WORKLOADS = {
    # 64 tokens × 16 experts, H = 3072, x ~ N(0, 3²), g ~ N(0, 1), router p
    "routed_r1024_h3072": Workload("routed_r1024_h3072", 1024, 3072, "normal", 3.0, 1.0, "router", "token", 0),
    # 1024 tokens × 16; x: N(0,3²) mixed with U[-80, 80] (tanh saturation) and exact ±0
    "saturating_mix_r16384_h3072": Workload("saturating_mix_r16384_h3072", 16384, 3072, "mixture", 3.0, 1.0,
                                            "router", "token", 1),
    # 16384 tokens × 16; x ~ N(0, 2²), g ~ N(0, 0.5²); rows grouped contiguously by expert id
    "expert_grouped_r262144_h3072": Workload("expert_grouped_r262144_h3072", 262144, 3072, "normal", 2.0, 0.5,
                                             "router", "expert", 2),
    # the pages' scale: ~100k tokens × 16 experts, H = 3072 (x alone is 19.66 GB)
    "pages_scale_r1600000_h3072": Workload("pages_scale_r1600000_h3072", 1_600_000, 3072, "normal", 3.0, 1.0,
                                           "router", "token", 3),
}

# Shape / tail sweep: H in {3584, 3072, 1000} × R in {1, 37, 65537, 524288}; x ~ N(0, 4²),
# g ~ N(0, 1), p ~ U(0, 1).
TAIL_SWEEP_H = (3584, 3072, 1000)
TAIL_SWEEP_R = (1, 37, 65537, 524288)


def tail_sweep(R: int, H: int, seed: int = 4) -> Workload:
    return Workload(f"tail_sweep_r{R}_h{H}", R, H, "normal", 4.0, 1.0, "uniform", "token", seed)


def custom(R: int, H: int, seed: int, x_std: float = 3.0, g_std: float = 1.0, p_kind: str = "uniform") -> Workload:
    return Workload(f"custom_r{R}_h{H}", R, H, "normal", x_std, g_std, p_kind, "token", seed)


def get(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    raise KeyError(name)


def router_rows(tokens: int, seed: int, order: str = "token"):
    """Router weights for ``tokens × 16`` routed rows.

    Per token: 896 N(0,1) router scores, keep the top 16 (ties: lower index,
    as ``torch.topk``), softmax over the kept scores. Returns
    ``(p [R] fp32, expert_id [R] int64, token_id [R] int64)`` in row order:
    token-major (row = 16·t + k, k in descending-score order), or, for
    ``order == "expert"``, stably sorted by expert id (ties by token, then k).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(1_000_003 * (seed + 1))
    p_rows, e_rows = [], []
    step = 8192
    for t0 in range(0, tokens, step):
        t1 = min(tokens, t0 + step)
        scores = torch.randn((t1 - t0, N_EXPERTS), generator=gen, dtype=torch.float32)
        top_vals, top_idx = torch.topk(scores, k=TOP_K, dim=-1)
        gates = torch.softmax(top_vals, dim=-1)
        p_rows.append(gates.reshape(-1))
        e_rows.append(top_idx.reshape(-1))
    p = torch.cat(p_rows) if p_rows else torch.empty(0, dtype=torch.float32)
    e = torch.cat(e_rows) if e_rows else torch.empty(0, dtype=torch.int64)
    tok = torch.arange(tokens, dtype=torch.int64).repeat_interleave(TOP_K)
    if order == "expert":
        perm = torch.sort(e, stable=True).indices
        p, e, tok = p[perm], e[perm], tok[perm]
    return p.contiguous(), e.contiguous(), tok.contiguous()


def _fill_x(dst: torch.Tensor, w: Workload, gen: torch.Generator, chunk_rows: int):
    R, H2 = dst.shape
    dev = dst.device
    for r0 in range(0, R, chunk_rows):
        r1 = min(R, r0 + chunk_rows)
        n = r1 - r0
        vals = torch.randn((n, H2), generator=gen, device=dev, dtype=torch.float32).mul_(w.x_std)
        if w.x_kind == "mixture":
            # 89 % N(0, σ²), 10 % U[-80, 80], 0.5 % exact +0, 0.5 % exact -0
            sel = torch.rand((n, H2), generator=gen, device=dev, dtype=torch.float32)
            uni = torch.rand((n, H2), generator=gen, device=dev, dtype=torch.float32).mul_(160.0).sub_(80.0)
            vals = torch.where(sel < 0.10, uni, vals)
            vals = torch.where((sel >= 0.10) & (sel < 0.105), torch.zeros((), device=dev), vals)
            vals = torch.where((sel >= 0.105) & (sel < 0.11), torch.full((), -0.0, device=dev), vals)
            del sel, uni
        dst[r0:r1].copy_(vals.to(torch.bfloat16))
        del vals


def _fill_normal(dst: torch.Tensor, std: float, gen: torch.Generator, chunk_rows: int):
    R = dst.shape[0]
    for r0 in range(0, R, chunk_rows):
        r1 = min(R, r0 + chunk_rows)
        vals = torch.randn((r1 - r0,) + tuple(dst.shape[1:]), generator=gen, device=dst.device,
                           dtype=torch.float32).mul_(std)
        dst[r0:r1].copy_(vals.to(dst.dtype))
        del vals


def generate(w: Workload, device="cpu", need_g: bool = True, chunk_rows: int = 32768):
    """Draw ``(x bf16 [R,2H], g bf16 [R,H] or None, p fp32 [R])`` on ``device``."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    x = torch.empty((w.R, 2 * w.H), dtype=torch.bfloat16, device=device)
    _fill_x(x, w, gen, chunk_rows)
    g = None
    if need_g:
        g = torch.empty((w.R, w.H), dtype=torch.bfloat16, device=device)
        _fill_normal(g, w.g_std, gen, chunk_rows)
    if w.p_kind == "router":
        assert w.R % TOP_K == 0, "router rows come in groups of 16 per token"
        p, _, _ = router_rows(w.tokens, w.seed, w.order)
        p = p.to(device)
    else:
        p = torch.rand((w.R,), generator=gen, device=device, dtype=torch.float32)
    return x, g, p

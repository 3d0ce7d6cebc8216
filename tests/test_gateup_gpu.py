"""Parity of the fused gate/up projection (tcgen05 grouped GEMM + SiTU-GLU forward) with the
oracle: x = [W_gate,e·h | W_up,e·h] in fp64 (numpy matmul), rounded to bf16 by the oracle's
round-to-nearest-even, and out = G·L in fp64 on those bf16 values.

x is a rounded fp32 accumulation. An fp32 sum of D products differs from the exact sum by a
small multiple of 2^-24·Σ_d|h_d·w_d|, so where the exact value lies that close to a midpoint
between two bf16 values either neighbour is a correct rounding. The test therefore requires
x_gpu = RNE(x_exact + δ) for some |δ| <= 2^-20·Σ_d|h_d·w_d| (rounding is monotone, so that is
every bf16 value in the closed range [RNE(x_exact - ε), RNE(x_exact + ε)], several values wide
where |x| is small next to Σ|h·w|; the margin is 16x the random-walk size of an fp32 sum of 3584
terms) and counts how often it differs from RNE(x_exact). Several results being correct there,
out is compared, with the bf16 tolerance, to the oracle's forward at the admissible x the
kernel chose."""
import numpy as np
import pytest
import torch

import oracle
import situ_inputs as si
from _parity import Parity, bf16_bits_to_f64, bits_of, for_expert_groups_parallel

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ACC_EPS = 2.0 ** -20


@pytest.fixture(scope="module")
def sg(cuda_lib):
    assert torch.cuda.is_available()
    return cuda_lib


def make(counts, H, D, seed, x_std=3.0, device="cpu"):
    """h ~ N(0, 1) and weights ~ N(0, x_std²/D), so each projection is ~ N(0, x_std²)."""
    gen = torch.Generator(device=device).manual_seed(seed)
    E = len(counts)
    R = int(sum(counts))
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int64)
    h = torch.randn(R, D, generator=gen, device=device).to(torch.bfloat16)
    w = torch.empty(E, 2 * H, D, dtype=torch.bfloat16, device=device)
    for e in range(E):
        w[e] = (torch.randn(2 * H, D, generator=gen, device=device) * (x_std / D ** 0.5)).to(torch.bfloat16)
    return h, w, off


def run(sg, h, w, off, beta=4.0, lbeta=25.0):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    x, out = sg.situ_glu_fwd_gateup(h.to(DEV), w.to(DEV), off.to(DEV), status=status, beta=beta, lbeta=lbeta)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return x, out


def check(name, x_gpu_bits, out_gpu_bits, x_exact, xb_ref, mag, beta=4.0, lbeta=25.0):
    """x: an admissible rounding of the exact projection; out: the oracle's forward at it."""
    lo = bf16_bits_to_f64(oracle.round_bf16_array(x_exact - ACC_EPS * mag))
    hi = bf16_bits_to_f64(oracle.round_bf16_array(x_exact + ACC_EPS * mag))
    xg = bf16_bits_to_f64(x_gpu_bits)
    admissible = (lo <= xg) & (xg <= hi)
    n_bad = int((~admissible).sum())
    if n_bad:
        idx = np.argwhere(~admissible)[:5]
        ex = [(tuple(int(k) for k in i), float(xg[tuple(i)]), float(x_exact[tuple(i)]), float(lo[tuple(i)]),
               float(hi[tuple(i)])) for i in idx]
        raise AssertionError(f"{name}: {n_bad} x elements are no rounding of the exact projection: {ex}")
    differs = int((x_gpu_bits != xb_ref).sum())
    assert differs <= max(8, x_gpu_bits.size // 200), f"{name}: {differs} x elements differ from RNE(exact)"
    # every bf16 value in [lo, hi] is a correct x; the forward is checked at the one the kernel chose
    out_ref = oracle.fwd_bf16(np.ascontiguousarray(x_gpu_bits), beta, lbeta)
    par = Parity(name)
    par.bf16("out", out_gpu_bits, out_ref)
    par.assert_ok()
    return differs


CASES = {
    "one_tile": ([128], 128, 64),
    "partial_tiles": ([100, 60], 256, 128),
    "empty_experts": ([0, 300, 1, 129, 0, 77, 0], 384, 192),
    "real_widths": ([200, 0, 317, 128, 90, 250, 33, 400, 1, 255, 256, 129], 3072, 3584),
    # H / 128 N-tiles shared by min(8, H / 128) CTAs: 10 over 8 (uneven)
    "uneven_split": ([300, 77], 1280, 128),
    # >= 512 rows per expert on average: work units of two M-tiles sharing each weight stage,
    # with odd tile counts (9 and 5: a last unit of one tile), an empty expert and partial tiles
    "two_tile_units": ([1100, 600, 0, 900], 256, 128),
    "two_tile_units_real_widths": ([700, 1300], 3072, 3584),
    # either side of the host's choice (experts averaging 512 rows or more: two-tile units)
    "unit_choice_511": ([510, 512], 256, 64),
    "unit_choice_512": ([512, 512], 256, 64),
    # shapes off the 128-column-pair N-tile and 64-deep K-block grid (H % 16 == 0, D % 8 == 0): the
    # weight rows past H and the K columns past D read as zeros, chunks past H are not stored
    "n_tail_h144": ([100, 60, 0], 144, 64),
    "k_tail_d200": ([200, 0, 129], 256, 200),
    "smallest_h16_d8": ([40, 1], 16, 8),
    "both_tails_h1040_d72": ([300, 292], 1040, 72),
    "both_tails_two_tile_units": ([600, 700], 400, 136),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_gateup_all_rows(sg, name):
    counts, H, D = CASES[name]
    h, w, off = make(counts, H, D, seed=len(name))
    x, out = run(sg, h, w, off)
    x_exact, xb_ref, _, mag = oracle.gateup_fwd(bits_of(h), bits_of(w).reshape(w.shape), off.numpy())
    check("gateup " + name, bits_of(x), bits_of(out), x_exact, xb_ref, mag)


@pytest.mark.parametrize("beta,lbeta", [(2.0, 100.0), (4.0, 100.0)])
def test_gateup_general_scales(sg, beta, lbeta):
    counts, H, D = [70, 200], 256, 128
    h, w, off = make(counts, H, D, seed=3)
    x, out = run(sg, h, w, off, beta, lbeta)
    x_exact, xb_ref, _, mag = oracle.gateup_fwd(bits_of(h), bits_of(w).reshape(w.shape), off.numpy(), beta, lbeta)
    check(f"gateup beta={beta} lbeta={lbeta}", bits_of(x), bits_of(out), x_exact, xb_ref, mag, beta, lbeta)


def test_gateup_saturating_inputs(sg):
    """Projections far into both tails (|x| up to ~80): G -> 4 or -0, L -> +-25."""
    counts, H, D = [256], 128, 64
    h, w, off = make(counts, H, D, seed=9, x_std=30.0)
    x, out = run(sg, h, w, off)
    x_exact, xb_ref, _, mag = oracle.gateup_fwd(bits_of(h), bits_of(w).reshape(w.shape), off.numpy())
    assert float(np.abs(x_exact).max()) > 60.0
    check("gateup saturating", bits_of(x), bits_of(out), x_exact, xb_ref, mag)


def test_gateup_matches_unfused_path(sg):
    """out of the fused kernel equals situ_glu_fwd applied to the x it wrote, bit for bit: the
    same forward on the same bf16 values, only without the round trip of x through memory."""
    counts, H, D = [130, 0, 250], 512, 256
    h, w, off = make(counts, H, D, seed=4)
    x, out = run(sg, h, w, off)
    out2 = sg.situ_glu_fwd(x)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_gateup_rejects_unsupported_shapes(sg):
    h, w, off = make([64], 128, 64, seed=1)
    with pytest.raises(sg.SituGluError):                  # H = 100 is not a multiple of 16
        sg.situ_glu_fwd_gateup(h.to(DEV), w.to(DEV)[:, :200].contiguous(), off.to(DEV))
    with pytest.raises(sg.SituGluError):                  # D = 60 is not a multiple of 8
        sg.situ_glu_fwd_gateup(h.to(DEV)[:, :60].contiguous(), w.to(DEV)[:, :, :60].contiguous(), off.to(DEV))


@pytest.mark.slow
def test_gateup_expert_grouped_full_size_all_rows(sg):
    """R = 262144 routed rows grouped by expert over 896 experts (16384 tokens x top-16),
    H = 3072, D = 3584: the full-size launch, every row of x and out checked (runs of
    consecutive experts streamed to the host, the fp64 projections on each run, several runs at
    once)."""
    wl = si.get("expert_grouped_r262144_h3072")
    _, experts, _ = si.router_rows(wl.tokens, wl.seed, order="expert")
    counts = np.bincount(experts.numpy(), minlength=si.N_EXPERTS)
    H, D, E = wl.H, 3584, si.N_EXPERTS
    gen = torch.Generator(device=DEV).manual_seed(6)
    h = torch.empty(wl.R, D, dtype=torch.bfloat16, device=DEV)
    for a in range(0, wl.R, 32768):
        h[a:a + 32768] = torch.randn(min(32768, wl.R - a), D, generator=gen, device=DEV).to(torch.bfloat16)
    w = torch.empty(E, 2 * H, D, dtype=torch.bfloat16, device=DEV)
    for e in range(E):
        w[e] = (torch.randn(2 * H, D, generator=gen, device=DEV) * (wl.x_std / D ** 0.5)).to(torch.bfloat16)
    off_np = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    off = torch.from_numpy(off_np).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    x, out = sg.situ_glu_fwd_gateup(h, w, off, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    def run_group(part, e0, e1, nthreads):
        r0, r1 = int(off_np[e0]), int(off_np[e1])
        if r1 == r0:
            return 0, 0
        x_exact, xb_ref, _, mag = oracle.gateup_fwd(bits_of(h[r0:r1]), bits_of(w[e0:e1]).reshape(e1 - e0, 2 * H, D),
                                                    off_np[e0:e1 + 1] - r0, nthreads=nthreads)
        xg = bits_of(x[r0:r1])
        differs = check(f"gateup expert_grouped_r262144 experts {e0}..{e1 - 1}", xg, bits_of(out[r0:r1]), x_exact,
                        xb_ref, mag)
        return differs, xg.size

    par = Parity("gateup expert_grouped_r262144 (all rows)")
    res = for_expert_groups_parallel(par, off_np, run_group, rows_per_group=2048)
    differs, n = sum(r[0] for r in res), sum(r[1] for r in res)
    assert n == wl.R * 2 * H
    assert differs <= max(8, n // 200)
    print(f"gateup expert_grouped_r262144: every row checked, {n} x elements, {differs} differ from RNE(exact)")
    del h, w, x, out
    torch.cuda.empty_cache()


def test_gateup_max_experts_mostly_empty(sg):
    """1024 experts, 600 rows over 37 of them, on a non-default stream."""
    rng = np.random.default_rng(9)
    counts = np.zeros(1024, dtype=np.int64)
    used = rng.choice(1024, 37, replace=False)
    counts[used] = rng.multinomial(600, np.ones(37) / 37)
    h, w, off = make(counts.tolist(), 128, 64, seed=23)
    s = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    with torch.cuda.stream(s):
        x, out = sg.situ_glu_fwd_gateup(h.to(DEV), w.to(DEV), off.to(DEV), status=status, stream=s)
    s.synchronize()
    assert int(status.item()) == 0
    x_exact, xb_ref, _, mag = oracle.gateup_fwd(bits_of(h), bits_of(w).reshape(w.shape), off.numpy())
    check("gateup 1024 experts", bits_of(x), bits_of(out), x_exact, xb_ref, mag)


def test_gateup_single_row(sg):
    h, w, off = make([0, 0, 1], 256, 64, seed=24)
    x, out = run(sg, h, w, off)
    x_exact, xb_ref, _, mag = oracle.gateup_fwd(bits_of(h), bits_of(w).reshape(w.shape), off.numpy())
    check("gateup single row", bits_of(x), bits_of(out), x_exact, xb_ref, mag)


@pytest.mark.slow
def test_gateup_large_experts_full_size_sampled(sg):
    """32 experts x 8192 rows (H = 3072, D = 3584): the two-M-tile form at full size, sampled rows
    of the first, a middle and the last expert plus their tile and unit boundaries."""
    E, per, H, D = 32, 8192, 3072, 3584
    counts = [per] * E
    gen = torch.Generator(device=DEV).manual_seed(7)
    R = E * per
    h = torch.empty(R, D, dtype=torch.bfloat16, device=DEV)
    for a in range(0, R, 32768):
        h[a:a + 32768] = torch.randn(min(32768, R - a), D, generator=gen, device=DEV).to(torch.bfloat16)
    w = torch.empty(E, 2 * H, D, dtype=torch.bfloat16, device=DEV)
    for e in range(E):
        w[e] = (torch.randn(2 * H, D, generator=gen, device=DEV) * (3.0 / D ** 0.5)).to(torch.bfloat16)
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    x, out = sg.situ_glu_fwd_gateup(h, w, off, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(13)
    for e in (0, 17, 31):
        local = np.unique(np.concatenate([rng.integers(0, per, 48), [0, 127, 128, 255, 256, 383, per - 1]]))
        rows = torch.from_numpy(e * per + local).to(DEV)
        x_exact, xb_ref, _, mag = oracle.gateup_fwd(bits_of(h.index_select(0, rows)), bits_of(w[e]).reshape(1, 2 * H, D),
                                                    np.array([0, len(local)], dtype=np.int64))
        check(f"gateup 32x8192 expert {e}", bits_of(x.index_select(0, rows)), bits_of(out.index_select(0, rows)),
              x_exact, xb_ref, mag)
    del h, w, x, out
    torch.cuda.empty_cache()

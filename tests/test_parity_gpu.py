"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on a GPU.

Every input is seeded and synthetic (situ_inputs); the very same tensors are fed
to both sides. Every workload is compared element by element over all rows, the pages' scale
(R = 1.6M, the benchmark's own launch) and the largest tail-sweep shapes
included (rows streamed to the host in blocks, several blocks at once); only
the FP8 pair at R = 1.6M is checked on sampled rows.
"""
import numpy as np
import pytest
import torch

import situ_inputs as si
from _parity import Parity, bits_of, compare_full, compare_full_parallel, for_blocks_parallel

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sg(cuda_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return cuda_lib


def run(sg, x, g, p, beta=4.0, lbeta=25.0):
    out = sg.situ_glu_fwd(x, beta=beta, lbeta=lbeta)
    dx, dp = sg.situ_glu_bwd_router(x, g, p, beta=beta, lbeta=lbeta)
    torch.cuda.synchronize()
    return out, dx, dp


def on_device(w, gen_on_device=False):
    if gen_on_device:
        return si.generate(w, device=DEV)
    return tuple(t.to(DEV) for t in si.generate(w, device="cpu"))


def free(*ts):
    del ts
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- the workloads

@pytest.mark.parametrize("name", ["routed_r1024_h3072", "saturating_mix_r16384_h3072"])
def test_workload_all_rows(sg, name):
    w = si.get(name)
    x, g, p = on_device(w)
    out, dx, dp = run(sg, x, g, p)
    par = Parity(name)
    compare_full(par, x, g, p, out, dx, dp)
    par.assert_ok()


@pytest.mark.slow
def test_expert_grouped_all_rows(sg):
    w = si.get("expert_grouped_r262144_h3072")
    x, g, p = on_device(w, gen_on_device=True)
    out, dx, dp = run(sg, x, g, p)
    par = Parity(w.name)
    compare_full_parallel(par, x, g, p, out, dx, dp)
    par.assert_ok()
    free(x, g, p, out, dx, dp)


@pytest.mark.slow
def test_pages_scale_full_launch_all_rows(sg):
    """R = 1.6M, H = 3072 (x alone 19.66 GB): the benchmark's launch, every element of out, dx
    and dp compared with the oracle (rows streamed to the host in blocks)."""
    w = si.get("pages_scale_r1600000_h3072")
    x, g, p = on_device(w, gen_on_device=True)
    out, dx, dp = run(sg, x, g, p)
    assert float(out.abs().max()) <= 100.0          # |out| <= beta·lambda at every element
    par = Parity(w.name)
    compare_full_parallel(par, x, g, p, out, dx, dp)
    par.assert_ok()
    free(x, g, p, out, dx, dp)


@pytest.mark.parametrize("H", si.TAIL_SWEEP_H)
@pytest.mark.parametrize("R", [1, 37, 65537])
def test_tail_sweep_all_rows(sg, R, H):
    w = si.tail_sweep(R, H)
    x, g, p = on_device(w)
    out, dx, dp = run(sg, x, g, p)
    par = Parity(w.name)
    compare_full(par, x, g, p, out, dx, dp)
    par.assert_ok()


@pytest.mark.slow
@pytest.mark.parametrize("H", si.TAIL_SWEEP_H)
def test_tail_sweep_largest_all_rows(sg, H):
    w = si.tail_sweep(524288, H)
    x, g, p = on_device(w, gen_on_device=True)
    out, dx, dp = run(sg, x, g, p)
    par = Parity(w.name)
    compare_full_parallel(par, x, g, p, out, dx, dp)
    par.assert_ok()
    free(x, g, p, out, dx, dp)


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("beta,lbeta", [(4.0, 25.0), (2.5, 7.0)])
@pytest.mark.parametrize("H", [1, 2, 7, 8, 9, 16, 999, 1000, 1016])
def test_odd_widths(sg, H, beta, lbeta):
    w = si.custom(37, H, seed=H, x_std=4.0)
    x, g, p = on_device(w)
    out, dx, dp = run(sg, x, g, p, beta, lbeta)
    par = Parity(f"H={H} beta={beta} lbeta={lbeta}")
    compare_full(par, x, g, p, out, dx, dp, beta, lbeta)
    par.assert_ok()


@pytest.mark.parametrize("beta,lbeta", [(4.0, 25.0), (1.0, 1.0), (0.5, 3.0), (4.0, 100.0), (8.0, 64.0),
                                        (1e6, 1e6), (4.0, 1e6)])
def test_other_scales(sg, beta, lbeta):
    """Fast (beta = 4, lbeta <= 64) and general kernels, including the SwiGLU-like limit."""
    w = si.custom(64, 1024, seed=7, x_std=3.0)
    x, g, p = on_device(w)
    out, dx, dp = run(sg, x, g, p, beta, lbeta)
    par = Parity(f"beta={beta} lbeta={lbeta}")
    compare_full(par, x, g, p, out, dx, dp, beta, lbeta)
    par.assert_ok()


@pytest.mark.parametrize("H", [3072, 1000, 8])
def test_misaligned_bases_take_the_element_path(sg, H):
    R = 21
    w = si.custom(R, H, seed=5)
    x0, g0, p0 = on_device(w)
    # views whose base addresses are 2 bytes past a 16-byte boundary
    xb = torch.empty(R * 2 * H + 8, dtype=torch.bfloat16, device=DEV)
    gb = torch.empty(R * H + 8, dtype=torch.bfloat16, device=DEV)
    ob = torch.empty(R * H + 8, dtype=torch.bfloat16, device=DEV)
    db = torch.empty(R * 2 * H + 8, dtype=torch.bfloat16, device=DEV)
    x = xb[1:1 + R * 2 * H].view(R, 2 * H)
    g = gb[1:1 + R * H].view(R, H)
    out = ob[1:1 + R * H].view(R, H)
    dx = db[1:1 + R * 2 * H].view(R, 2 * H)
    assert x.data_ptr() % 16 == 2
    x.copy_(x0)
    g.copy_(g0)
    dp = torch.empty(R, dtype=torch.float32, device=DEV)
    sg.situ_glu_fwd(x, out)
    sg.situ_glu_bwd_router(x, g, p0, dx, dp)
    torch.cuda.synchronize()
    par = Parity(f"misaligned H={H}")
    compare_full(par, x, g, p0, out, dx, dp)
    par.assert_ok()
    # the aligned vector path gives the same bits elementwise; dp is summed in another order
    # (per lane: strided elements here, 8-element chunks there), so it agrees to fp32 rounding
    out2, dx2, dp2 = run(sg, x0, g0, p0)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(dx.view(torch.int16), dx2.view(torch.int16))
    torch.testing.assert_close(dp, dp2, rtol=1e-5, atol=1e-4)


def test_extreme_and_nonfinite_inputs(sg):
    H = 16
    big = 3.3895313892515355e38  # largest finite bf16
    vals = [0.0, -0.0, 1e-30, -1e-30, 1e-3, -1e-3, 80.0, -80.0, 500.0, -500.0, big, -big,
            float("inf"), float("-inf"), 3.0, -3.0]
    gate = torch.tensor(vals, dtype=torch.float32)
    rows = []
    for k in range(H):
        lin = torch.roll(gate, k)
        rows.append(torch.cat([gate, lin]))
    x = torch.stack(rows).to(torch.bfloat16).to(DEV)
    R = x.shape[0]
    g = torch.linspace(-2, 2, R * H).reshape(R, H).to(torch.bfloat16).to(DEV)
    p = torch.linspace(0.1, 1.0, R).to(DEV)
    out, dx, dp = run(sg, x, g, p)
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(dx).all()) and bool(torch.isfinite(dp).all())
    par = Parity("extreme")
    compare_full(par, x, g, p, out, dx, dp)
    par.assert_ok()
    # NaN propagates to the outputs of its own element (and to dp of its row)
    xn = x.clone()
    xn[3, 5] = float("nan")
    outn, dxn, dpn = run(sg, xn, g, p)
    assert bool(torch.isnan(outn[3, 5])) and bool(torch.isnan(dxn[3, 5])) and bool(torch.isnan(dpn[3]))
    mask = torch.ones_like(outn, dtype=torch.bool)
    mask[3, 5] = False
    assert torch.equal(outn[mask].view(torch.int16), out[mask].view(torch.int16))


def test_zero_and_saturated_rows(sg):
    """Closed forms through the GPU: G(0) = L(0) = 0, G'(0) = 1/2, L'(0) = 1, G(+inf) = 4,
    L(-inf) = -25, G(-inf) = G'(+-inf) = L'(+-inf) = 0 (|x| = 1024 saturates every exponential)."""
    H = 3072
    x = torch.zeros(4, 2 * H, dtype=torch.bfloat16, device=DEV)
    x[1, :H] = 1024.0         # gate saturated high, linear zero
    x[2, H:] = -1024.0        # gate zero, linear saturated low
    x[3, :H] = -1024.0        # both saturated
    x[3, H:] = 1024.0
    g = torch.ones(4, H, dtype=torch.bfloat16, device=DEV)
    p = torch.full((4,), 0.5, device=DEV)
    out, dx, dp = run(sg, x, g, p)
    assert torch.all(out == 0) and torch.all(dp == 0)
    assert torch.all(dx[0] == 0) and torch.all(dx[3] == 0)
    assert torch.all(dx[1, :H] == 0) and torch.all(dx[1, H:] == 2.0)      # p·g·G(+inf)·L'(0) = 0.5·4·1
    assert torch.all(dx[2, :H] == -6.25) and torch.all(dx[2, H:] == 0)    # p·g·L(-inf)·G'(0) = 0.5·(-25)·0.5
    par = Parity("zero/saturated rows")
    compare_full(par, x, g, p, out, dx, dp)
    par.assert_ok()


def test_empty_is_a_noop(sg):
    x = torch.empty(0, 6144, dtype=torch.bfloat16, device=DEV)
    g = torch.empty(0, 3072, dtype=torch.bfloat16, device=DEV)
    p = torch.empty(0, dtype=torch.float32, device=DEV)
    out, dx, dp = run(sg, x, g, p)
    assert out.shape == (0, 3072) and dx.shape == (0, 6144) and dp.shape == (0,)


# ---------------------------------------------------------------- behaviour of the boundary

def test_in_place_backward_matches_out_of_place(sg):
    w = si.custom(300, 3072, seed=11)
    x, g, p = on_device(w)
    _, dx_ref, dp_ref = run(sg, x, g, p)
    xi = x.clone()
    dx_i, dp_i = sg.situ_glu_bwd_router(xi, g, p, dx=xi)
    torch.cuda.synchronize()
    assert dx_i.data_ptr() == xi.data_ptr()
    assert torch.equal(dx_i.view(torch.int16), dx_ref.view(torch.int16))
    assert torch.equal(dp_i, dp_ref)
    # element path in place as well
    w2 = si.custom(30, 999, seed=12)
    x2, g2, p2 = on_device(w2)
    _, dxr, dpr = run(sg, x2, g2, p2)
    x2i = x2.clone()
    sg.situ_glu_bwd_router(x2i, g2, p2, dx=x2i)
    torch.cuda.synchronize()
    assert torch.equal(x2i.view(torch.int16), dxr.view(torch.int16))


@pytest.mark.parametrize("R,H", [(37, 3072), (5, 1000), (3, 999)])
def test_guard_bands_untouched(sg, R, H):
    """Outputs sit inside larger buffers filled with a NaN pattern; nothing outside them changes."""
    pad = 64
    w = si.custom(R, H, seed=2)
    x, g, p = on_device(w)
    poison = torch.tensor(0x7FC1, dtype=torch.int16)
    ob = torch.full((R * H + 2 * pad,), int(poison), dtype=torch.int16, device=DEV)
    db = torch.full((R * 2 * H + 2 * pad,), int(poison), dtype=torch.int16, device=DEV)
    pb = torch.full((R + 2 * pad,), float("nan"), dtype=torch.float32, device=DEV)
    out = ob[pad:pad + R * H].view(torch.bfloat16).view(R, H)
    dx = db[pad:pad + R * 2 * H].view(torch.bfloat16).view(R, 2 * H)
    dp = pb[pad:pad + R]
    sg.situ_glu_fwd(x, out)
    sg.situ_glu_bwd_router(x, g, p, dx, dp)
    torch.cuda.synchronize()
    for buf, n in ((ob, R * H), (db, R * 2 * H)):
        assert bool((buf[:pad] == poison).all()) and bool((buf[pad + n:] == poison).all())
    assert bool(torch.isnan(pb[:pad]).all()) and bool(torch.isnan(pb[pad + R:]).all())
    par = Parity(f"guarded R={R} H={H}")
    compare_full(par, x, g, p, out, dx, dp)
    par.assert_ok()


def test_bitwise_reproducible(sg):
    w = si.custom(2048, 3072, seed=21)
    x, g, p = on_device(w)
    a = run(sg, x, g, p)
    b = run(sg, x, g, p)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
    assert torch.equal(a[2], b[2])


def test_library_allocates_no_device_memory(sg):
    w = si.custom(4096, 3072, seed=8)
    x, g, p = on_device(w)
    out = torch.empty(4096, 3072, dtype=torch.bfloat16, device=DEV)
    dx = torch.empty_like(x)
    dp = torch.empty(4096, dtype=torch.float32, device=DEV)
    sg.situ_glu_fwd(x, out)
    sg.situ_glu_bwd_router(x, g, p, dx, dp)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        sg.situ_glu_fwd(x, out)
        sg.situ_glu_bwd_router(x, g, p, dx, dp)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before


def test_runs_on_the_given_stream(sg):
    w = si.custom(512, 3072, seed=4)
    x, g, p = on_device(w)
    ref = run(sg, x, g, p)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = sg.situ_glu_fwd(x)
        dx, dp = sg.situ_glu_bwd_router(x, g, p)
    s.synchronize()
    assert torch.equal(out.view(torch.int16), ref[0].view(torch.int16))
    assert torch.equal(dx.view(torch.int16), ref[1].view(torch.int16))
    assert torch.equal(dp, ref[2])


def test_binding_rejects_bad_tensors(sg):
    x = torch.zeros(4, 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(TypeError):
        sg.situ_glu_fwd(x.float())
    with pytest.raises(ValueError):
        sg.situ_glu_fwd(x[:, ::2])
    with pytest.raises(sg.SituGluError) as ei:
        sg.situ_glu_fwd(x, beta=-1.0)
    assert ei.value.status == 1
    # a partial overlap of dx with x is rejected before any launch
    big = torch.zeros(8, 16, dtype=torch.bfloat16, device=DEV)
    xo = big[0:4]
    dxo = big[2:6]
    with pytest.raises(sg.SituGluError) as ei:
        sg.situ_glu_bwd_router(xo, torch.zeros(4, 8, dtype=torch.bfloat16, device=DEV),
                               torch.zeros(4, device=DEV), dx=dxo)
    assert ei.value.status == 2


# ---------------------------------------------------------------- block-wise FP8 saved x

import oracle  # noqa: E402
from _parity import compare_rows  # noqa: E402


def run_fp8(sg, x, g, p, beta=4.0, lbeta=25.0):
    out, xq, xs = sg.situ_glu_fwd_save_fp8(x, beta=beta, lbeta=lbeta)
    dx, dp = sg.situ_glu_bwd_router_fp8(xq, xs, g, p, beta=beta, lbeta=lbeta)
    torch.cuda.synchronize()
    return out, xq, xs, dx, dp


def check_fp8_rows(par, x, g, p, out, xq, xs, dx, dp, beta=4.0, lbeta=25.0, row0=0, nthreads=0):
    """Codes and scales bit-exact against the oracle's quantiser; out against the oracle's
    forward; dx and dp against the oracle's backward at the dequantised x."""
    xb = bits_of(x)
    q_ref, s_ref = oracle.quantize_fp8(xb)
    q_gpu = xq.detach().cpu().numpy()
    s_gpu = xs.detach().cpu().numpy()
    nq = int((q_gpu != q_ref).sum())
    ns = int((s_gpu.view(np.uint32) != s_ref.view(np.uint32)).sum())
    assert nq == 0, f"{par.name}: {nq} FP8 codes differ from the oracle, rows from {row0}"
    assert ns == 0, f"{par.name}: {ns} FP8 scales differ from the oracle, rows from {row0}"
    par.bf16("out", bits_of(out), oracle.fwd_bf16(xb, beta, lbeta, nthreads), row0)
    dx_ref, dp_ref, dpa = oracle.bwd_router_fp8(q_ref, s_ref, bits_of(g), p.detach().cpu().numpy(), beta, lbeta,
                                                nthreads)
    par.bf16("dx", bits_of(dx), dx_ref, row0)
    par.dp(dp.detach().cpu().numpy(), dp_ref, dpa, row0)


def check_fp8_full(par, x, g, p, out, xq, xs, dx, dp, beta=4.0, lbeta=25.0, chunk_rows=8192, workers=4):
    def check(part, a, b, nthreads):
        check_fp8_rows(part, x[a:b], g[a:b], p[a:b], out[a:b], xq[a:b], xs[a:b], dx[a:b], dp[a:b], beta, lbeta, a,
                       nthreads)

    for_blocks_parallel(par, x.shape[0], check, chunk_rows, workers)


@pytest.mark.parametrize("name", ["routed_r1024_h3072", "saturating_mix_r16384_h3072"])
def test_fp8_workload_all_rows(sg, name):
    w = si.get(name)
    x, g, p = on_device(w)
    out, xq, xs, dx, dp = run_fp8(sg, x, g, p)
    par = Parity("fp8 " + name)
    check_fp8_full(par, x, g, p, out, xq, xs, dx, dp)
    par.assert_ok()
    # the forward output is exactly the bf16-saved forward's
    assert torch.equal(out.view(torch.int16), sg.situ_glu_fwd(x).view(torch.int16))


@pytest.mark.parametrize("H", si.TAIL_SWEEP_H)
@pytest.mark.parametrize("R", [1, 37, 65537])
def test_fp8_tail_sweep_all_rows(sg, R, H):
    w = si.tail_sweep(R, H)
    x, g, p = on_device(w)
    out, xq, xs, dx, dp = run_fp8(sg, x, g, p)
    par = Parity("fp8 " + w.name)
    check_fp8_full(par, x, g, p, out, xq, xs, dx, dp)
    par.assert_ok()


@pytest.mark.slow
def test_fp8_pages_scale_full_launch_all_rows(sg):
    """R = 1.6M, H = 3072 through the FP8-saved pair, the benchmark's launch: on every row the
    codes and scales are bit-exact against the oracle's quantiser and out, dx and dp are within
    tolerance (rows streamed to the host in blocks, one block per host core at once: the
    oracle's quantiser runs single-threaded per block)."""
    w = si.get("pages_scale_r1600000_h3072")
    x, g, p = on_device(w, gen_on_device=True)
    out, xq, xs, dx, dp = run_fp8(sg, x, g, p)
    par = Parity(w.name + " fp8 (all rows)")
    check_fp8_full(par, x, g, p, out, xq, xs, dx, dp, chunk_rows=8192, workers=oracle.default_threads())
    assert par.t["dx"].n == w.R * 2 * w.H and par.t["dp"].n == w.R and par.t["out"].n == w.R * w.H
    par.assert_ok()
    free(x, g, p, out, xq, xs, dx, dp)


@pytest.mark.parametrize("beta,lbeta", [(4.0, 25.0), (2.5, 7.0)])
@pytest.mark.parametrize("H", [1, 7, 8, 16, 128, 130, 136, 999])
def test_fp8_odd_widths(sg, H, beta, lbeta):
    w = si.custom(37, H, seed=100 + H, x_std=4.0)
    x, g, p = on_device(w)
    out, xq, xs, dx, dp = run_fp8(sg, x, g, p, beta, lbeta)
    par = Parity(f"fp8 H={H} beta={beta}")
    check_fp8_full(par, x, g, p, out, xq, xs, dx, dp, beta, lbeta)
    par.assert_ok()


def test_fp8_zero_tiny_and_huge_blocks(sg):
    H = 384
    x = torch.zeros(5, 2 * H, dtype=torch.float32)
    x[1] = torch.linspace(-1e-37, 1e-37, 2 * H)          # below the amax floor: scale 2^-126
    x[2] = torch.linspace(-1.0, 1.0, 2 * H) * 3e38       # near the bf16 maximum
    x[3, ::7] = 5.0                                       # sparse block contents
    x[4] = torch.randn(2 * H, generator=torch.Generator().manual_seed(1)) * 1e-3
    x = x.to(torch.bfloat16).to(DEV)
    g = torch.ones(5, H, dtype=torch.bfloat16, device=DEV)
    p = torch.full((5,), 0.25, device=DEV)
    out, xq, xs, dx, dp = run_fp8(sg, x, g, p)
    assert float(xs[0].min()) == float(xs[0].max()) == 2.0 ** -126 and int(xq[0].max()) == 0
    par = Parity("fp8 zero/tiny/huge")
    check_fp8_full(par, x, g, p, out, xq, xs, dx, dp)
    par.assert_ok()


def test_fp8_scale_for_every_amax_mantissa(sg):
    """Block maxima with each of the 128 bf16 mantissas at exponents from 2^-100 to 2^120 (and
    a zero block): the inverse scales and scales follow the block amax through a mantissa table
    and a power of two, so every code and scale must still equal the oracle's divisions."""
    H = 3072                                   # 24 blocks per half, 48 per row
    R = 128
    rng = np.random.default_rng(21)
    x = rng.uniform(-1.0, 1.0, (R, 2 * H)).astype(np.float32)
    nb = 2 * H // 128
    for r in range(R):
        for b in range(nb):
            f = (r + 37 * b) % 128
            e = int(rng.integers(-100, 121))
            amax = np.float32((1.0 + f / 128.0) * 2.0 ** e)     # exactly a bf16 value
            blk = x[r, b * 128:(b + 1) * 128] * np.float32(0.99) * amax
            blk[int(rng.integers(0, 128))] = amax if rng.random() < 0.5 else -amax
            x[r, b * 128:(b + 1) * 128] = blk
    x[0, :128] = 0.0                            # a zero block: the floor
    xt = torch.from_numpy(x).to(torch.bfloat16).to(DEV)
    g = torch.randn(R, H, generator=torch.Generator().manual_seed(22)).to(torch.bfloat16).to(DEV)
    p = torch.rand(R, generator=torch.Generator().manual_seed(23)).to(DEV)
    out, xq, xs, dx, dp = run_fp8(sg, xt, g, p)
    par = Parity("fp8 amax mantissa sweep")
    check_fp8_full(par, xt, g, p, out, xq, xs, dx, dp)
    par.assert_ok()


def test_fp8_misaligned_codes_take_the_element_path(sg):
    R, H = 9, 1000
    w = si.custom(R, H, seed=3)
    x, g, p = on_device(w)
    qb = torch.empty(R * 2 * H + 16, dtype=torch.uint8, device=DEV)
    xq = qb[1:1 + R * 2 * H].view(R, 2 * H)              # 1 byte past an 8-byte boundary
    out, xq, xs = sg.situ_glu_fwd_save_fp8(x, xq=xq)
    dx, dp = sg.situ_glu_bwd_router_fp8(xq, xs, g, p)
    torch.cuda.synchronize()
    par = Parity("fp8 misaligned codes")
    check_fp8_full(par, x, g, p, out, xq, xs, dx, dp)
    par.assert_ok()
    ref = run_fp8(sg, x, g, p)                            # aligned vector path: same codes and dx
    assert torch.equal(ref[1], xq) and torch.equal(ref[2], xs)
    assert torch.equal(ref[3].view(torch.int16), dx.view(torch.int16))


def test_fp8_guard_bands_untouched(sg):
    R, H, pad = 37, 1000, 64
    nb = sg.fp8_scale_blocks(H)
    w = si.custom(R, H, seed=6)
    x, g, p = on_device(w)
    qb = torch.full((R * 2 * H + 2 * pad,), 0xA5, dtype=torch.uint8, device=DEV)
    sb = torch.full((R * 2 * nb + 2 * pad,), float("nan"), dtype=torch.float32, device=DEV)
    xq = qb[pad:pad + R * 2 * H].view(R, 2 * H)
    xs = sb[pad:pad + R * 2 * nb].view(R, 2 * nb)
    out, _, _ = sg.situ_glu_fwd_save_fp8(x, xq=xq, xs=xs)
    dx, dp = sg.situ_glu_bwd_router_fp8(xq, xs, g, p)
    torch.cuda.synchronize()
    assert bool((qb[:pad] == 0xA5).all()) and bool((qb[pad + R * 2 * H:] == 0xA5).all())
    assert bool(torch.isnan(sb[:pad]).all()) and bool(torch.isnan(sb[pad + R * 2 * nb:]).all())
    par = Parity("fp8 guarded")
    check_fp8_full(par, x, g, p, out, xq, xs, dx, dp)
    par.assert_ok()


@pytest.mark.parametrize("scale", [1e-3, 3e-2, 1e-5])
def test_small_magnitude_rows(sg, scale):
    """Rows of small pre-activations: the backward's dp keeps its relative tolerance (the
    numerators 1 - e^{-y} are evaluated by a series for small y instead of as a difference)."""
    w = si.custom(512, 3072, seed=int(1 / scale) % 997, x_std=scale)
    x, g, p = on_device(w)
    out, dx, dp = run(sg, x, g, p)
    par = Parity(f"small magnitude x ~ N(0, {scale}^2)")
    compare_full(par, x, g, p, out, dx, dp)
    par.assert_ok()
    out8, xq, xs, dx8, dp8 = run_fp8(sg, x, g, p)
    par8 = Parity(f"fp8, small magnitude x ~ N(0, {scale}^2)")
    check_fp8_full(par8, x, g, p, out8, xq, xs, dx8, dp8)
    par8.assert_ok()


def test_situ_and_mul_autograd(sg):
    """The autograd operator: forward equals the oracle's, the gradient it passes back equals the
    oracle's backward at p = 1 with the incoming gradient as g, and it saves only x."""
    gen = torch.Generator().manual_seed(41)
    x = (torch.randn(300, 2 * 1024, generator=gen) * 3).to(torch.bfloat16).to(DEV).requires_grad_(True)
    g = torch.randn(300, 1024, generator=gen).to(torch.bfloat16).to(DEV)
    saved = []
    with torch.autograd.graph.saved_tensors_hooks(lambda t: saved.append(t) or t, lambda t: t):
        a = sg.situ_and_mul(x)
    a.backward(g)
    torch.cuda.synchronize()
    assert len(saved) == 1 and saved[0].data_ptr() == x.data_ptr()
    xb, gb = bits_of(x.detach()), bits_of(g)
    par = Parity("situ_and_mul autograd")
    par.bf16("out", bits_of(a.detach()), oracle.fwd_bf16(xb))
    dx_ref, _, _ = oracle.bwd_router_bf16(xb, gb, np.ones(300, dtype=np.float32))
    par.bf16("dx", bits_of(x.grad), dx_ref)
    par.assert_ok()

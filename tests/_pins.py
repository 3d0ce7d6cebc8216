"""Pins of the fp64 oracle against what the pages and the mathematics fix (shared bodies).

Each pin_* takes an oracle instance (the real one, or a deliberately broken copy in
tests/test_oracle_mutants.py) and raises AssertionError when the oracle disagrees.

Nothing here runs on a GPU. Each test is chosen so that a plausible mistake in
the oracle (a dropped term of G', a wrong sign in the overflow-safe sigmoid, a
swapped gate/linear half, p folded into dp, a transposed W_down) fails at least
one of them:

* closed forms at points where tanh and sigmoid are rational (tests/golden/closed_forms.txt);
* limits and symmetries of the definition;
* the SwiGLU limit (beta, lbeta -> infinity), a textbook special case;
* central finite differences of  Λ(x, p) = Σ_r p_r Σ_j g_rj a_rj(x)  for every dx and dp;
* a brute-force tiny expert  y = Σ_e p_e W_e a_e(x_e)  for the router-gradient rewrite;
* the definition run under PyTorch autograd in float64 (an independent derivative).

Definition: "Frontier-scale RL with Kimi K3", section "Streaming activations".
Router rewrite: "Kimi K3 模型结构（9）：显存", section "MoE 反向：推一下为什么可以不存 expert 输出".
"""
import math
import os

import numpy as np
import pytest
import torch


GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _eval(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"log": math.log}))


def closed_form_rows():
    rows = []
    with open(os.path.join(GOLDEN, "closed_forms.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, qty, u, v, beta, lbeta, expect = [t.strip() for t in line.split("|")]
            rows.append((name, qty, _eval(u), _eval(v), float(beta), float(lbeta), _eval(expect)))
    return rows


def pin_closed_forms(o):
    for row in closed_form_rows():
        _pin_closed_form_row(o, row)


def _pin_closed_form_row(o, row):
    name, qty, u, v, beta, lbeta, expect = row
    G, L, Gp, Lp = o.point(u, v, beta, lbeta)
    got = {"G": G, "L": L, "Gp": Gp, "Lp": Lp}[qty]
    assert abs(got - expect) <= 1e-13 * max(1.0, abs(expect)), (name, got, expect)


def pin_bf16_bits_exact(o):
    assert o.bf16_to_double(0x3F80) == 1.0
    assert o.bf16_to_double(0xC000) == -2.0
    assert o.bf16_to_double(0x3E80) == 0.25
    z = o.bf16_to_double(0x8000)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    assert o.bf16_to_double(0x7F7F) == float.fromhex("0x1.fep127")  # bf16 max
    assert o.bf16_to_double(0x0001) == 2.0 ** -133                   # smallest subnormal
    assert math.isinf(o.bf16_to_double(0x7F80))


def pin_zero_rows(o):
    # a = G·L vanishes when either half is zero (±0 compare equal; the pages fix no signed-zero rule)
    # rows are [gate (3) | linear (3)]
    x = np.array([[0.0, 1.5, -0.0, 3.0, 0.0, 0.0], [2.0, -7.0, 0.5, 0.0, -0.0, 1.0]])
    out = o.fwd_f64(x)
    assert out[0, 0] == 0.0 and out[0, 1] == 0.0 and out[0, 2] == 0.0
    assert out[1, 0] == 0.0 and out[1, 1] == 0.0
    assert out[1, 2] > 0.0


def pin_saturation_limits(o):
    # G -> beta as u -> +inf (tanh -> 1, sigmoid -> 1); G -> 0- as u -> -inf (≈ -beta·e^u)
    G, L, Gp, Lp = o.point(80.0, 1000.0)
    assert G == 4.0 and L == 25.0 and Gp == 0.0 and Lp == 0.0
    G, L, Gp, Lp = o.point(-80.0, -1000.0)
    assert G < 0 and abs(G - (-4.0 * math.exp(-80.0))) <= 1e-12 * 4.0 * math.exp(-80.0)
    assert L == -25.0 and Lp == 0.0
    assert Gp < 0 and abs(Gp) < 1e-33
    big = float.fromhex("0x1.fep127")  # largest finite bf16, ~3.39e38
    for u in (big, -big):
        for v in (big, -big):
            G, L, Gp, Lp = o.point(u, v)
            assert all(math.isfinite(t) for t in (G, L, Gp, Lp))
            assert G == (4.0 if u > 0 else 0.0)
            assert L == math.copysign(25.0, v)
            assert Gp == 0.0 and Lp == 0.0
    # other beta / lbeta saturate at beta / lbeta
    G, L, _, _ = o.point(1e4, 1e4, 2.5, 7.0)
    assert G == 2.5 and L == 7.0


def pin_small_argument_expansion(o):
    # 4 tanh(u/4) = u - u^3/48 + ..., sigmoid(u) = 1/2 + u/4 - u^3/48 + ...
    # so G(u) = u/2 + u^2/4 - u^3/96 + O(u^4) and G'(u) = 1/2 + u/2 + O(u^2);
    # L(v) = v + O(v^3), L'(v) = 1 - (v/25)^2 + O(v^4)
    for u in (1e-4, -1e-4, 3e-6):
        G, _, Gp, _ = o.point(u, 0.0)
        assert abs(G - (u / 2 + u * u / 4 - u ** 3 / 96)) <= abs(u) ** 4 + 4e-16 * abs(G)
        assert abs(Gp - (0.5 + u / 2)) <= abs(u) ** 2
    for v in (1e-3, -2e-3):
        _, L, _, Lp = o.point(0.0, v)
        assert abs(L - v) <= abs(v) ** 3
        assert abs(Lp - (1 - (v / 25) ** 2)) <= 1e-12


def pin_symmetries(o):
    rng = np.random.default_rng(11)
    for beta, lbeta in ((4.0, 25.0), (1.5, 3.0), (9.0, 60.0)):
        for t in np.concatenate([rng.normal(0, 3, 50), rng.uniform(-60, 60, 50)]):
            t = float(t)
            Gp_, Lp_, Gpp, Lpp = o.point(t, t, beta, lbeta)
            Gm, Lm, Gpm, Lpm = o.point(-t, -t, beta, lbeta)
            # L is odd, L' is even
            assert Lm == -Lp_ and Lpm == Lpp
            # sigmoid(u) + sigmoid(-u) = 1  =>  G(u) - G(-u) = beta·tanh(u/beta)
            #                               =>  G'(u) + G'(-u) = 1 - tanh(u/beta)^2
            th = math.tanh(t / beta)
            assert abs((Gp_ - Gm) - beta * th) <= 1e-14 * beta
            assert abs((Gpp + Gpm) - (1 - th * th)) <= 1e-14


def pin_swiglu_limit(o):
    # beta, lbeta -> inf: beta·tanh(u/beta) -> u and lbeta·tanh(v/lbeta) -> v, so SiTU-GLU
    # becomes SwiGLU  a = silu(u)·v  with  silu'(u) = sigmoid(u)·(1 + u·(1 - sigmoid(u))).
    rng = np.random.default_rng(5)
    for u, v in zip(rng.normal(0, 4, 200), rng.normal(0, 4, 200)):
        u, v = float(u), float(v)
        G, L, Gp, Lp = o.point(u, v, 1e8, 1e8)
        s = 1.0 / (1.0 + math.exp(-u))
        silu = u * s
        dsilu = s * (1.0 + u * (1.0 - s))
        assert abs(G - silu) <= 1e-12 * max(1.0, abs(silu))
        assert abs(L - v) <= 1e-12 * max(1.0, abs(v))
        assert abs(Gp - dsilu) <= 1e-12
        assert abs(Lp - 1.0) <= 1e-12


def _lam(o, x, g, p, beta, lbeta):
    """Λ(x, p) = Σ_r p_r Σ_j g_rj·a_rj(x), with a from the oracle's forward."""
    a = o.fwd_f64(x, beta, lbeta)
    return float(np.sum(p[:, None] * g * a))


def pin_finite_differences(o, beta=4.0, lbeta=25.0):
    rng = np.random.default_rng(7)
    R, H = 3, 5
    x = rng.normal(0, 3, (R, 2 * H))
    x[0, 0], x[1, H + 1] = 0.0, -0.0          # include the origin
    x[2, 1], x[2, H + 2] = -9.0, 40.0         # and a saturating pair
    g = rng.normal(0, 1, (R, H))
    p = rng.uniform(0.05, 1, R)
    dx, dp, dpa = o.bwd_router_f64(x, g, p, beta, lbeta)
    for r in range(R):
        for j in range(2 * H):
            h = 1e-6 * max(1.0, abs(x[r, j]))
            xp, xm = x.copy(), x.copy()
            xp[r, j] += h
            xm[r, j] -= h
            fd = (_lam(o, xp, g, p, beta, lbeta) - _lam(o, xm, g, p, beta, lbeta)) / (2 * h)
            assert abs(fd - dx[r, j]) <= 1e-7 * max(1.0, abs(dx[r, j])), (r, j, fd, dx[r, j])
        # Λ is linear in p_r, so the central difference is exact up to rounding
        hp = 1e-3
        pp, pm = p.copy(), p.copy()
        pp[r] += hp
        pm[r] -= hp
        fd = (_lam(o, x, g, pp, beta, lbeta) - _lam(o, x, g, pm, beta, lbeta)) / (2 * hp)
        assert abs(fd - dp[r]) <= 1e-9 * max(1.0, abs(dp[r]))
        a = o.fwd_f64(x[r:r + 1], beta, lbeta)[0]
        assert abs(dpa[r] - np.sum(np.abs(g[r] * a))) <= 1e-12 * dpa[r]


def pin_tiny_expert_router_rewrite(o):
    """y = Σ_e p_e W_e a_e(x_e); loss = <c, y>. The naive router gradient <c, o_e> with the
    stored expert output o_e = W_e a_e must equal the rewritten <W_eᵀ c, a_e>, which is the
    oracle's dp with g = W_eᵀ c; and dL/dx_e must equal the oracle's dx with the same g and p_e."""
    rng = np.random.default_rng(3)
    D, H, E = 8, 6, 3
    W = rng.normal(0, 0.5, (E, D, H))
    xs = rng.normal(0, 3, (E, 2 * H))
    p = rng.dirichlet(np.ones(E))
    c = rng.normal(0, 1, D)

    def loss(xs_, p_):
        a = o.fwd_f64(xs_)
        y = sum(p_[e] * (W[e] @ a[e]) for e in range(E))
        return float(c @ y)

    a = o.fwd_f64(xs)
    g = np.stack([W[e].T @ c for e in range(E)])          # g_e = W_eᵀ dL/dy
    dx, dp, _ = o.bwd_router_f64(xs, g, p)
    for e in range(E):
        o_e = W[e] @ a[e]
        naive = float(c @ o_e)                               # <dL/dy, o_e>
        rewritten = float(g[e] @ a[e])                       # <W_eᵀ dL/dy, a_e>
        assert abs(naive - rewritten) <= 1e-12 * max(1.0, abs(naive))
        assert abs(dp[e] - naive) <= 1e-12 * max(1.0, abs(naive))
        hp = 1e-4
        pp, pm = p.copy(), p.copy()
        pp[e] += hp
        pm[e] -= hp
        fd_p = (loss(xs, pp) - loss(xs, pm)) / (2 * hp)
        assert abs(fd_p - dp[e]) <= 1e-9 * max(1.0, abs(dp[e]))
        for j in range(2 * H):
            h = 1e-6 * max(1.0, abs(xs[e, j]))
            xp, xm = xs.copy(), xs.copy()
            xp[e, j] += h
            xm[e, j] -= h
            fd = (loss(xp, p) - loss(xm, p)) / (2 * h)
            assert abs(fd - dx[e, j]) <= 1e-7 * max(1.0, abs(dx[e, j])), (e, j)


def _definition_torch(x: torch.Tensor, beta: float, lbeta: float) -> torch.Tensor:
    """The forward definition written as plain PyTorch ops (float64, CPU) so autograd can
    differentiate it independently of the oracle's hand-derived G' and L'."""
    H = x.shape[-1] // 2
    u, v = x[..., :H], x[..., H:]
    return torch.tanh(u / beta).mul(beta).mul(torch.sigmoid(u)) * torch.tanh(v / lbeta).mul(lbeta)


def pin_autograd_of_definition(o, beta=4.0, lbeta=25.0):
    gen = torch.Generator().manual_seed(17)
    R, H = 9, 33
    x = (torch.randn(R, 2 * H, generator=gen, dtype=torch.float64) * 4).requires_grad_(True)
    g = torch.randn(R, H, generator=gen, dtype=torch.float64)
    p = torch.rand(R, generator=gen, dtype=torch.float64).requires_grad_(True)
    a = _definition_torch(x, beta, lbeta)
    lam = (p[:, None] * g * a).sum()
    lam.backward()
    out_o = o.fwd_f64(x.detach().numpy(), beta, lbeta)
    dx_o, dp_o, _ = o.bwd_router_f64(x.detach().numpy(), g.numpy(), p.detach().numpy(), beta, lbeta)
    np.testing.assert_allclose(out_o, a.detach().numpy(), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dx_o, x.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dp_o, p.grad.numpy(), rtol=1e-12, atol=1e-13)


def pin_bf16_entry_matches_f64_entry(o):
    rng = np.random.default_rng(1)
    R, H = 5, 24
    xb = torch.from_numpy(rng.normal(0, 3, (R, 2 * H)).astype(np.float32)).to(torch.bfloat16)
    gb = torch.from_numpy(rng.normal(0, 1, (R, H)).astype(np.float32)).to(torch.bfloat16)
    p = rng.uniform(0, 1, R).astype(np.float32)
    xbits = xb.view(torch.int16).numpy().view(np.uint16)
    gbits = gb.view(torch.int16).numpy().view(np.uint16)
    out_b = o.fwd_bf16(xbits)
    out_d = o.fwd_f64(xb.to(torch.float64).numpy())
    assert np.array_equal(out_b, out_d)
    dx_b, dp_b, dpa_b = o.bwd_router_bf16(xbits, gbits, p)
    dx_d, dp_d, dpa_d = o.bwd_router_f64(xb.to(torch.float64).numpy(), gb.to(torch.float64).numpy(),
                                              p.astype(np.float64))
    assert np.array_equal(dx_b, dx_d) and np.array_equal(dp_b, dp_d) and np.array_equal(dpa_b, dpa_d)


def pin_thread_count_independent(o):
    rng = np.random.default_rng(2)
    R, H = 37, 40
    x = rng.normal(0, 3, (R, 2 * H))
    g = rng.normal(0, 1, (R, H))
    p = rng.uniform(0, 1, R)
    r1 = o.bwd_router_f64(x, g, p, nthreads=1)
    r5 = o.bwd_router_f64(x, g, p, nthreads=5)
    for a, b in zip(r1, r5):
        assert np.array_equal(a, b)
    assert np.array_equal(o.fwd_f64(x, nthreads=1), o.fwd_f64(x, nthreads=7))


def pin_extreme_finite_inputs(o):
    big = float.fromhex("0x1.fep127")
    x = np.array([[big, -big, 0.0, big, -big, 1.0, 3.0, -big]])
    g = np.array([[1.0, -2.0, 0.5, 3.0]])
    p = np.array([0.7])
    dx, dp, dpa = o.bwd_router_f64(x, g, p)
    assert np.all(np.isfinite(dx)) and np.isfinite(dp).all() and np.isfinite(dpa).all()
    out = o.fwd_f64(x)
    assert np.all(np.isfinite(out))
    # u = +big: G = 4; v = -big: L = -25  ->  a = -100
    assert out[0, 0] == -100.0


def pin_empty_rows(o):
    out = o.fwd_f64(np.zeros((0, 8)))
    assert out.shape == (0, 4)
    dx, dp, dpa = o.bwd_router_f64(np.zeros((0, 8)), np.zeros((0, 4)), np.zeros((0,)))
    assert dx.shape == (0, 8) and dp.shape == (0,)


# ---------------------------------------------------------------- block-wise FP8 saved x

def _e4m3_table():
    """Values of the non-negative finite E4M3 codes 0x00..0x7E from the OCP 8-bit floating point
    format definition: exponent field e (bias 7), mantissa m/8, subnormals at e = 0."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append(m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return vals


def _brute_e4m3(v: float) -> int:
    """Nearest code by exhaustive search over all finite codes, ties to the even code,
    saturating beyond the largest finite value (an implementation independent of the oracle's)."""
    if math.isnan(v):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    vals = _e4m3_table()
    if a >= vals[-1]:
        return sign | 0x7E
    best = min(range(len(vals)), key=lambda c: (abs(vals[c] - a), c & 1))
    return sign | best


def pin_e4m3_codec(o):
    vals = _e4m3_table()
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6 and vals[0x38] == 1.0
    for c in range(0x7F):                                   # exact round trip of every finite code
        assert o.e4m3_decode(c) == vals[c] and o.e4m3_decode(c | 0x80) == -vals[c]
        assert o.e4m3_encode(vals[c]) == c and o.e4m3_encode(-vals[c]) == (c | 0x80 if c else 0x80)
    assert math.isnan(o.e4m3_decode(0x7F)) and math.isnan(o.e4m3_decode(0xFF))
    probes = [0.0, 448.0, 449.0, 464.0, 479.0, 1e6, 3e38, 2.0 ** -10, 2.0 ** -11, 1e-30]
    for c in range(0x7E):                                    # every midpoint and its fp32 neighbours
        mid = (vals[c] + vals[c + 1]) / 2
        probes += [mid, float(np.nextafter(np.float32(mid), np.float32(0))),
                   float(np.nextafter(np.float32(mid), np.float32(1e9)))]
    rng = np.random.default_rng(8)
    probes += list(np.exp2(rng.uniform(-12, 9.5, 400)).astype(np.float32))
    for v in probes:
        v = float(np.float32(v))
        for s in (v, -v):
            assert o.e4m3_encode(s) == _brute_e4m3(s), (s, o.e4m3_encode(s), _brute_e4m3(s))
    assert o.e4m3_encode(float("nan")) & 0x7F == 0x7F
    # PyTorch's float8_e4m3fn cast (round to nearest even) agrees inside the finite range
    inrange = torch.tensor([p for p in probes if abs(p) <= 448.0], dtype=torch.float32)
    tq = inrange.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    assert tq == [o.e4m3_encode(float(p)) for p in inrange.tolist()]


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def pin_fp8_block_quantization(o):
    rng = np.random.default_rng(4)
    for H in (256, 200, 1):                                  # whole blocks, a short last block, H = 1
        R, blk = 5, 128
        nb = -(-H // blk)
        x = rng.normal(0, 3, (R, 2 * H)).astype(np.float32)
        x[1, :min(H, blk)] = 0.0                             # an all-zero gate block
        x[2, H] = 1e30                                       # a huge value in the first linear block
        x[3, :] *= 1e-38                                     # tiny values (subnormal codes)
        xb = _bf16_bits(x)
        xf = _bits_to_f32(xb)
        q, sc = o.quantize_fp8(xb, blk)
        xh = o.dequantize_fp8(q, sc, blk)
        assert q.shape == (R, 2 * H) and sc.shape == (R, 2 * nb)
        for r in range(R):
            for half in range(2):
                for b in range(nb):
                    lo, hi = half * H + b * blk, half * H + min(H, (b + 1) * blk)
                    blkv = xf[r, lo:hi]
                    amax = np.float32(np.max(np.abs(blkv)))
                    s = sc[r, half * nb + b]
                    floor = np.float32(448.0 * 2.0 ** -126)
                    assert s == np.float32(max(amax, floor) / np.float32(448.0))
                    if amax == 0:
                        assert np.all(q[r, lo:hi] == 0) and np.all(xh[r, lo:hi] == 0)
                        continue
                    if amax >= floor:                                   # the amax element saturates the range
                        assert (q[r, lo:hi][np.argmax(np.abs(blkv))] & 0x7F) == 0x7E
                    # half an E4M3 step: 2^-4 relative for normal codes, 2^-10·s absolute for subnormal
                    # codes; plus the fp32 rounding of the products and of a subnormal fp32 result
                    err = np.abs(xh[r, lo:hi].astype(np.float64) - blkv.astype(np.float64))
                    bound = np.maximum(2.0 ** -4 * np.abs(blkv), 2.0 ** -10 * float(s)) * (1 + 2 ** -20) \
                        + 2.0 ** -23 * np.abs(blkv) + 2.0 ** -149
                    assert np.all(err <= bound), (H, r, half, b, float(err.max()))
        # locality: changing one element only changes its own block
        x2 = x.copy()
        x2[0, H + (H - 1)] = 77.0
        q2, sc2 = o.quantize_fp8(_bf16_bits(x2), blk)
        changed = np.nonzero(sc2 != sc)
        assert set(zip(*changed)) <= {(0, nb + (H - 1) // blk)}
        assert np.array_equal(q2[1:], q[1:]) and np.array_equal(q2[0, :H], q[0, :H])
    # dequantisation uses the scale of the element's own half and block
    q = np.full((1, 2 * 256), 0x38, dtype=np.uint8)          # every code = 1.0
    sc = np.array([[1.0, 2.0, 4.0, 8.0]], dtype=np.float32)
    xh = o.dequantize_fp8(q, sc, 128)
    assert np.array_equal(xh[0], np.repeat(np.array([1.0, 2.0, 4.0, 8.0], dtype=np.float32), 128))


def pin_fp8_backward_is_backward_of_dequantized(o):
    """The FP8 backward is the bf16 backward evaluated on the dequantised x (exactly)."""
    rng = np.random.default_rng(9)
    R, H = 3, 200
    xb = _bf16_bits(rng.normal(0, 3, (R, 2 * H)))
    gb = _bf16_bits(rng.normal(0, 1, (R, H)))
    p = rng.uniform(0, 1, R).astype(np.float32)
    q, sc = o.quantize_fp8(xb)
    dx, dp, dpa = o.bwd_router_fp8(q, sc, gb, p)
    xh = o.dequantize_fp8(q, sc).astype(np.float64)
    dx2, dp2, _ = o.bwd_router_f64(xh, _bits_to_f32(gb).astype(np.float64), p.astype(np.float64))
    assert np.array_equal(dx, dx2) and np.array_equal(dp, dp2)


# ---------------------------------------------------------------- fused down-projection dgrad

def pin_grouped_dgrad(o_mod):
    """The oracle's grouped dgrad equals a brute-force triple loop, experts with 0 rows included;
    and the fused dp equals the naive router gradient <dL/dy, o_e> with stored o_e = W_e·a_e."""
    rng = np.random.default_rng(12)
    E, H, D = 4, 3, 5
    counts = [2, 0, 3, 1]
    off = np.concatenate([[0], np.cumsum(counts)])
    R = int(off[-1])
    dy = _bf16_bits(rng.normal(0, 1, (R, D)))
    wt = _bf16_bits(rng.normal(0, 0.5, (E, H, D)).reshape(E * H, D)).reshape(E, H, D)
    x = _bf16_bits(rng.normal(0, 3, (R, 2 * H)))
    p = rng.uniform(0.1, 1, R).astype(np.float32)
    g = o_mod.grouped_dgrad(dy, wt, off)
    dyf, wtf = _bits_to_f32(dy).astype(np.float64), _bits_to_f32(wt).astype(np.float64)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            for j in range(H):
                ref = sum(dyf[r, d] * wtf[e, j, d] for d in range(D))
                assert abs(g[r, j] - ref) <= 1e-12 * max(1.0, abs(ref))
    dx, dp, _ = o_mod.dgrad_bwd_router(x, dy, wt, off, p)
    xf = _bits_to_f32(x).astype(np.float64)
    a = o_mod.fwd_f64(xf)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            o_e = wtf[e].T @ a[r]                          # o_e = W_down,e · a_e  (W_down,e = wt[e]ᵀ)
            naive = float(dyf[r] @ o_e)                    # <dL/dy, o_e>
            assert abs(dp[r] - naive) <= 1e-12 * max(1.0, abs(naive))
            # dx: central differences of p_r·<dL/dy, W_down,e·a_e(x_r)> in each input
            for k in range(2 * H):
                hk = 1e-6 * max(1.0, abs(xf[r, k]))
                xp, xm = xf[r].copy(), xf[r].copy()
                xp[k] += hk
                xm[k] -= hk
                fp = float(dyf[r] @ (wtf[e].T @ o_mod.fwd_f64(xp[None, :])[0]))
                fm = float(dyf[r] @ (wtf[e].T @ o_mod.fwd_f64(xm[None, :])[0]))
                fd = float(p[r]) * (fp - fm) / (2 * hk)
                assert abs(dx[r, k] - fd) <= 1e-6 * max(1.0, abs(fd))


# ---------------------------------------------------------------- bf16 rounding, gate/up projection

def pin_round_bf16(o):
    """Round-to-nearest-even from double to bf16, against what fixes it independently:
    - for doubles that are exact fp32 values, PyTorch's fp32 -> bf16 cast (RNE) on 40000 random
      finite bit patterns (normals, subnormals, both signs) plus signed zeros and the extremes;
    - exact midpoints between consecutive bf16 values go to the even significand, and the
      nearest double on either side of a midpoint goes to the nearer value (this is where a
      double -> fp32 -> bf16 double rounding would differ);
    - overflow: the largest finite bf16 plus half its spacing rounds to infinity, anything
      below that midpoint to the largest finite value; NaN stays NaN;
    - bf16_neighbours brackets v with consecutive values and contains the rounded value."""
    rng = np.random.default_rng(21)
    bits = rng.integers(0, 2 ** 32, 40000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    f = np.concatenate([f, np.array([0.0, -0.0, 1.0, -1.0, 3.3895313892515355e38, -3.3895313892515355e38,
                                     1e-45, -1e-45, 2.0 ** -133, 2.0 ** -126, 65504.0], dtype=np.float32)])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = o.round_bf16_array(f.astype(np.float64))
    assert np.array_equal(got, want)
    # midpoints and their neighbours, across binades and in the subnormal range
    for b in [0x3F80, 0x3F81, 0x4049, 0x0001, 0x0002, 0x007F, 0x0080, 0x7F7E, 0xBF80, 0xBF81, 0x8001]:
        lo = o.bf16_to_double(b)
        hi = o.bf16_to_double(b + 1)
        mid = (lo + hi) / 2.0                                  # exact in double
        even = b if (b & 1) == 0 else b + 1
        assert o.round_bf16(mid) == even, hex(b)
        toward_hi = math.nextafter(mid, hi)
        toward_lo = math.nextafter(mid, lo)
        assert o.round_bf16(toward_hi) == b + 1 and o.round_bf16(toward_lo) == b, hex(b)
    maxf = o.bf16_to_double(0x7F7F)
    half = 2.0 ** 119                                          # half the spacing at the top binade
    assert o.round_bf16(maxf + half) == 0x7F80
    assert o.round_bf16(math.nextafter(maxf + half, 0.0)) == 0x7F7F
    assert o.round_bf16(-(maxf + half)) == 0xFF80
    assert o.round_bf16(float("inf")) == 0x7F80 and o.round_bf16(float("-inf")) == 0xFF80
    assert (o.round_bf16(float("nan")) & 0x7FFF) > 0x7F80
    assert o.round_bf16(-0.0) == 0x8000 and o.round_bf16(0.0) == 0x0000
    for v in [1.001, -1.001, 2.0 ** -130 * 1.3, 1e30, -7.77e-3, 3.0, 0.0]:
        lo, hi = o.bf16_neighbours(v)
        dlo, dhi = o.bf16_to_double(lo), o.bf16_to_double(hi)
        assert dlo <= v <= dhi
        r = o.round_bf16(v)
        assert r in (lo, hi)
        if dlo != dhi:
            assert abs(int(hi) - int(lo)) == 1                 # consecutive bf16 values


def pin_grouped_gateup(o):
    """The oracle's gate/up projection equals a brute-force triple loop (experts with 0 rows
    included), puts W_gate,e·h in columns 0..H-1 and W_up,e·h in H..2H-1, and its out is
    SiTU(gate, linear) of the bf16-rounded projections, element by element through the
    oracle's point function (a_e = SiTU(W_gate,e x_e, W_up,e x_e))."""
    rng = np.random.default_rng(13)
    E, H, D = 4, 3, 5
    counts = [2, 0, 3, 1]
    off = np.concatenate([[0], np.cumsum(counts)])
    R = int(off[-1])
    h = _bf16_bits(rng.normal(0, 1, (R, D)))
    w = _bf16_bits(rng.normal(0, 1.5, (E * 2 * H, D))).reshape(E, 2 * H, D)
    x, mag = o.grouped_gateup(h, w, off)
    x2, xb, out, mag2 = o.gateup_fwd(h, w, off)
    hf, wf = _bits_to_f32(h).astype(np.float64), _bits_to_f32(w).astype(np.float64)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            for n in range(2 * H):
                ref = sum(hf[r, d] * wf[e, n, d] for d in range(D))
                refa = sum(abs(hf[r, d] * wf[e, n, d]) for d in range(D))
                assert abs(x[r, n] - ref) <= 1e-12 * max(1.0, abs(ref))
                assert abs(mag[r, n] - refa) <= 1e-12 * max(1.0, refa)
                assert xb[r, n] == o.round_bf16(ref)
            for j in range(H):
                u, v = o.bf16_to_double(int(xb[r, j])), o.bf16_to_double(int(xb[r, H + j]))
                G, L, _, _ = o.point(u, v)
                assert abs(out[r, j] - G * L) <= 1e-14 * max(1.0, abs(G * L))
    assert np.array_equal(x, x2) and np.array_equal(mag, mag2)


# ---------------------------------------------------------------- Adam on host-resident state

def _torch_adam_steps(w0, grads, lr, b1, b2, eps, wd):
    """PyTorch's own Adam / AdamW (float64, CPU, single-tensor path) over a list of gradients."""
    p = torch.nn.Parameter(torch.tensor(w0, dtype=torch.float64))
    cls = torch.optim.AdamW if wd > 0 else torch.optim.Adam
    opt = cls([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    for g in grads:
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def pin_adam_matches_torch(o):
    """The oracle's textbook Adam (double) equals PyTorch's Adam and AdamW in float64 over several
    steps, including a large eps (where its placement outside the bias-corrected sqrt matters)."""
    import oracle as omod
    rng = np.random.default_rng(31)
    n = 257
    for lr, b1, b2, eps, wd in [(1e-3, 0.9, 0.999, 1e-8, 0.0), (3e-2, 0.8, 0.95, 0.1, 0.0),
                                (1e-2, 0.9, 0.99, 1e-6, 0.1)]:
        w0 = rng.normal(0, 1, n)
        grads = [rng.normal(0, 1, n) * 10.0 ** rng.uniform(-3, 1, n) for _ in range(5)]
        w, m, v = w0.copy(), np.zeros(n), np.zeros(n)
        for t, g in enumerate(grads, start=1):
            w, m, v = o.adam_f64(w, m, v, g, omod.adam_hp(lr, b1, b2, eps, wd, t))
        tw, tm, tv = _torch_adam_steps(w0, grads, lr, b1, b2, eps, wd)
        assert np.allclose(w, tw, rtol=1e-12, atol=1e-14), (lr, eps, wd)
        assert np.allclose(m, tm, rtol=1e-12, atol=1e-300) and np.allclose(v, tv, rtol=1e-12, atol=1e-300)


def pin_adam_first_step_closed_form(o):
    """From zero moments at t = 1 the bias corrections cancel (1 - b^1 = 1 - b): m = (1-b1)·g,
    v = (1-b2)·g², and w moves by exactly lr·g / (|g| + eps), in both precisions."""
    import oracle as omod
    g = np.array([0.5, -2.0, 1e-3, 3e4, -7.25e-6, 0.0])
    lr, eps = 1e-2, 1e-8
    hp = omod.adam_hp(lr, 0.9, 0.999, eps, 0.0, 1)
    w, m, v = o.adam_f64(np.ones(g.size), np.zeros(g.size), np.zeros(g.size), g, hp)
    assert np.allclose(m, 0.1 * g, rtol=1e-15, atol=0) and np.allclose(v, 0.001 * g * g, rtol=1e-14, atol=0)
    assert np.allclose(w, 1.0 - lr * g / (np.abs(g) + eps), rtol=1e-14, atol=0)
    ms, mb, vb, wb = o.adam_stored(np.ones(g.size, np.float32), np.zeros(g.size, np.uint16),
                                   np.zeros(g.size, np.uint16), g.astype(np.float32), hp)
    ref = 1.0 - lr * g / (np.abs(g) + eps)
    assert np.all(np.abs(ms - ref) <= 4 * np.spacing(np.float32(1.0)))
    assert np.array_equal(wb, _bf16_bits(ms))


def pin_adam_stored_is_a_rounding_of_f64(o):
    """One stored-precision step (fp32 arithmetic, bf16 moments) from any state is the double
    step up to fp32 rounding: the master weight within a few fp32 ulps of the step and of w;
    the moment codes are round-to-nearest-even of the double moments, except where the double
    value lies within the fp32 error of a bf16 midpoint; the working weight is RNE of the
    master. Weight decay on and off, late steps (small bias corrections) too."""
    import oracle as omod
    rng = np.random.default_rng(32)
    n = 4096
    for t, wd in [(1, 0.0), (7, 0.0), (1000, 0.05), (3, 0.1)]:
        hp = omod.adam_hp(2e-3, 0.9, 0.999, 1e-8, wd, t)
        w0 = rng.normal(0, 0.05, n).astype(np.float32)
        m0 = _bf16_bits(rng.normal(0, 1e-2, n))
        v0 = _bf16_bits(rng.uniform(0, 1e-3, n))
        g = (rng.normal(0, 1, n) * 10.0 ** rng.uniform(-4, 0, n)).astype(np.float32)
        ms, mb, vb, wb = o.adam_stored(w0, m0, v0, g, hp)
        wd_, md, vd = o.adam_f64(w0.astype(np.float64), _bits_to_f32(m0).astype(np.float64),
                                  _bits_to_f32(v0).astype(np.float64), g.astype(np.float64), hp)
        # the update s·m/q rounded in fp32: m = b1·m0 + (1-b1)·g may cancel, so its error scales
        # with |b1·m0| + |(1-b1)·g|; the rest contributes a few ulps of the update and of w
        bc1, bc2 = 1 - 0.9 ** t, 1 - 0.999 ** t
        q = np.sqrt(vd) / np.sqrt(bc2) + 1e-8
        u_abs = 2e-3 / bc1 * (0.9 * np.abs(_bits_to_f32(m0)) + 0.1 * np.abs(g)) / q
        big = np.maximum(np.abs(w0).astype(np.float64), np.abs(wd_))
        tol_w = 4 * np.spacing(big.astype(np.float32)).astype(np.float64) + 8 * 2.0 ** -24 * u_abs
        assert np.all(np.abs(ms - wd_) <= tol_w)
        for bits, ref, scale in ((mb, md, 0.9 * np.abs(_bits_to_f32(m0)) + 0.1 * np.abs(g)),
                                 (vb, vd, 0.999 * _bits_to_f32(v0) + 0.001 * g.astype(np.float64) ** 2)):
            lo = o.round_bf16_array(ref - 4 * 2.0 ** -24 * scale)
            hi = o.round_bf16_array(ref + 4 * 2.0 ** -24 * scale)
            val, vlo, vhi = (_bits_to_f32(x).astype(np.float64) for x in (bits, lo, hi))
            assert np.all((vlo <= val) & (val <= vhi))
            assert np.mean(bits == o.round_bf16_array(ref)) > 0.99
        assert np.array_equal(wb, _bf16_bits(ms))

"""The seeded synthetic inputs: determinism, shapes, distributions and row structure."""
import math

import torch

import situ_inputs as si


def test_deterministic_and_seed_sensitive():
    w = si.custom(64, 40, seed=9)
    a = si.generate(w)
    b = si.generate(w)
    for s, t in zip(a, b):
        assert torch.equal(s.view(torch.int16) if s.dtype == torch.bfloat16 else s,
                           t.view(torch.int16) if t.dtype == torch.bfloat16 else t)
    c = si.generate(si.custom(64, 40, seed=10))
    assert not torch.equal(a[0].float(), c[0].float())


def test_chunking_does_not_change_values():
    w = si.custom(50, 16, seed=3)
    x1, g1, p1 = si.generate(w, chunk_rows=7)
    x2, g2, p2 = si.generate(w, chunk_rows=1000)
    # torch's CPU generator draws sequentially, so chunked draws concatenate to the same stream
    assert torch.equal(x1.float(), x2.float()) and torch.equal(g1.float(), g2.float())
    assert torch.equal(p1, p2)


def test_router_rows_structure():
    p, e, tok = si.router_rows(300, seed=0)
    assert p.shape == (300 * 16,) and p.dtype == torch.float32
    sums = p.view(300, 16).double().sum(-1)
    assert torch.allclose(sums, torch.ones_like(sums), atol=1e-6)
    # k in descending-score order => descending softmax weights within a token
    pv = p.view(300, 16)
    assert bool((pv[:, :-1] >= pv[:, 1:]).all())
    ev = e.view(300, 16)
    assert all(len(set(row.tolist())) == 16 for row in ev)          # 16 distinct experts per token
    assert int(e.min()) >= 0 and int(e.max()) < si.N_EXPERTS
    assert torch.equal(tok, torch.arange(300).repeat_interleave(16))


def test_expert_grouped_order():
    p0, e0, t0 = si.router_rows(200, seed=2, order="token")
    p1, e1, t1 = si.router_rows(200, seed=2, order="expert")
    assert bool((e1[1:] >= e1[:-1]).all())                             # grouped by expert id
    same = e1[1:] == e1[:-1]
    assert bool((t1[1:][same] > t1[:-1][same]).all())                  # ties by token
    # same multiset of (token, expert, p) rows
    key0 = sorted(zip(t0.tolist(), e0.tolist(), p0.tolist()))
    key1 = sorted(zip(t1.tolist(), e1.tolist(), p1.tolist()))
    assert key0 == key1


def test_saturating_mixture_fractions():
    w = si.get("saturating_mix_r16384_h3072")
    small = si.Workload(w.name, 512, w.H, w.x_kind, w.x_std, w.g_std, w.p_kind, w.order, w.seed)
    x, g, p = si.generate(small)
    xf = x.float()
    n = xf.numel()
    bits = x.view(torch.int16)
    pos0 = int((bits == 0).sum()) / n
    neg0 = int((bits == torch.tensor(-32768, dtype=torch.int16)).sum()) / n
    big = int((xf.abs() > 20).sum()) / n                               # only the uniform part reaches |x| > 20
    assert abs(pos0 - 0.005) < 0.001 and abs(neg0 - 0.005) < 0.001
    assert abs(big - 0.10 * 60 / 80) < 0.005
    assert float(xf.abs().max()) <= 80.0


def test_normal_scales():
    w = si.custom(256, 512, seed=1, x_std=3.0, g_std=0.5)
    x, g, p = si.generate(w)
    assert math.isclose(float(x.float().std()), 3.0, rel_tol=0.02)
    assert math.isclose(float(g.float().std()), 0.5, rel_tol=0.02)
    assert float(p.min()) >= 0.0 and float(p.max()) < 1.0


def test_workload_table():
    assert si.get("routed_r1024_h3072").R == 1024
    assert si.get("pages_scale_r1600000_h3072").R == 1_600_000
    assert si.get("expert_grouped_r262144_h3072").order == "expert"
    assert si.tail_sweep(37, 1000).H == 1000

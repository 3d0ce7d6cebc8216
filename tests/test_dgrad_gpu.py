"""Parity of the fused down-projection dgrad (tcgen05 grouped GEMM + SiTU-GLU backward + router
gradient) with the oracle: g = dY·W_down,e in fp64 (numpy matmul), then the fp64 backward."""
import numpy as np
import pytest
import torch

import oracle
import situ_inputs as si
from _parity import Parity, bits_of, for_expert_groups_parallel

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sg(cuda_lib):
    assert torch.cuda.is_available()
    return cuda_lib


def make(counts, H, D, seed, x_std=3.0, device="cpu"):
    gen = torch.Generator(device=device).manual_seed(seed)
    E, R = len(counts), int(sum(counts))
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int64)
    x = (torch.randn(R, 2 * H, generator=gen, device=device) * x_std).to(torch.bfloat16)
    dy = torch.randn(R, D, generator=gen, device=device).to(torch.bfloat16)
    wt = torch.empty(E, H, D, dtype=torch.bfloat16, device=device)
    for e in range(E):                       # W_down entries ~ N(0, 1/D): g ~ N(0, 1)
        wt[e] = (torch.randn(H, D, generator=gen, device=device) / D ** 0.5).to(torch.bfloat16)
    p = torch.rand(R, generator=gen, device=device)
    return x, dy, wt, off, p


def run(sg, x, dy, wt, off, p, beta=4.0, lbeta=25.0):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    dx, dp = sg.situ_glu_bwd_router_dgrad(x.to(DEV), dy.to(DEV), wt.to(DEV), off.to(DEV), p.to(DEV), status=status,
                                          beta=beta, lbeta=lbeta)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dx, dp


CASES = {
    "one_tile": ([128], 256, 64),
    "partial_tiles": ([100, 60], 256, 128),
    "empty_experts": ([0, 300, 1, 129, 0, 77, 0], 512, 256),
    "real_widths": ([200, 0, 317, 128, 90, 250, 33, 400, 1, 255, 256, 129], 3072, 3584),
    # H / 256 N-tiles shared by min(4, H / 256) CTAs (one cluster of 3; four CTAs as two clusters
    # of 2, or as one cluster of 4 when the experts average 512 rows or more): 3 of 3, 5 over 4
    # (uneven), and 4 over one cluster of 4
    "three_way_split": ([129, 0, 200], 768, 64),
    "uneven_split": ([300, 77], 1280, 128),
    "large_experts": ([600, 517, 1000], 1024, 128),
    # either side of the host's choice (experts averaging 512 rows or more: one cluster of 4)
    "cluster_choice_511": ([510, 512], 1024, 64),
    "cluster_choice_512": ([512, 512], 1024, 64),
    # shapes off the 256-column N-tile and 64-deep K-block grid (H % 16 == 0, D % 8 == 0): the last
    # N-tile computes columns past H that are never used, the last K-block reads zeros past D
    "n_tail_h272": ([200, 77, 0, 129], 272, 128),
    "k_tail_d72": ([150, 300], 512, 72),
    "smallest_h16_d8": ([33, 0, 100], 16, 8),
    "both_tails_h1040_d200": ([300, 292, 250], 1040, 200),
    "both_tails_large_experts": ([600, 700], 400, 136),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_dgrad_all_rows(sg, name):
    counts, H, D = CASES[name]
    x, dy, wt, off, p = make(counts, H, D, seed=len(name))
    dx, dp = run(sg, x, dy, wt, off, p)
    dx_ref, dp_ref, dpa = oracle.dgrad_bwd_router(bits_of(x), bits_of(dy), bits_of(wt).reshape(wt.shape),
                                                 off.numpy(), p.numpy())
    par = Parity("dgrad " + name)
    par.bf16("dx", bits_of(dx), dx_ref)
    par.dp(dp.cpu().numpy(), dp_ref, dpa)
    par.assert_ok()


@pytest.mark.parametrize("beta,lbeta", [(2.5, 7.0), (4.0, 100.0)])
def test_dgrad_general_scales(sg, beta, lbeta):
    x, dy, wt, off, p = make([130, 0, 200], 512, 128, seed=9)
    dx, dp = run(sg, x, dy, wt, off, p, beta, lbeta)
    dx_ref, dp_ref, dpa = oracle.dgrad_bwd_router(bits_of(x), bits_of(dy), bits_of(wt).reshape(wt.shape),
                                                 off.numpy(), p.numpy(), beta, lbeta)
    par = Parity(f"dgrad beta={beta} lbeta={lbeta}")
    par.bf16("dx", bits_of(dx), dx_ref)
    par.dp(dp.cpu().numpy(), dp_ref, dpa)
    par.assert_ok()


def test_dgrad_matches_unfused_path(sg):
    """Same g through the separate route (bf16 g written out, then situ_glu_bwd_router): the fused
    result is at least as close to the oracle (it never rounds g to bf16)."""
    x, dy, wt, off, p = make([300, 200], 512, 256, seed=4)
    dx, dp = run(sg, x, dy, wt, off, p)
    g = torch.cat([dy[:300].float() @ wt[0].float().T, dy[300:].float() @ wt[1].float().T]).to(torch.bfloat16)
    dx2, dp2 = sg.situ_glu_bwd_router(x.to(DEV), g.to(DEV), p.to(DEV))
    torch.cuda.synchronize()
    dx_ref, dp_ref, _ = oracle.dgrad_bwd_router(bits_of(x), bits_of(dy), bits_of(wt).reshape(wt.shape),
                                               off.numpy(), p.numpy())
    e_fused = np.abs(dp.cpu().numpy() - dp_ref).max()
    e_split = np.abs(dp2.cpu().numpy() - dp_ref).max()
    assert e_fused <= e_split


def test_dgrad_rejects_unsupported_shapes(sg):
    x, dy, wt, off, p = make([64], 256, 64, seed=1)
    with pytest.raises(sg.SituGluError):
        sg.situ_glu_bwd_router_dgrad(x.to(DEV)[:, :500].contiguous().view(64, 500), dy.to(DEV), wt.to(DEV)[:, :250],
                                     off.to(DEV), p.to(DEV))


@pytest.mark.slow
def test_dgrad_expert_grouped_full_size_all_rows(sg):
    """R = 262144 routed rows grouped by expert over 896 experts (16384 tokens x top-16),
    H = 3072, D = 3584: the full-size launch, every row of dx and dp compared with the oracle
    (runs of consecutive experts streamed to the host, the fp64 grouped GEMM and backward on
    each run, several runs at once)."""
    w = si.get("expert_grouped_r262144_h3072")
    _, experts, _ = si.router_rows(w.tokens, w.seed, order="expert")
    counts = np.bincount(experts.numpy(), minlength=si.N_EXPERTS)
    H, D, E = w.H, 3584, si.N_EXPERTS
    gen = torch.Generator(device=DEV).manual_seed(5)
    x = (torch.randn(w.R, 2 * H, generator=gen, device=DEV) * w.x_std).to(torch.bfloat16)
    dy = torch.empty(w.R, D, dtype=torch.bfloat16, device=DEV)
    for a in range(0, w.R, 32768):
        dy[a:a + 32768] = torch.randn(min(32768, w.R - a), D, generator=gen, device=DEV).to(torch.bfloat16)
    wt = torch.empty(E, H, D, dtype=torch.bfloat16, device=DEV)
    for e in range(E):
        wt[e] = (torch.randn(H, D, generator=gen, device=DEV) / D ** 0.5).to(torch.bfloat16)
    off_np = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    off = torch.from_numpy(off_np).to(DEV)
    p, _, _ = si.router_rows(w.tokens, w.seed, order="expert")
    p_np = p.numpy()
    p = p.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    dx, dp = sg.situ_glu_bwd_router_dgrad(x, dy, wt, off, p, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    dp_np = dp.cpu().numpy()

    def check(part, e0, e1, nthreads):
        r0, r1 = int(off_np[e0]), int(off_np[e1])
        if r1 == r0:
            return
        dx_ref, dp_ref, dpa = oracle.dgrad_bwd_router(bits_of(x[r0:r1]), bits_of(dy[r0:r1]),
                                                     bits_of(wt[e0:e1]).reshape(e1 - e0, H, D),
                                                     off_np[e0:e1 + 1] - r0, p_np[r0:r1], nthreads=nthreads)
        part.bf16("dx", bits_of(dx[r0:r1]), dx_ref, row0=r0)
        part.dp(dp_np[r0:r1], dp_ref, dpa, row0=r0)

    par = Parity("dgrad expert_grouped_r262144 (all rows)")
    for_expert_groups_parallel(par, off_np, check, rows_per_group=4096)
    assert par.t["dx"].n == w.R * 2 * H and par.t["dp"].n == w.R
    par.assert_ok()
    del x, dy, wt, dx, dp
    torch.cuda.empty_cache()


def test_dgrad_max_experts_mostly_empty(sg):
    """1024 experts (the per-launch maximum; the whole M-tile prefix in shared memory), 600 rows
    spread over 37 of them, the rest empty; on a non-default stream."""
    rng = np.random.default_rng(8)
    counts = np.zeros(1024, dtype=np.int64)
    used = rng.choice(1024, 37, replace=False)
    counts[used] = rng.multinomial(600, np.ones(37) / 37)
    counts[1023] += 1                                   # the last expert owns the last row
    x, dy, wt, off, p = make(counts.tolist(), 256, 64, seed=17, x_std=2.0)
    s = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    with torch.cuda.stream(s):
        dx, dp = sg.situ_glu_bwd_router_dgrad(x.to(DEV), dy.to(DEV), wt.to(DEV), off.to(DEV), p.to(DEV),
                                              status=status, stream=s)
    s.synchronize()
    assert int(status.item()) == 0
    dx_ref, dp_ref, dpa = oracle.dgrad_bwd_router(bits_of(x), bits_of(dy), bits_of(wt).reshape(wt.shape),
                                                 off.numpy(), p.numpy())
    par = Parity("dgrad 1024 experts")
    par.bf16("dx", bits_of(dx), dx_ref)
    par.dp(dp.cpu().numpy(), dp_ref, dpa)
    par.assert_ok()


def test_dgrad_single_row(sg):
    x, dy, wt, off, p = make([0, 1, 0], 512, 128, seed=18)
    dx, dp = run(sg, x, dy, wt, off, p)
    dx_ref, dp_ref, dpa = oracle.dgrad_bwd_router(bits_of(x), bits_of(dy), bits_of(wt).reshape(wt.shape),
                                                 off.numpy(), p.numpy())
    par = Parity("dgrad single row")
    par.bf16("dx", bits_of(dx), dx_ref)
    par.dp(dp.cpu().numpy(), dp_ref, dpa)
    par.assert_ok()


def test_dgrad_rejects_too_many_experts(sg):
    x, dy, wt, off, p = make([1] * 2, 256, 64, seed=19)
    big = torch.zeros(1025, 256, 64, dtype=torch.bfloat16, device=DEV)
    offs = torch.zeros(1026, dtype=torch.int64, device=DEV)
    offs[-1] = 2
    with pytest.raises(sg.SituGluError):
        sg.situ_glu_bwd_router_dgrad(x.to(DEV), dy.to(DEV), big, offs, p.to(DEV))


def test_malformed_offsets_stay_in_bounds_and_bounded(sg):
    """Offsets that are negative, decreasing, far beyond R or overlapping: results are undefined,
    but both fused GEMMs return promptly with status 0 and write nothing outside their outputs
    (guard bands of NaN bits around dx, x and out stay intact)."""
    import time
    R, H, D, E = 200, 256, 64, 5
    gen = torch.Generator().manual_seed(30)
    off = torch.tensor([0, -5, 1 << 40, 100, 50, R], dtype=torch.int64, device=DEV)
    x = (torch.randn(R, 2 * H, generator=gen) * 3).to(torch.bfloat16).to(DEV)
    dy = torch.randn(R, D, generator=gen).to(torch.bfloat16).to(DEV)
    wt = (torch.randn(E, H, D, generator=gen) * 0.1).to(torch.bfloat16).to(DEV)
    wgu = (torch.randn(E, 2 * H, D, generator=gen) * 0.1).to(torch.bfloat16).to(DEV)
    p = torch.rand(R, generator=gen).to(DEV)
    guard = 4096                                     # elements of NaN bits before and after each output
    def padded(n):
        buf = torch.full((n + 2 * guard,), -1, dtype=torch.int16, device=DEV)   # 0xFFFF: a NaN
        return buf, buf[guard:guard + n].view(torch.bfloat16)
    dxb, dx = padded(R * 2 * H)
    xb_, xo = padded(R * 2 * H)
    ob, oo = padded(R * H)
    dp = torch.empty(R, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.time()
    sg.situ_glu_bwd_router_dgrad(x, dy, wt, off, p, dx.view(R, 2 * H), dp, status=st)
    h = dy                                           # [R, D] as the gate/up input
    sg.situ_glu_fwd_gateup(h, wgu, off, xo.view(R, 2 * H), oo.view(R, H), status=st)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30.0
    assert int(st.item()) == 0
    for buf, n in ((dxb, R * 2 * H), (xb_, R * 2 * H), (ob, R * H)):
        assert bool((buf[:guard] == -1).all()) and bool((buf[guard + n:] == -1).all())


def test_dgrad_dp_is_deterministic(sg):
    """Four CTAs share each M-tile as two clusters of two, and the two cluster sums meet in dp
    through atomic adds: two addends commute exactly, so repeated runs give bit-identical dp."""
    counts, H, D = CASES["real_widths"]
    x, dy, wt, off, p = make(counts, H, D, seed=77)
    runs = [run(sg, x, dy, wt, off, p) for _ in range(3)]
    for dx, dp in runs[1:]:
        assert torch.equal(dx.view(torch.int16), runs[0][0].view(torch.int16))
        assert torch.equal(dp.view(torch.int32), runs[0][1].view(torch.int32))


@pytest.mark.parametrize("name", ["partial_tiles", "empty_experts", "uneven_split", "real_widths", "large_experts",
                                  "n_tail_h272"])
def test_dgrad_nn_linear_weight_layout(sg, name):
    """W_down in its nn.Linear layout [E, D, H] (read N-major by the tensor cores) gives exactly
    the results of the transposed weights [E, H, D]; and both match the oracle."""
    counts, H, D = CASES[name]
    x, dy, wt, off, p = make(counts, H, D, seed=len(name) + 50)
    wd = wt.transpose(1, 2).contiguous()                      # [E, D, H]
    dx1, dp1 = run(sg, x, dy, wt, off, p)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    dx2, dp2 = sg.situ_glu_bwd_router_dgrad_wd(x.to(DEV), dy.to(DEV), wd.to(DEV), off.to(DEV), p.to(DEV),
                                               status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(dx1.view(torch.int16), dx2.view(torch.int16))
    assert torch.equal(dp1.view(torch.int32), dp2.view(torch.int32))
    dx_ref, dp_ref, dpa = oracle.dgrad_bwd_router(bits_of(x), bits_of(dy), bits_of(wt).reshape(wt.shape),
                                                 off.numpy(), p.numpy())
    par = Parity("dgrad nn.Linear layout " + name)
    par.bf16("dx", bits_of(dx2), dx_ref)
    par.dp(dp2.cpu().numpy(), dp_ref, dpa)
    par.assert_ok()

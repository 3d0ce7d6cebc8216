"""The library's host Adam update (the arithmetic of the streamed optimizer step) against the
oracle's stored-precision Adam, bit for bit: master fp32, both bf16 moments and the bf16 working
weight. Runs on the CPU: situ_adam_update_host makes no CUDA call. Argument validation of the
streamed entry point is checked here too (every call fails before any CUDA call)."""
import numpy as np
import pytest

import bwd_situ_glu_gb300 as sg
import oracle


@pytest.fixture(scope="module")
def lib():
    sg.build()
    return sg.load()


def bf16_bits(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def state(n, seed, g_scale_exp=(-6, 1)):
    rng = np.random.default_rng(seed)
    master = rng.normal(0, 0.02, n).astype(np.float32)
    m = bf16_bits(rng.normal(0, 1e-3, n))
    v = bf16_bits(rng.uniform(0, 1e-5, n))
    g = (rng.normal(0, 1, n) * 10.0 ** rng.uniform(*g_scale_exp, n)).astype(np.float32)
    return master, m, v, g


def run_lib(master, m, v, g, hp, nthreads=0):
    master, m, v = master.copy(), m.copy(), v.copy()
    w = np.zeros(master.size, dtype=np.uint16)
    sg.situ_adam_update_host(master, m, v, g, w, sg.adam_params(hp.lr, hp.beta1, hp.beta2, hp.eps,
                                                                hp.weight_decay, hp.step), nthreads)
    return master, m, v, w


def assert_same(a, b):
    for x, y, name in zip(a, b, ("master", "m", "v", "w_out")):
        assert np.array_equal(np.asarray(x).view(np.uint32 if x.dtype == np.float32 else np.uint16),
                              np.asarray(y).view(np.uint32 if y.dtype == np.float32 else np.uint16)), name


@pytest.mark.parametrize("lr,b1,b2,eps,wd,step", [
    (1e-3, 0.9, 0.999, 1e-8, 0.0, 1),
    (1e-3, 0.9, 0.999, 1e-8, 0.0, 10),
    (3e-4, 0.9, 0.95, 1e-8, 0.1, 1000),
    (1e-2, 0.5, 0.9, 0.1, 0.0, 3),
    (0.0, 0.9, 0.999, 1e-8, 0.0, 2),
])
def test_host_update_bit_exact(lib, lr, b1, b2, eps, wd, step):
    n = 100003
    master, m, v, g = state(n, seed=step)
    hp = oracle.adam_hp(lr, b1, b2, eps, wd, step)
    assert_same(run_lib(master, m, v, g, hp), oracle.adam_stored(master, m, v, g, hp))


def test_host_update_special_values(lib):
    """Zero gradients and moments, gradients from 1e-30 to 1e30 (g² overflowing to inf), exact
    zeros and a NaN gradient (propagates to its own element only)."""
    g = np.array([0.0, -0.0, 1e-30, -1e-30, 1e30, -1e30, 3.0, np.nan, 1e19, 65504.0], dtype=np.float32)
    n = g.size
    master = np.linspace(-1, 1, n).astype(np.float32)
    m = np.zeros(n, np.uint16)
    v = np.zeros(n, np.uint16)
    for step in (1, 2):
        hp = oracle.adam_hp(1e-3, 0.9, 0.999, 1e-8, 0.01, step)
        got = run_lib(master, m, v, g, hp)
        ref = oracle.adam_stored(master, m, v, g, hp)
        assert_same(got, ref)
        master, m, v = ref[0], ref[1], ref[2]


def test_host_update_many_steps_stay_identical(lib):
    """Twenty steps, each side evolving its own state from its own outputs: still identical."""
    n = 5000
    master, m, v, _ = state(n, seed=77)
    a = (master, m, v)
    b = (master, m, v)
    rng = np.random.default_rng(78)
    for step in range(1, 21):
        g = (rng.normal(0, 1, n) * 10.0 ** rng.uniform(-5, 0, n)).astype(np.float32)
        hp = oracle.adam_hp(1e-3, 0.9, 0.999, 1e-8, 0.01, step)
        ra = run_lib(*a, g, hp)
        rb = oracle.adam_stored(*b, g, hp)
        assert_same(ra, rb)
        a, b = ra[:3], rb[:3]


def test_host_update_thread_count_independent(lib):
    master, m, v, g = state(200001, seed=5)
    hp = oracle.adam_hp(1e-3, 0.9, 0.999, 1e-8, 0.0, 4)
    assert_same(run_lib(master, m, v, g, hp, nthreads=1), run_lib(master, m, v, g, hp, nthreads=7))


A = 1 << 20
B = 1 << 40


def test_host_update_validates(lib):
    P = sg.adam_params
    upd = lambda hp, n=8, ptrs=(A, A + 4096, A + 8192, A + 12288, A + 16384): lib.situ_adam_update_host(
        *ptrs, n, __import__("ctypes").byref(hp), 1)
    assert upd(P(), 0, (None,) * 5) == 0                              # n == 0 is a no-op
    for hp in (P(lr=-1.0), P(lr=float("nan")), P(beta1=1.0), P(beta2=-0.1), P(eps=0.0), P(eps=float("inf")),
               P(weight_decay=-1e-3), P(step=0)):
        assert upd(hp) == 1
    assert upd(P(), -1) == 1
    assert upd(P(), 8, (A, None, A + 8192, A + 12288, A + 16384)) == 1
    assert upd(P(), 8, (A + 2, A + 4096, A + 8192, A + 12288, A + 16384)) == 1     # master needs 4 bytes
    assert upd(P(), 8, (A, A + 4096 + 1, A + 8192, A + 12288, A + 16384)) == 1     # m needs 2 bytes
    assert upd(P(), 8, (A, A + 16, A + 8192, A + 12288, A + 16384)) == 2           # m over master
    assert upd(P(), 8, (A, A + 4096, A + 8192, A + 8192, A + 16384)) == 2          # g over v
    assert upd(P(), 8, (A, A + 4096, A + 8192, A + 12288, A + 4100)) == 2          # w_out over m


def test_stream_step_validates_before_any_cuda_call(lib):
    import ctypes
    P = sg.adam_params
    def step(hp=None, n=1000, chunk=128, nslots=2, ptrs=None):
        g, w = B, B + (1 << 20)
        master, m, v, st = A, A + (1 << 20), A + (2 << 20), A + (3 << 20)
        ptrs = ptrs or (g, w, master, m, v, st)
        hp = hp or P()
        return lib.situ_adam_stream_step(*ptrs[:5], n, ctypes.byref(hp), ptrs[5], chunk, nslots, 1, None)
    assert step(n=0, ptrs=(None,) * 6) == 0
    assert step(P(step=0)) == 1
    assert step(chunk=100) == 1                                      # chunk % 64
    assert step(chunk=0) == 1
    assert step(nslots=1) == 1
    assert step(nslots=65) == 1
    assert step(n=-5) == 1
    assert step(ptrs=(B, B + (1 << 20), A, A + (1 << 20), A + (2 << 20), A + (3 << 20) + 8)) == 1  # staging 16 B
    assert step(ptrs=(B, None, A, A + (1 << 20), A + (2 << 20), A + (3 << 20))) == 1
    assert step(ptrs=(B, B + 100, A, A + (1 << 20), A + (2 << 20), A + (3 << 20))) == 2           # weights over grads
    assert step(ptrs=(B, B + (1 << 20), A, A + 400, A + (2 << 20), A + (3 << 20))) == 2          # m over master
    assert step(ptrs=(B, B + (1 << 20), A, A + (1 << 20), A + (2 << 20), A + (2 << 20) + 64)) == 2  # staging over v

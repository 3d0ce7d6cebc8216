"""The streamed Adam step through the device: fp32 gradients on the GPU, optimizer state on the
host, new bf16 working weights back on the GPU, compared bit for bit with the oracle's
stored-precision Adam (the gradients the oracle sees are the same host copies)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sg(cuda_lib):
    assert torch.cuda.is_available()
    return cuda_lib


def pinned(nbytes):
    t = torch.empty(nbytes, dtype=torch.uint8)
    rc = torch.cuda.cudart().cudaHostRegister(t.data_ptr(), nbytes, 0)
    assert int(rc) == 0
    return t


def make(n, seed):
    rng = np.random.default_rng(seed)
    master = rng.normal(0, 0.02, n).astype(np.float32)
    m = torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    v = torch.from_numpy(rng.uniform(0, 1e-5, n).astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return master, m.copy(), v.copy()


def grads(n, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(n, generator=gen, device=DEV) * 10.0 ** (torch.rand(n, generator=gen, device=DEV) * 5 - 5)


@pytest.mark.parametrize("n,chunk,nslots", [(1_000_003, 65536, 2), (1_000_003, 131072, 3), (777, 1024, 2),
                                            (64 * 5, 64, 4), (3_000_000, 1 << 20, 8)])
def test_stream_step_bit_exact(sg, n, chunk, nslots):
    master, m, v = make(n, seed=n % 97)
    staging = pinned(sg.adam_staging_bytes(chunk, nslots))
    weight = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    ref = (master.copy(), m.copy(), v.copy())
    for step in (1, 2, 3):
        g = grads(n, seed=step)
        hp = oracle.adam_hp(1e-3, 0.9, 0.999, 1e-8, 0.01, step)
        sg.situ_adam_stream_step(g, weight, master, m, v, sg.adam_params(1e-3, 0.9, 0.999, 1e-8, 0.01, step),
                                 staging, chunk, nslots)
        torch.cuda.synchronize()
        rm, rmb, rvb, rw = oracle.adam_stored(*ref, g.cpu().numpy(), hp)
        assert np.array_equal(master.view(np.uint32), rm.view(np.uint32))
        assert np.array_equal(m, rmb) and np.array_equal(v, rvb)
        assert np.array_equal(weight.cpu().view(torch.int16).numpy().view(np.uint16), rw)
        ref = (rm, rmb, rvb)
    torch.cuda.cudart().cudaHostUnregister(staging.data_ptr())


def test_stream_step_orders_after_queued_work(sg):
    """The gradient copies follow the kernels already queued on the stream: gradients produced
    by a kernel launched just before (on the same stream) are the ones applied."""
    n, chunk = 500_000, 65536
    master, m, v = make(n, seed=3)
    staging = pinned(sg.adam_staging_bytes(chunk, 2))
    weight = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.zeros(n, device=DEV)
        torch.cuda._sleep(20_000_000)                    # a long kernel ahead of the gradients
        g.add_(0.5)
        sg.situ_adam_stream_step(g, weight, master, m, v, sg.adam_params(step=1), staging, chunk, 2, stream=s)
    ref = oracle.adam_stored(make(n, seed=3)[0], make(n, seed=3)[1], make(n, seed=3)[2],
                             np.full(n, 0.5, np.float32), oracle.adam_hp(step=1))
    assert np.array_equal(master.view(np.uint32), ref[0].view(np.uint32))
    torch.cuda.cudart().cudaHostUnregister(staging.data_ptr())


@pytest.mark.slow
def test_stream_step_bench_configuration_sampled(sg):
    """The configuration bench.py times: 2^28 parameters, chunks of 2^24, 2 slots, two chained
    steps; checked bit for bit on 2^20 sampled parameters plus every chunk boundary (the update
    is elementwise, so the oracle on the sample is the oracle of the whole)."""
    n, chunk, nslots = 1 << 28, 1 << 24, 2
    gen = torch.Generator(device=DEV).manual_seed(21)
    master = (torch.randn(n, generator=gen, device=DEV) * 0.02).cpu().numpy()
    m = (torch.randn(n, generator=gen, device=DEV) * 1e-3).to(torch.bfloat16).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    v = (torch.rand(n, generator=gen, device=DEV) * 1e-5).to(torch.bfloat16).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    rng = np.random.default_rng(22)
    edges = np.concatenate([np.arange(0, n, chunk), np.arange(chunk - 1, n, chunk), [n - 1]])
    idx = np.unique(np.concatenate([rng.integers(0, n, 1 << 20), edges]))
    ref = (master[idx].copy(), m[idx].copy(), v[idx].copy())
    staging = pinned(sg.adam_staging_bytes(chunk, nslots))
    weight = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    for step in (1, 2):
        g = grads(n, seed=100 + step)
        sg.situ_adam_stream_step(g, weight, master, m, v, sg.adam_params(step=step), staging, chunk, nslots)
        torch.cuda.synchronize()
        gi = g[torch.from_numpy(idx).to(DEV)].cpu().numpy()
        rm, rmb, rvb, rw = oracle.adam_stored(*ref, gi, oracle.adam_hp(step=step))
        assert np.array_equal(master[idx].view(np.uint32), rm.view(np.uint32))
        assert np.array_equal(m[idx], rmb) and np.array_equal(v[idx], rvb)
        wi = weight[torch.from_numpy(idx).to(DEV)].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(wi, rw)
        ref = (rm, rmb, rvb)
    torch.cuda.cudart().cudaHostUnregister(staging.data_ptr())
    del weight
    torch.cuda.empty_cache()

"""The failure path of the tensor-core kernels, exercised without faulting anything: a bounded
mbarrier wait (the helper every GEMM pipeline uses) runs out on a barrier nothing completes,
reports through the status word, and the kernel returns normally; the context stays usable."""
import time

import numpy as np
import pytest
import torch

import oracle
from _parity import Parity, bits_of

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sg(cuda_lib):
    assert torch.cuda.is_available()
    return cuda_lib


def test_bounded_wait_times_out_reports_and_returns(sg):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    elapsed = torch.zeros(1, dtype=torch.int64, device=DEV)
    t0 = time.time()
    sg.selftest_wait_timeout(status, elapsed)
    torch.cuda.synchronize()
    wall = time.time() - t0
    assert int(status.item()) == 1                        # gave up and said so (2 would mean it completed)
    ns = int(elapsed.item())
    assert 1.5e9 <= ns <= 20e9, ns                        # the ~2 s limit, not an endless spin
    assert wall < 60.0
    # the context is intact: an ordinary launch right after is correct
    gen = torch.Generator().manual_seed(3)
    x = (torch.randn(64, 512, generator=gen) * 3).to(torch.bfloat16)
    out = sg.situ_glu_fwd(x.to(DEV))
    torch.cuda.synchronize()
    par = Parity("after the timeout")
    par.bf16("out", bits_of(out), oracle.fwd_bf16(bits_of(x)))
    par.assert_ok()


def test_status_stays_zero_on_success(sg):
    """A successful fused launch never writes the status word (the caller's value stays)."""
    status = torch.full((1,), 0, dtype=torch.int32, device=DEV)
    gen = torch.Generator().manual_seed(4)
    h = torch.randn(200, 128, generator=gen).to(torch.bfloat16).to(DEV)
    w = (torch.randn(2, 256, 128, generator=gen) * 0.2).to(torch.bfloat16).to(DEV)
    off = torch.tensor([0, 150, 200], dtype=torch.int64, device=DEV)
    sg.situ_glu_fwd_gateup(h, w, off, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

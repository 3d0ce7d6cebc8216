"""The C ABI library loads, exports every function include/*.h declares, and rejects bad
arguments on the host before any CUDA call.

No test here launches a kernel: every call below fails validation first, so the
pointers are plain integers that are never dereferenced. (A fully valid set of
fake pointers would reach a launch; none is ever passed.)
"""
import glob
import os
import re

import pytest

import bwd_situ_glu_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, OVERLAP = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    sg.build()
    return sg.load()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(situ_glu_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("situ_glu_fwd", "situ_glu_bwd_router", "situ_glu_status_string", "situ_glu_version",
              "situ_glu_last_cuda_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert sg.version() == 10600
    for s in (0, 1, 2, 3, 99, -1):
        assert isinstance(sg.status_string(s), str) and sg.status_string(s)
    assert sg.status_string(0) == "ok"
    assert lib.situ_glu_last_cuda_error() == 0


A = 1 << 20  # fake, 16-byte aligned "device" addresses: never dereferenced
B = 1 << 40


def fwd(lib, x, out, R, H, beta=4.0, lbeta=25.0):
    return lib.situ_glu_fwd(x, out, R, H, beta, lbeta, None)


def bwd(lib, x, g, p, dx, dp, R, H, beta=4.0, lbeta=25.0):
    return lib.situ_glu_bwd_router(x, g, p, dx, dp, R, H, beta, lbeta, None)


def test_empty_is_a_noop(lib):
    assert fwd(lib, None, None, 0, 3072) == OK
    assert bwd(lib, None, None, None, None, None, 0, 3072) == OK


@pytest.mark.parametrize("R,H", [(-1, 8), (4, 0), (4, -8), (4, (1 << 30) + 1), (1 << 62, 3072)])
def test_bad_shapes(lib, R, H):
    assert fwd(lib, A, B, R, H) == INVALID
    assert bwd(lib, A, A + (1 << 36), A + (2 << 36), B, B + (1 << 36), R, H) == INVALID


@pytest.mark.parametrize("beta,lbeta", [(0.0, 25.0), (-4.0, 25.0), (4.0, 0.0), (float("nan"), 25.0),
                                        (4.0, float("inf")), (float("inf"), 25.0)])
def test_bad_scales(lib, beta, lbeta):
    assert fwd(lib, A, B, 4, 8, beta, lbeta) == INVALID
    assert bwd(lib, A, A + 4096, A + 8192, B, B + 4096, 4, 8, beta, lbeta) == INVALID


def test_null_pointers(lib):
    assert fwd(lib, None, B, 4, 8) == INVALID
    assert fwd(lib, A, None, 4, 8) == INVALID
    args = [A, A + 4096, A + 8192, B, B + 4096]
    for i in range(5):
        a = list(args)
        a[i] = None
        assert bwd(lib, *a, 4, 8) == INVALID


def test_misaligned_pointers(lib):
    assert fwd(lib, A + 1, B, 4, 8) == INVALID               # bf16 needs 2-byte alignment
    assert fwd(lib, A, B + 1, 4, 8) == INVALID
    assert bwd(lib, A, A + 4096, A + 8192 + 2, B, B + 4096, 4, 8) == INVALID   # p needs 4 bytes
    assert bwd(lib, A, A + 4096, A + 8192, B, B + 4096 + 2, 4, 8) == INVALID   # dp needs 4 bytes
    assert bwd(lib, A, A + 4096 + 1, A + 8192, B, B + 4096, 4, 8) == INVALID   # g


def test_forward_overlap(lib):
    R, H = 4, 8                      # x: 128 B, out: 64 B
    assert fwd(lib, A, A, R, H) == OVERLAP
    assert fwd(lib, A, A + 126, R, H) == OVERLAP
    assert fwd(lib, A + 62, A, R, H) == OVERLAP


def test_backward_overlap(lib):
    R, H = 4, 8                      # x, dx: 128 B; g: 64 B; p, dp: 16 B
    x, g, p = A, A + 4096, A + 8192
    dx, dp = B, B + 4096
    assert bwd(lib, x, g, p, x + 2, dp, R, H) == OVERLAP        # partial dx/x overlap
    assert bwd(lib, x, g, p, g, dp, R, H) == OVERLAP            # dx over g
    assert bwd(lib, x, g, p, p - 64, dp, R, H) == OVERLAP       # dx over p
    assert bwd(lib, x, g, p, dx, dx + 64, R, H) == OVERLAP      # dp inside dx
    assert bwd(lib, x, g, p, dx, x + 32, R, H) == OVERLAP       # dp over x
    assert bwd(lib, x, g, p, dx, g, R, H) == OVERLAP            # dp over g
    assert bwd(lib, x, g, p, dx, p, R, H) == OVERLAP            # dp over p
    # the in-place form dx == x passes the overlap checks; it must still not overlap g / p / dp
    assert bwd(lib, x, x + 64, p, x, dp, R, H) == OVERLAP       # g inside x == dx
    assert bwd(lib, x, g, p, x, x + 16, R, H) == OVERLAP        # dp inside x == dx


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib
    mod = importlib.import_module("bwd_situ_glu_gb300")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        mod.load()


def fwd8(lib, x, out, xq, xs, R, H, beta=4.0, lbeta=25.0):
    return lib.situ_glu_fwd_save_fp8(x, out, xq, xs, R, H, beta, lbeta, None)


def bwd8(lib, xq, xs, g, p, dx, dp, R, H, beta=4.0, lbeta=25.0):
    return lib.situ_glu_bwd_router_fp8(xq, xs, g, p, dx, dp, R, H, beta, lbeta, None)


def test_fp8_entry_points_validate_before_any_launch(lib):
    R, H = 4, 256                    # x 4096 B, out 2048 B, xq 2048 B, xs 4*2*2*4 = 64 B
    x, out, xq, xs = A, A + (1 << 16), A + (2 << 16), A + (3 << 16)
    assert fwd8(lib, None, None, None, None, 0, H) == OK
    assert fwd8(lib, x, out, xq, xs, -1, H) == INVALID
    assert fwd8(lib, x, out, xq, xs, R, 0) == INVALID
    assert fwd8(lib, x, out, xq, xs, R, H, 0.0) == INVALID
    assert fwd8(lib, x, out, None, xs, R, H) == INVALID
    assert fwd8(lib, x, out, xq, xs + 2, R, H) == INVALID      # scales need 4-byte alignment
    assert fwd8(lib, x + 1, out, xq, xs, R, H) == INVALID
    assert fwd8(lib, x, out, x + 100, xs, R, H) == OVERLAP     # codes over x
    assert fwd8(lib, x, out, xq, out + 64, R, H) == OVERLAP    # scales over out
    assert fwd8(lib, x, out, out + 1024, xs, R, H) == OVERLAP  # codes over out
    g, p, dx, dp = B, B + (1 << 16), B + (2 << 16), B + (3 << 16)
    assert bwd8(lib, None, None, None, None, None, None, 0, H) == OK
    assert bwd8(lib, xq, xs, g, p, dx, dp, R, -3) == INVALID
    assert bwd8(lib, xq, None, g, p, dx, dp, R, H) == INVALID
    assert bwd8(lib, xq, xs, g, p + 2, dx, dp, R, H) == INVALID
    assert bwd8(lib, xq, xs, g, p, xq, dp, R, H) == OVERLAP      # dx over the codes
    assert bwd8(lib, xq, xs, g, p, dx, xs, R, H) == OVERLAP      # dp over the scales
    assert bwd8(lib, xq, xs, g, p, dx, dx + 8, R, H) == OVERLAP  # dp inside dx


# ---------------------------------------------------------------- tensor-core entry points

def dgrad(lib, x, dy, wt, off, E, p, dx, dp, st, R, H, D, beta=4.0, lbeta=25.0):
    return lib.situ_glu_bwd_router_dgrad(x, dy, wt, off, E, p, dx, dp, st, R, H, D, beta, lbeta, None)


def gateup(lib, h, w, off, E, x, out, st, R, H, D, beta=4.0, lbeta=25.0):
    return lib.situ_glu_fwd_gateup(h, w, off, E, x, out, st, R, H, D, beta, lbeta, None)


def test_dgrad_validates_before_any_launch(lib):
    R, H, D, E = 4, 256, 64, 2       # x, dx 4 KB; dy 512 B; wt 64 KB
    x, dy, wt, off, p = A, A + (1 << 20), A + (2 << 20), A + (3 << 20), A + (4 << 20)
    dx, dp, st = B, B + (1 << 20), B + (2 << 20)
    args = [x, dy, wt, off, E, p, dx, dp, st]
    assert dgrad(lib, *[None] * 4, E, None, None, None, None, 0, H, D) == OK
    assert dgrad(lib, *args, R, 248, D) == INVALID                 # H % 16
    assert dgrad(lib, *args, R, H, 60) == INVALID                  # D % 8
    assert dgrad(lib, *args, R, H, 0) == INVALID
    assert dgrad(lib, *args, -1, H, D) == INVALID
    assert dgrad(lib, *args, R, H, D, 0.0) == INVALID
    for bad_e in (0, 4097):
        a = list(args)
        a[4] = bad_e
        assert dgrad(lib, *a, R, H, D) == INVALID
    for i in (0, 1, 2, 3, 5, 6, 7):                                # every pointer but status is required
        a = list(args)
        a[i] = None
        assert dgrad(lib, *a, R, H, D) == INVALID
    for i, misalign in ((0, 16), (6, 16), (1, 8), (2, 8), (3, 4), (5, 2), (7, 2), (8, 2)):
        a = list(args)
        a[i] += misalign                                            # x, dx need 32 B; dy, wt 16 B; ...
        assert dgrad(lib, *a, R, H, D) == INVALID, i
    assert dgrad(lib, x, dy, wt, off, E, p, x + 1024, dp, st, R, H, D) == OVERLAP      # dx over x
    assert dgrad(lib, x, dy, wt, off, E, p, dx, wt + 64, st, R, H, D) == OVERLAP      # dp over wt
    assert dgrad(lib, x, dy, wt, off, E, p, dx, dx + 512, st, R, H, D) == OVERLAP     # dp inside dx
    assert dgrad(lib, x, dy, wt, off, E, p, dx, dp, off, R, H, D) == OVERLAP          # status over offsets
    assert dgrad(lib, x, dy, wt, off, E, p, dx, dp, dx + 4, R, H, D) == OVERLAP       # status inside dx


def test_gateup_validates_before_any_launch(lib):
    R, H, D, E = 4, 128, 64, 2       # h 512 B; w 64 KB; x 2 KB; out 1 KB
    h, w, off = A, A + (1 << 20), A + (2 << 20)
    x, out, st = B, B + (1 << 20), B + (2 << 20)
    args = [h, w, off, E, x, out, st]
    assert gateup(lib, None, None, None, E, None, None, None, 0, H, D) == OK
    assert gateup(lib, *args, R, 120, D) == INVALID                # H % 16
    assert gateup(lib, *args, R, 8, D) == INVALID
    assert gateup(lib, *args, R, H, 36) == INVALID                 # D % 8
    assert gateup(lib, *args, -1, H, D) == INVALID
    assert gateup(lib, *args, R, H, D, 4.0, float("nan")) == INVALID
    for bad_e in (0, -1, 4097):
        a = list(args)
        a[3] = bad_e
        assert gateup(lib, *a, R, H, D) == INVALID
    for i in (0, 1, 2, 4, 5):                                      # every pointer but status is required
        a = list(args)
        a[i] = None
        assert gateup(lib, *a, R, H, D) == INVALID
    for i, misalign in ((0, 8), (1, 8), (2, 4), (4, 16), (5, 16), (6, 2)):
        a = list(args)
        a[i] += misalign                                            # h, w need 16 B; x, out 32 B; ...
        assert gateup(lib, *a, R, H, D) == INVALID, i
    assert gateup(lib, h, w, off, E, h + 256, out, st, R, H, D) == OVERLAP      # x over h
    assert gateup(lib, h, w, off, E, x, w + 1024, st, R, H, D) == OVERLAP      # out over w
    assert gateup(lib, h, w, off, E, x, x + 1024, st, R, H, D) == OVERLAP      # out inside x
    assert gateup(lib, h, w, off, E, x, off - 32, st, R, H, D) == OVERLAP      # out over offsets
    assert gateup(lib, h, w, off, E, x, out, out + 8, R, H, D) == OVERLAP      # status inside out


def test_selftest_validates(lib):
    assert lib.situ_glu_selftest_wait_timeout(None, None, None) == INVALID
    assert lib.situ_glu_selftest_wait_timeout(A + 2, None, None) == INVALID        # status needs 4 bytes
    assert lib.situ_glu_selftest_wait_timeout(A, A + 4, None) == INVALID           # elapsed needs 8 bytes


def test_dgrad_wd_validates_before_any_launch(lib):
    R, H, D, E = 4, 256, 64, 2
    x, dy, w, off, p = A, A + (1 << 20), A + (2 << 20), A + (3 << 20), A + (4 << 20)
    dx, dp, st = B, B + (1 << 20), B + (2 << 20)
    f = lambda *a: lib.situ_glu_bwd_router_dgrad_wd(*a, None)
    assert f(None, None, None, None, E, None, None, None, None, 0, H, D, 4.0, 25.0) == OK
    assert f(x, dy, w, off, E, p, dx, dp, st, R, 248, D, 4.0, 25.0) == INVALID          # H % 16
    assert f(x, dy, w, off, E, p, dx, dp, st, R, H, 96, 4.0, 25.0) == INVALID           # D % 64 (nn.Linear layout)
    assert f(x, dy, w + 8, off, E, p, dx, dp, st, R, H, D, 4.0, 25.0) == INVALID        # w 16-byte aligned
    assert f(x, dy, w, off, E, p, w + 64, dp, st, R, H, D, 4.0, 25.0) == OVERLAP        # dx over w

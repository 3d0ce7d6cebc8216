"""SiTU-GLU oracle: plain fp64 CPU restatement of the method (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package. The product path (``bwd_situ_glu_gb300``)
never imports it, and the two share no code.

The arithmetic lives in ``situ_glu_oracle.c`` (plain C, double, libm), which
states the formulas and cites the passages they come from:

* "Frontier-scale RL with Kimi K3", section "Streaming activations":
  the forward definition ``situ_and_mul``.
* "Kimi K3 模型结构（9）：显存", section "MoE 反向：推一下为什么可以不存 expert 输出":
  the router-gradient rewrite ``dL/dp_e = <W_down^T dL/dy, a_e>`` and
  ``dL/da_e = p_e W_down^T dL/dy``.

This module only compiles that file with gcc, loads it with ctypes and
marshals numpy arrays. Pins (closed forms, limits, finite differences,
brute-force tiny expert, the page's own code under autograd) live in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "situ_glu_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_situ_glu.so")
_lock = threading.Lock()
_lib = None

# The same flags on x86_64 and aarch64: no FMA contraction, no fast-math, so
# both machines evaluate exactly the expressions written in the C file.
FP8_BLOCK = 128  # elements per FP8 scale block (along a row, within each half)

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc) if missing or stale; return its path."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm", "-lpthread"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


class AdamHP(ctypes.Structure):
    """Adam hyper-parameters and the 1-based step count t (bias corrections 1 - beta^t)."""
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("step", ctypes.c_int64)]


def adam_hp(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=1) -> AdamHP:
    return AdamHP(lr, beta1, beta2, eps, weight_decay, step)


class Oracle:
    """ctypes wrapper over one build of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, dbl, vp, cint = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.oracle_situ_point.argtypes = [dbl, dbl, dbl, dbl, vp]
        lib.oracle_situ_point.restype = None
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = dbl
        lib.oracle_default_threads.argtypes = []
        lib.oracle_default_threads.restype = cint
        lib.oracle_situ_glu_fwd_f64.argtypes = [vp, vp, i64, i64, dbl, dbl, cint]
        lib.oracle_situ_glu_fwd_f64.restype = cint
        lib.oracle_situ_glu_bwd_router_f64.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, dbl, dbl, cint]
        lib.oracle_situ_glu_bwd_router_f64.restype = cint
        lib.oracle_situ_glu_fwd_bf16.argtypes = [vp, vp, i64, i64, dbl, dbl, cint]
        lib.oracle_situ_glu_fwd_bf16.restype = cint
        lib.oracle_situ_glu_bwd_router_bf16.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, dbl, dbl, cint]
        lib.oracle_situ_glu_bwd_router_bf16.restype = cint
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_float
        lib.oracle_quantize_fp8.argtypes = [vp, vp, vp, i64, i64, i64]
        lib.oracle_quantize_fp8.restype = cint
        lib.oracle_dequantize_fp8.argtypes = [vp, vp, vp, i64, i64, i64]
        lib.oracle_dequantize_fp8.restype = cint
        lib.oracle_round_bf16.argtypes = [dbl]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16_array.argtypes = [vp, vp, i64]
        lib.oracle_round_bf16_array.restype = cint
        lib.oracle_bf16_neighbours.argtypes = [dbl, vp, vp]
        lib.oracle_bf16_neighbours.restype = None
        lib.oracle_adam_f64.argtypes = [vp, vp, vp, vp, i64, ctypes.POINTER(AdamHP)]
        lib.oracle_adam_f64.restype = cint
        lib.oracle_adam_stored.argtypes = [vp, vp, vp, vp, vp, i64, ctypes.POINTER(AdamHP)]
        lib.oracle_adam_stored.restype = cint
        self.lib = lib
        self.path = path

    def default_threads(self) -> int:
        return int(self.lib.oracle_default_threads())

    def point(self, u: float, v: float, beta: float = 4.0, lbeta: float = 25.0):
        """(G, L, G', L') at one element pair, in double."""
        res = np.zeros(4, dtype=np.float64)
        self.lib.oracle_situ_point(float(u), float(v), float(beta), float(lbeta), _ptr(res))
        return tuple(float(t) for t in res)

    def bf16_to_double(self, bits: int) -> float:
        return float(self.lib.oracle_bf16_to_double(int(bits) & 0xFFFF))

    def fwd_f64(self, x: np.ndarray, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0) -> np.ndarray:
        """out[R,H] = G(gate)·L(linear) in double, from an fp64 x [R,2H]."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        R, H2 = x.shape
        assert H2 % 2 == 0
        out = np.empty((R, H2 // 2), dtype=np.float64)
        _check(self.lib.oracle_situ_glu_fwd_f64(_ptr(x), _ptr(out), R, H2 // 2, beta, lbeta, nthreads))
        return out

    def bwd_router_f64(self, x, g, p, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0):
        """(dx [R,2H], dp [R], dp_abs [R]) in double from fp64 x [R,2H], g [R,H], p [R]."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        g = np.ascontiguousarray(g, dtype=np.float64)
        p = np.ascontiguousarray(p, dtype=np.float64)
        R, H2 = x.shape
        H = H2 // 2
        assert g.shape == (R, H) and p.shape == (R,)
        dx = np.empty((R, H2), dtype=np.float64)
        dp = np.empty((R,), dtype=np.float64)
        dpa = np.empty((R,), dtype=np.float64)
        _check(self.lib.oracle_situ_glu_bwd_router_f64(_ptr(x), _ptr(g), _ptr(p), _ptr(dx), _ptr(dp), _ptr(dpa),
                                                       R, H, beta, lbeta, nthreads))
        return dx, dp, dpa

    def fwd_bf16(self, x_bits: np.ndarray, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0) -> np.ndarray:
        """Forward on bf16 storage bits (uint16 [R,2H]); unrounded double result [R,H]."""
        x_bits = np.ascontiguousarray(x_bits).view(np.uint16)
        R, H2 = x_bits.shape
        assert H2 % 2 == 0
        out = np.empty((R, H2 // 2), dtype=np.float64)
        _check(self.lib.oracle_situ_glu_fwd_bf16(_ptr(x_bits), _ptr(out), R, H2 // 2, beta, lbeta, nthreads))
        return out

    def bwd_router_bf16(self, x_bits, g_bits, p, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0):
        """Backward with the router rewrite on bf16 bits x [R,2H], g [R,H] and fp32 p [R].

        Returns unrounded double (dx [R,2H], dp [R], dp_abs [R]) where
        dp_abs = Σ_j |g_j·a_j|."""
        x_bits = np.ascontiguousarray(x_bits).view(np.uint16)
        g_bits = np.ascontiguousarray(g_bits).view(np.uint16)
        p = np.ascontiguousarray(p, dtype=np.float32)
        R, H2 = x_bits.shape
        H = H2 // 2
        assert g_bits.shape == (R, H) and p.shape == (R,)
        dx = np.empty((R, H2), dtype=np.float64)
        dp = np.empty((R,), dtype=np.float64)
        dpa = np.empty((R,), dtype=np.float64)
        _check(self.lib.oracle_situ_glu_bwd_router_bf16(_ptr(x_bits), _ptr(g_bits), _ptr(p), _ptr(dx), _ptr(dp),
                                                        _ptr(dpa), R, H, beta, lbeta, nthreads))
        return dx, dp, dpa


    # ---------------- block-wise FP8 saved x ----------------

    def e4m3_encode(self, v: float) -> int:
        """OCP E4M3 code of fp32 v: round to nearest (ties to even code), saturate to +-448."""
        return int(self.lib.oracle_e4m3_encode(float(v)))

    def e4m3_decode(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_decode(int(code) & 0xFF))

    def quantize_fp8(self, x_bits, block: int = FP8_BLOCK):
        """bf16 bits x [R,2H] -> (codes uint8 [R,2H], scales fp32 [R, 2*ceil(H/block)])."""
        x_bits = np.ascontiguousarray(x_bits).view(np.uint16)
        R, H2 = x_bits.shape
        H = H2 // 2
        nb = -(-H // block)
        q = np.empty((R, H2), dtype=np.uint8)
        sc = np.empty((R, 2 * nb), dtype=np.float32)
        _check(self.lib.oracle_quantize_fp8(_ptr(x_bits), _ptr(q), _ptr(sc), R, H, block))
        return q, sc

    def dequantize_fp8(self, q, sc, block: int = FP8_BLOCK):
        """(codes [R,2H], scales [R,2nb]) -> x^ fp32 [R,2H] = decode(code) * scale."""
        q = np.ascontiguousarray(q, dtype=np.uint8)
        sc = np.ascontiguousarray(sc, dtype=np.float32)
        R, H2 = q.shape
        xh = np.empty((R, H2), dtype=np.float32)
        _check(self.lib.oracle_dequantize_fp8(_ptr(q), _ptr(sc), _ptr(xh), R, H2 // 2, block))
        return xh

    def bwd_router_fp8(self, q, sc, g_bits, p, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0,
                       block: int = FP8_BLOCK):
        """Backward with the router rewrite from the FP8-saved x: the definition evaluated on
        x^ = decode(q) * s (fp32, widened exactly to double)."""
        xh = self.dequantize_fp8(q, sc, block).astype(np.float64)
        g = (np.ascontiguousarray(g_bits).view(np.uint16).astype(np.uint32) << 16).view(np.float32)
        return self.bwd_router_f64(xh, g.astype(np.float64), np.asarray(p, dtype=np.float32).astype(np.float64),
                                   beta, lbeta, nthreads)


    # ---------------- bf16 rounding of exact values ----------------

    def round_bf16(self, v: float) -> int:
        """bf16 bits of v rounded to nearest, ties to even (IEEE roundTiesToEven)."""
        return int(self.lib.oracle_round_bf16(float(v)))

    def round_bf16_array(self, v) -> np.ndarray:
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(v.shape, dtype=np.uint16)
        _check(self.lib.oracle_round_bf16_array(_ptr(v), _ptr(out), v.size))
        return out

    def bf16_neighbours(self, v: float):
        """(lo, hi) bf16 bits with lo <= v <= hi, consecutive or equal."""
        lo = np.zeros(1, dtype=np.uint16)
        hi = np.zeros(1, dtype=np.uint16)
        self.lib.oracle_bf16_neighbours(float(v), _ptr(lo), _ptr(hi))
        return int(lo[0]), int(hi[0])

    # ---------------- Adam on host-resident optimizer state ----------------

    def adam_f64(self, w, m, v, g, hp: AdamHP):
        """One textbook Adam step in double on double state; returns new (w, m, v)."""
        w = np.array(w, dtype=np.float64, copy=True)
        m = np.array(m, dtype=np.float64, copy=True)
        v = np.array(v, dtype=np.float64, copy=True)
        g = np.ascontiguousarray(g, dtype=np.float64)
        _check(self.lib.oracle_adam_f64(_ptr(w), _ptr(m), _ptr(v), _ptr(g), w.size, ctypes.byref(hp)))
        return w, m, v

    def adam_stored(self, master, m_bits, v_bits, g, hp: AdamHP):
        """One Adam step on the stored precisions (fp32 master, bf16 moments, fp32 gradient);
        returns new (master fp32, m bits, v bits, working-weight bf16 bits)."""
        master = np.array(master, dtype=np.float32, copy=True)
        m = np.array(np.asarray(m_bits).view(np.uint16), dtype=np.uint16, copy=True)
        v = np.array(np.asarray(v_bits).view(np.uint16), dtype=np.uint16, copy=True)
        g = np.ascontiguousarray(g, dtype=np.float32)
        w = np.empty(master.shape, dtype=np.uint16)
        _check(self.lib.oracle_adam_stored(_ptr(master), _ptr(m), _ptr(v), _ptr(g), _ptr(w), master.size,
                                           ctypes.byref(hp)))
        return master, m, v, w

    # ---------------- fused gate/up projection forward ----------------

    @staticmethod
    def grouped_gateup(h_bits, w_bits, offsets):
        return grouped_gateup(h_bits, w_bits, offsets)

    def gateup_fwd(self, h_bits, w_bits, offsets, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0):
        """The gate/up projection with the SiTU-GLU forward after it: x (exact, double), its bf16
        bits (rounded to nearest even: the saved tensor), out = G(gate)·L(linear) in double from
        those bf16 values (the forward reads the saved bf16 x), and the accumulation scale of x."""
        x, mag = grouped_gateup(h_bits, w_bits, offsets)
        xb = self.round_bf16_array(x)
        out = self.fwd_bf16(xb, beta, lbeta, nthreads)
        return x, xb, out, mag


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check(rc: int):
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")


def _default() -> Oracle:
    global _lib
    if _lib is None:
        build()
        _lib = Oracle(_LIB)
    return _lib


def compile_variant(src_text: str, out_path: str) -> Oracle:
    """Compile C source text with the oracle's flags into out_path and load it (used by tests)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *GCC_FLAGS, "-o", out_path, src, "-lm", "-lpthread"], check=True)
    return Oracle(out_path)


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def default_threads() -> int:
    return _default().default_threads()


def point(u: float, v: float, beta: float = 4.0, lbeta: float = 25.0):
    return _default().point(u, v, beta, lbeta)


def bf16_to_double(bits: int) -> float:
    return _default().bf16_to_double(bits)


def fwd_f64(x, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0):
    return _default().fwd_f64(x, beta, lbeta, nthreads)


def bwd_router_f64(x, g, p, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0):
    return _default().bwd_router_f64(x, g, p, beta, lbeta, nthreads)


def fwd_bf16(x_bits, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0):
    return _default().fwd_bf16(x_bits, beta, lbeta, nthreads)


def bwd_router_bf16(x_bits, g_bits, p, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0):
    return _default().bwd_router_bf16(x_bits, g_bits, p, beta, lbeta, nthreads)


def e4m3_encode(v: float) -> int:
    return _default().e4m3_encode(v)


def e4m3_decode(code: int) -> float:
    return _default().e4m3_decode(code)


def quantize_fp8(x_bits, block: int = FP8_BLOCK):
    return _default().quantize_fp8(x_bits, block)


def dequantize_fp8(q, sc, block: int = FP8_BLOCK):
    return _default().dequantize_fp8(q, sc, block)


def bwd_router_fp8(q, sc, g_bits, p, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0,
                   block: int = FP8_BLOCK):
    return _default().bwd_router_fp8(q, sc, g_bits, p, beta, lbeta, nthreads, block)


# ---------------------------------------------------------------- fused down-projection dgrad

def grouped_dgrad(dy_bits, wt_bits, offsets):
    """g = dY·W_down per expert, in double: rows offsets[e]..offsets[e+1] of dY (bf16 bits
    [R, D]) times W_down of expert e, given as its transpose wt_bits[e] = W_downᵀ (bf16 bits
    [H, D]), so g[r, j] = Σ_d dY[r, d]·W_down,e[d, j] = Σ_d dY[r, d]·wt[e, j, d].

    "Kimi K3 模型结构（9）：显存", section "MoE 反向…": (W_down,e)ᵀ·dL/dy is the quantity the
    backward already computes on its way to a_e; here it is formed with numpy's fp64 matmul."""
    dy = (np.ascontiguousarray(dy_bits).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wt = (np.ascontiguousarray(wt_bits).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    E, H, D = wt.shape
    assert dy.shape[1] == D and offsets.shape == (E + 1,) and offsets[0] == 0 and offsets[-1] == dy.shape[0]
    g = np.zeros((dy.shape[0], H), dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            g[a:b] = dy[a:b] @ wt[e].T
    return g


def dgrad_bwd_router(x_bits, dy_bits, wt_bits, offsets, p, beta: float = 4.0, lbeta: float = 25.0,
                     nthreads: int = 0):
    """Fused down-projection dgrad + SiTU-GLU backward + router gradient, in double:
    g = grouped_dgrad(dY, W_downᵀ), then the backward of bwd_router_f64 at g (never rounded)."""
    g = grouped_dgrad(dy_bits, wt_bits, offsets)
    x = (np.ascontiguousarray(x_bits).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return _default().bwd_router_f64(x, g, np.asarray(p, dtype=np.float32).astype(np.float64), beta, lbeta, nthreads)


# ---------------------------------------------------------------- fused gate/up projection forward

def round_bf16(v: float) -> int:
    return _default().round_bf16(v)


def round_bf16_array(v) -> np.ndarray:
    return _default().round_bf16_array(v)


def bf16_neighbours(v: float):
    return _default().bf16_neighbours(v)


def grouped_gateup(h_bits, w_bits, offsets):
    """x = [W_gate,e·h | W_up,e·h] per routed row, in double: rows offsets[e]..offsets[e+1] of
    h (bf16 bits [R, D], the expert's dispatched inputs) times expert e's stacked weights
    w_bits[e] (bf16 bits [2H, D]: rows 0..H-1 are W_gate,e, rows H..2H-1 are W_up,e), so
    x[r, n] = Σ_d h[r, d]·w[e, n, d]. Also returns Σ_d |h[r, d]·w[e, n, d]|, the scale of the
    fp32 accumulation error of any summation order.

    "Kimi K3 模型结构（9）：显存", section "MoE 反向…": a_e = SiTU(W_gate,e x_e, W_up,e x_e);
    the two projections are formed here with numpy's fp64 matmul."""
    h = (np.ascontiguousarray(h_bits).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = (np.ascontiguousarray(w_bits).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    offsets = np.asarray(offsets, dtype=np.int64)
    E, H2, D = w.shape
    assert h.shape[1] == D and offsets.shape == (E + 1,) and offsets[0] == 0 and offsets[-1] == h.shape[0]
    x = np.zeros((h.shape[0], H2), dtype=np.float64)
    mag = np.zeros((h.shape[0], H2), dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            x[a:b] = h[a:b] @ w[e].T
            mag[a:b] = np.abs(h[a:b]) @ np.abs(w[e]).T
    return x, mag


def gateup_fwd(h_bits, w_bits, offsets, beta: float = 4.0, lbeta: float = 25.0, nthreads: int = 0):
    return _default().gateup_fwd(h_bits, w_bits, offsets, beta, lbeta, nthreads)


# ---------------------------------------------------------------- Adam on host-resident state

def adam_f64(w, m, v, g, hp: AdamHP):
    return _default().adam_f64(w, m, v, g, hp)


def adam_stored(master, m_bits, v_bits, g, hp: AdamHP):
    return _default().adam_stored(master, m_bits, v_bits, g, hp)

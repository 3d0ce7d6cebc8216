"""bwd_situ_glu_gb300 — SiTU-GLU forward and fused backward + router gradient on GB300.

Thin Python binding over the C ABI in ``include/situ_glu.h`` (``libsitu_glu.so``,
built in-tree from ``csrc/`` for sm_103a). Every step of the computation runs in
the library's CUDA kernels; this module only checks tensor metadata, marshals
pointers and raises on a non-zero status. There is no CPU fallback: if the
library is missing or cannot load, every call raises.

Binding names match the C entry points:

* ``situ_glu_fwd(x, out=None, beta=4.0, lbeta=25.0, stream=None) -> out``
* ``situ_glu_bwd_router(x, g, p, dx=None, dp=None, beta=4.0, lbeta=25.0, stream=None) -> (dx, dp)``
* ``situ_glu_fwd_save_fp8`` / ``situ_glu_bwd_router_fp8``: the same with x saved as block-wise
  FP8 (E4M3 codes + fp32 scales of 128-element blocks)
* ``situ_glu_bwd_router_dgrad`` / ``situ_glu_bwd_router_dgrad_wd``: g = dY·W_down,e per expert on
  the tensor cores with the backward in the GEMM's epilogue (weights [E, H, D] or [E, D, H])
* ``situ_glu_fwd_gateup``: x = [W_gate,e·h | W_up,e·h] per expert on the tensor cores with the
  forward in the GEMM's epilogue
* ``situ_adam_update_host`` / ``situ_adam_stream_step``: Adam on host-resident state, the
  streamed form moving gradients and weights chunk by chunk
* ``situ_and_mul(x, beta, linear_beta)``: autograd function (forward kernel; backward kernel
  with p = 1), the pages' operator interface

Shapes: ``x`` bf16 [R, 2H] (gate | linear), ``g`` bf16 [R, H], ``p`` fp32 [R];
``out`` bf16 [R, H], ``dx`` bf16 [R, 2H], ``dp`` fp32 [R]. All on one CUDA device.
``dx`` may be ``x`` itself (in-place backward).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
CSRC = os.path.join(_HERE, "csrc")
INCLUDE = os.path.join(_ROOT, "include")
LIB_DIR = os.path.join(_HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libsitu_glu.so")
SOURCES = [os.path.join(CSRC, n) for n in ("situ_glu.cu", "situ_glu_fp8.cu", "situ_glu_dgrad.cu",
                                             "situ_glu_gateup.cu", "situ_adam.cu", "situ_glu_selftest.cu")]
# per-source extra flags: the host Adam update is a fixed sequence of IEEE fp32 operations
SOURCE_FLAGS = {"situ_adam.cu": ["-Xcompiler", "-ffp-contract=off,-fno-fast-math,-fno-math-errno"]}
DEPENDS = SOURCES + [os.path.join(CSRC, n) for n in ("situ_math.cuh", "situ_device.cuh", "situ_host.h",
                                                     "situ_tc.cuh")] + [os.path.join(INCLUDE, "situ_glu.h")]

NVCC_FLAGS = [
    "-std=c++17", "-O3", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC", "-shared",
]

STATUS_OK, STATUS_INVALID_ARG, STATUS_OVERLAP, STATUS_CUDA_ERROR = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


class AdamParams(ctypes.Structure):
    """situ_adam_params: Adam hyper-parameters and the 1-based step count of the update."""
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("step", ctypes.c_int64)]


def adam_params(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=1) -> AdamParams:
    return AdamParams(lr, beta1, beta2, eps, weight_decay, step)


class SituGluError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"situ_glu status {status}: {msg}")
        self.status = status


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``libsitu_glu.so`` in-tree for sm_103a if missing or older than its sources."""
    with _lock:
        os.makedirs(LIB_DIR, exist_ok=True)
        newest = max(os.path.getmtime(p) for p in DEPENDS)
        if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < newest:
            # one object per translation unit, compiled in parallel, then one link
            tag = f".tmp{os.getpid()}"
            objs, procs = [], []
            for src in SOURCES:
                obj = os.path.join(LIB_DIR, os.path.basename(src) + tag + ".o")
                cmd = [_nvcc(), *[f for f in NVCC_FLAGS if f != "-shared"],
                       *SOURCE_FLAGS.get(os.path.basename(src), []), "-I", INCLUDE, "-c", "-o", obj, src]
                if verbose:
                    cmd.insert(1, "-Xptxas=-v")
                objs.append(obj)
                procs.append((subprocess.Popen(cmd), cmd))
            failed = [cmd for proc, cmd in procs if proc.wait() != 0]
            try:
                if failed:
                    raise subprocess.CalledProcessError(1, failed[0])
                tmp = LIB_PATH + tag
                subprocess.run([_nvcc(), *NVCC_FLAGS, "-o", tmp, *objs], check=True)
                os.replace(tmp, LIB_PATH)
            finally:
                for obj in objs:
                    if os.path.exists(obj):
                        os.remove(obj)
    return LIB_PATH


def load():
    """Load the CUDA library (does not compile). Raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing (run bwd_situ_glu_gb300.build())")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, f32, cint = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    lib.situ_glu_fwd.argtypes = [vp, vp, i64, i64, f32, f32, vp]
    lib.situ_glu_fwd.restype = cint
    lib.situ_glu_bwd_router.argtypes = [vp, vp, vp, vp, vp, i64, i64, f32, f32, vp]
    lib.situ_glu_bwd_router.restype = cint
    lib.situ_glu_fwd_save_fp8.argtypes = [vp, vp, vp, vp, i64, i64, f32, f32, vp]
    lib.situ_glu_fwd_save_fp8.restype = cint
    lib.situ_glu_bwd_router_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, f32, f32, vp]
    lib.situ_glu_bwd_router_fp8.restype = cint
    lib.situ_glu_bwd_router_dgrad.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, i64, i64, i64, f32, f32, vp]
    lib.situ_glu_bwd_router_dgrad.restype = cint
    lib.situ_glu_bwd_router_dgrad_wd.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, i64, i64, i64, f32, f32, vp]
    lib.situ_glu_bwd_router_dgrad_wd.restype = cint
    lib.situ_glu_fwd_gateup.argtypes = [vp, vp, vp, i64, vp, vp, vp, i64, i64, i64, f32, f32, vp]
    lib.situ_glu_fwd_gateup.restype = cint
    lib.situ_glu_selftest_wait_timeout.argtypes = [vp, vp, vp]
    lib.situ_glu_selftest_wait_timeout.restype = cint
    lib.situ_adam_update_host.argtypes = [vp, vp, vp, vp, vp, i64, ctypes.POINTER(AdamParams), cint]
    lib.situ_adam_update_host.restype = cint
    lib.situ_adam_stream_step.argtypes = [vp, vp, vp, vp, vp, i64, ctypes.POINTER(AdamParams), vp, i64, cint, cint,
                                          vp]
    lib.situ_adam_stream_step.restype = cint
    lib.situ_glu_status_string.argtypes = [cint]
    lib.situ_glu_status_string.restype = ctypes.c_char_p
    lib.situ_glu_last_cuda_error.argtypes = []
    lib.situ_glu_last_cuda_error.restype = cint
    lib.situ_glu_version.argtypes = []
    lib.situ_glu_version.restype = cint
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().situ_glu_status_string(int(status)).decode()


def version() -> int:
    return int(load().situ_glu_version())


def _check(status: int):
    if status != STATUS_OK:
        msg = status_string(status)
        if status == STATUS_CUDA_ERROR:
            msg += f" (cudaError {load().situ_glu_last_cuda_error()})"
        raise SituGluError(status, msg)


# ---------------- raw pointer calls (ints are device addresses) ----------------

def situ_glu_fwd_ptr(x: int, out: int, R: int, H: int, beta: float = 4.0, lbeta: float = 25.0,
                     stream: int = 0) -> None:
    _check(load().situ_glu_fwd(x, out, R, H, beta, lbeta, stream))


def situ_glu_bwd_router_ptr(x: int, g: int, p: int, dx: int, dp: int, R: int, H: int, beta: float = 4.0,
                            lbeta: float = 25.0, stream: int = 0) -> None:
    _check(load().situ_glu_bwd_router(x, g, p, dx, dp, R, H, beta, lbeta, stream))


# ---------------- torch tensor calls ----------------

def _need(t, dtype, shape, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream, device) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def situ_glu_fwd(x, out=None, beta: float = 4.0, lbeta: float = 25.0, stream=None):
    """out[R,H] (bf16) = SiTU-GLU(x[R,2H] bf16). Enqueued on ``stream`` (default: current)."""
    import torch
    if x.dim() != 2 or x.shape[1] % 2 != 0:
        raise ValueError("x must be [R, 2H]")
    R, H = x.shape[0], x.shape[1] // 2
    _need(x, torch.bfloat16, (R, 2 * H), "x")
    if out is None:
        out = torch.empty((R, H), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (R, H), "out")
    if out.device != x.device:
        raise ValueError("x and out must be on the same device")
    with torch.cuda.device(x.device):
        situ_glu_fwd_ptr(x.data_ptr(), out.data_ptr(), R, H, beta, lbeta, _stream_handle(stream, x.device))
    return out


def situ_glu_bwd_router(x, g, p, dx=None, dp=None, beta: float = 4.0, lbeta: float = 25.0, stream=None):
    """(dx[R,2H] bf16, dp[R] fp32) of the fused backward + router gradient. ``dx`` may be ``x``."""
    import torch
    if x.dim() != 2 or x.shape[1] % 2 != 0:
        raise ValueError("x must be [R, 2H]")
    R, H = x.shape[0], x.shape[1] // 2
    _need(x, torch.bfloat16, (R, 2 * H), "x")
    _need(g, torch.bfloat16, (R, H), "g")
    _need(p, torch.float32, (R,), "p")
    if dx is None:
        dx = torch.empty((R, 2 * H), dtype=torch.bfloat16, device=x.device)
    if dp is None:
        dp = torch.empty((R,), dtype=torch.float32, device=x.device)
    _need(dx, torch.bfloat16, (R, 2 * H), "dx")
    _need(dp, torch.float32, (R,), "dp")
    if len({t.device for t in (x, g, p, dx, dp)}) != 1:
        raise ValueError("all tensors must be on the same device")
    with torch.cuda.device(x.device):
        situ_glu_bwd_router_ptr(x.data_ptr(), g.data_ptr(), p.data_ptr(), dx.data_ptr(), dp.data_ptr(), R, H,
                                beta, lbeta, _stream_handle(stream, x.device))
    return dx, dp


FP8_BLOCK = 128  # elements per FP8 scale block (SITU_GLU_FP8_BLOCK)


def fp8_scale_blocks(H: int) -> int:
    return -(-H // FP8_BLOCK)


_SituAndMul = None


def _situ_and_mul_fn():
    """The autograd Function, created on first use (torch is imported lazily by this module)."""
    global _SituAndMul
    if _SituAndMul is None:
        import torch

        class SituAndMul(torch.autograd.Function):
            """SiTU-GLU as an autograd operator that keeps only the bf16 input for the backward
            ("Frontier-scale RL with Kimi K3", section "Streaming activations": the custom
            operator drops every tensor but x and recomputes tanh and sigmoid). Forward: the
            forward kernel. Backward: the fused backward kernel with a unit router weight, so
            dL/dx = dL/da · da/dx (its router gradient, <dL/da, a>, is not needed here)."""

            @staticmethod
            def forward(ctx, x, beta, lbeta):
                ctx.save_for_backward(x)
                ctx.beta, ctx.lbeta = beta, lbeta
                return situ_glu_fwd(x, beta=beta, lbeta=lbeta)

            @staticmethod
            def backward(ctx, grad_out):
                (x,) = ctx.saved_tensors
                g = grad_out.contiguous()
                ones = torch.ones(x.shape[0], dtype=torch.float32, device=x.device)
                dx, _ = situ_glu_bwd_router(x, g, ones, beta=ctx.beta, lbeta=ctx.lbeta)
                return dx, None, None

        _SituAndMul = SituAndMul
    return _SituAndMul


def situ_and_mul(x, beta: float = 4.0, linear_beta: float = 25.0):
    """a = beta·tanh(gate/beta)·sigmoid(gate) · linear_beta·tanh(linear/linear_beta) for
    x = [gate | linear] (bf16 [R, 2H] on the GPU), differentiable; only x is kept for the
    backward. The same interface as the pages' custom operator, on this library's kernels."""
    return _situ_and_mul_fn().apply(x, float(beta), float(linear_beta))


def situ_glu_fwd_save_fp8(x, out=None, xq=None, xs=None, beta: float = 4.0, lbeta: float = 25.0, stream=None):
    """(out bf16 [R,H], xq uint8 [R,2H], xs fp32 [R,2*nb]): the forward plus x saved in block-wise FP8."""
    import torch
    if x.dim() != 2 or x.shape[1] % 2 != 0:
        raise ValueError("x must be [R, 2H]")
    R, H = x.shape[0], x.shape[1] // 2
    nb = fp8_scale_blocks(H)
    _need(x, torch.bfloat16, (R, 2 * H), "x")
    if out is None:
        out = torch.empty((R, H), dtype=torch.bfloat16, device=x.device)
    if xq is None:
        xq = torch.empty((R, 2 * H), dtype=torch.uint8, device=x.device)
    if xs is None:
        xs = torch.empty((R, 2 * nb), dtype=torch.float32, device=x.device)
    _need(out, torch.bfloat16, (R, H), "out")
    _need(xq, torch.uint8, (R, 2 * H), "xq")
    _need(xs, torch.float32, (R, 2 * nb), "xs")
    if len({t.device for t in (x, out, xq, xs)}) != 1:
        raise ValueError("all tensors must be on the same device")
    with torch.cuda.device(x.device):
        _check(load().situ_glu_fwd_save_fp8(x.data_ptr(), out.data_ptr(), xq.data_ptr(), xs.data_ptr(), R, H,
                                            beta, lbeta, _stream_handle(stream, x.device)))
    return out, xq, xs


def situ_glu_bwd_router_fp8(xq, xs, g, p, dx=None, dp=None, beta: float = 4.0, lbeta: float = 25.0, stream=None):
    """(dx bf16 [R,2H], dp fp32 [R]) of the fused backward + router gradient from the FP8-saved x."""
    import torch
    if xq.dim() != 2 or xq.shape[1] % 2 != 0:
        raise ValueError("xq must be [R, 2H]")
    R, H = xq.shape[0], xq.shape[1] // 2
    nb = fp8_scale_blocks(H)
    _need(xq, torch.uint8, (R, 2 * H), "xq")
    _need(xs, torch.float32, (R, 2 * nb), "xs")
    _need(g, torch.bfloat16, (R, H), "g")
    _need(p, torch.float32, (R,), "p")
    if dx is None:
        dx = torch.empty((R, 2 * H), dtype=torch.bfloat16, device=xq.device)
    if dp is None:
        dp = torch.empty((R,), dtype=torch.float32, device=xq.device)
    _need(dx, torch.bfloat16, (R, 2 * H), "dx")
    _need(dp, torch.float32, (R,), "dp")
    if len({t.device for t in (xq, xs, g, p, dx, dp)}) != 1:
        raise ValueError("all tensors must be on the same device")
    with torch.cuda.device(xq.device):
        _check(load().situ_glu_bwd_router_fp8(xq.data_ptr(), xs.data_ptr(), g.data_ptr(), p.data_ptr(), dx.data_ptr(),
                                              dp.data_ptr(), R, H, beta, lbeta, _stream_handle(stream, xq.device)))
    return dx, dp


def situ_glu_bwd_router_dgrad(x, dy, w_down_t, expert_offsets, p, dx=None, dp=None, status=None, beta: float = 4.0,
                              lbeta: float = 25.0, stream=None):
    """(dx bf16 [R,2H], dp fp32 [R]) from dY [R,D] and the experts' W_downᵀ [E,H,D]: the dgrad GEMM
    g = dY·W_down,e on the tensor cores with the backward + router gradient fused into it.
    ``status`` (int32 [1] on the device, zeroed by the caller) turns 1 if a pipeline wait timed out."""
    import torch
    if x.dim() != 2 or x.shape[1] % 2 != 0:
        raise ValueError("x must be [R, 2H]")
    R, H = x.shape[0], x.shape[1] // 2
    if w_down_t.dim() != 3:
        raise ValueError("w_down_t must be [E, H, D]")
    E, D = w_down_t.shape[0], w_down_t.shape[2]
    _need(x, torch.bfloat16, (R, 2 * H), "x")
    _need(dy, torch.bfloat16, (R, D), "dy")
    _need(w_down_t, torch.bfloat16, (E, H, D), "w_down_t")
    _need(expert_offsets, torch.int64, (E + 1,), "expert_offsets")
    _need(p, torch.float32, (R,), "p")
    if dx is None:
        dx = torch.empty((R, 2 * H), dtype=torch.bfloat16, device=x.device)
    if dp is None:
        dp = torch.empty((R,), dtype=torch.float32, device=x.device)
    _need(dx, torch.bfloat16, (R, 2 * H), "dx")
    _need(dp, torch.float32, (R,), "dp")
    sptr = 0
    if status is not None:
        _need(status, torch.int32, (1,), "status")
        sptr = status.data_ptr()
    with torch.cuda.device(x.device):
        _check(load().situ_glu_bwd_router_dgrad(x.data_ptr(), dy.data_ptr(), w_down_t.data_ptr(),
                                                expert_offsets.data_ptr(), E, p.data_ptr(), dx.data_ptr(),
                                                dp.data_ptr(), sptr, R, H, D, beta, lbeta,
                                                _stream_handle(stream, x.device)))
    return dx, dp


def situ_glu_bwd_router_dgrad_wd(x, dy, w_down, expert_offsets, p, dx=None, dp=None, status=None,
                                 beta: float = 4.0, lbeta: float = 25.0, stream=None):
    """As situ_glu_bwd_router_dgrad, with the experts' W_down in the nn.Linear layout [E, D, H]."""
    import torch
    if x.dim() != 2 or x.shape[1] % 2 != 0:
        raise ValueError("x must be [R, 2H]")
    R, H = x.shape[0], x.shape[1] // 2
    if w_down.dim() != 3:
        raise ValueError("w_down must be [E, D, H]")
    E, D = w_down.shape[0], w_down.shape[1]
    _need(x, torch.bfloat16, (R, 2 * H), "x")
    _need(dy, torch.bfloat16, (R, D), "dy")
    _need(w_down, torch.bfloat16, (E, D, H), "w_down")
    _need(expert_offsets, torch.int64, (E + 1,), "expert_offsets")
    _need(p, torch.float32, (R,), "p")
    if dx is None:
        dx = torch.empty((R, 2 * H), dtype=torch.bfloat16, device=x.device)
    if dp is None:
        dp = torch.empty((R,), dtype=torch.float32, device=x.device)
    _need(dx, torch.bfloat16, (R, 2 * H), "dx")
    _need(dp, torch.float32, (R,), "dp")
    sptr = 0
    if status is not None:
        _need(status, torch.int32, (1,), "status")
        sptr = status.data_ptr()
    with torch.cuda.device(x.device):
        _check(load().situ_glu_bwd_router_dgrad_wd(x.data_ptr(), dy.data_ptr(), w_down.data_ptr(),
                                                   expert_offsets.data_ptr(), E, p.data_ptr(), dx.data_ptr(),
                                                   dp.data_ptr(), sptr, R, H, D, beta, lbeta,
                                                   _stream_handle(stream, x.device)))
    return dx, dp


def situ_glu_fwd_gateup(h, w_gate_up, expert_offsets, x=None, out=None, status=None, beta: float = 4.0,
                        lbeta: float = 25.0, stream=None):
    """(x bf16 [R,2H], out bf16 [R,H]) from the dispatched inputs h [R,D] and the experts' stacked
    [W_gate; W_up] [E,2H,D]: the gate/up GEMM on the tensor cores with the forward fused into it
    (x is the bf16-rounded projection, out the forward of that x).
    ``status`` (int32 [1] on the device, zeroed by the caller) turns 1 if a pipeline wait timed out."""
    import torch
    if h.dim() != 2:
        raise ValueError("h must be [R, D]")
    if w_gate_up.dim() != 3 or w_gate_up.shape[1] % 2 != 0:
        raise ValueError("w_gate_up must be [E, 2H, D]")
    R, D = h.shape
    E, H = w_gate_up.shape[0], w_gate_up.shape[1] // 2
    _need(h, torch.bfloat16, (R, D), "h")
    _need(w_gate_up, torch.bfloat16, (E, 2 * H, D), "w_gate_up")
    _need(expert_offsets, torch.int64, (E + 1,), "expert_offsets")
    if x is None:
        x = torch.empty((R, 2 * H), dtype=torch.bfloat16, device=h.device)
    if out is None:
        out = torch.empty((R, H), dtype=torch.bfloat16, device=h.device)
    _need(x, torch.bfloat16, (R, 2 * H), "x")
    _need(out, torch.bfloat16, (R, H), "out")
    sptr = 0
    if status is not None:
        _need(status, torch.int32, (1,), "status")
        sptr = status.data_ptr()
    with torch.cuda.device(h.device):
        _check(load().situ_glu_fwd_gateup(h.data_ptr(), w_gate_up.data_ptr(), expert_offsets.data_ptr(), E,
                                          x.data_ptr(), out.data_ptr(), sptr, R, H, D, beta, lbeta,
                                          _stream_handle(stream, h.device)))
    return x, out


def selftest_wait_timeout(status, elapsed_ns=None, stream=None):
    """Launch the failure-path self-test: one CTA waits on an mbarrier nothing completes, with the
    pipelines' bounded wait; after ~2 s it writes 1 to ``status`` (int32 [1], device, zeroed by
    the caller) and ``elapsed_ns`` (int64 [1], device) receives the wait's duration."""
    import torch
    _need(status, torch.int32, (1,), "status")
    eptr = 0
    if elapsed_ns is not None:
        _need(elapsed_ns, torch.int64, (1,), "elapsed_ns")
        eptr = elapsed_ns.data_ptr()
    with torch.cuda.device(status.device):
        _check(load().situ_glu_selftest_wait_timeout(status.data_ptr(), eptr, _stream_handle(stream, status.device)))


def _host_ptr(t, dtype, n, name):
    """Pointer of a contiguous CPU tensor or numpy array of `n` elements of `dtype` (torch dtype)."""
    import numpy as np
    import torch
    if isinstance(t, np.ndarray):
        want = {torch.float32: np.float32, torch.bfloat16: np.uint16, torch.uint8: np.uint8}[dtype]
        if t.dtype != want or t.size != n or not t.flags["C_CONTIGUOUS"]:
            raise ValueError(f"{name}: expected a contiguous {want.__name__} array of {n} elements")
        return t.ctypes.data
    if t.device.type != "cpu" or t.dtype != dtype or t.numel() != n or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CPU {dtype} tensor of {n} elements")
    return t.data_ptr()


def situ_adam_update_host(master, m, v, g, w_out, params: AdamParams, nthreads: int = 0):
    """One Adam step on host memory (master fp32, m / v bf16 updated in place; g fp32 read;
    w_out bf16 written). Accepts CPU tensors or numpy arrays (bf16 as uint16 bits)."""
    import torch
    n = master.numel() if hasattr(master, "numel") else master.size
    _check(load().situ_adam_update_host(_host_ptr(master, torch.float32, n, "master"),
                                        _host_ptr(m, torch.bfloat16, n, "m"), _host_ptr(v, torch.bfloat16, n, "v"),
                                        _host_ptr(g, torch.float32, n, "g"),
                                        _host_ptr(w_out, torch.bfloat16, n, "w_out"), n, ctypes.byref(params),
                                        int(nthreads)))


def adam_staging_bytes(chunk: int, nslots: int) -> int:
    return nslots * chunk * 6


def situ_adam_stream_step(grad, weight, master, m, v, params: AdamParams, staging, chunk: int, nslots: int = 2,
                          nthreads: int = 0, stream=None):
    """The streamed Adam step: device fp32 gradients `grad` [n] in, device bf16 `weight` [n]
    overwritten with the new working weights, host master fp32 / m, v bf16 updated in place;
    `staging` page-locked host memory of adam_staging_bytes(chunk, nslots) bytes."""
    import torch
    n = grad.numel()
    _need(grad, torch.float32, (n,), "grad")
    _need(weight, torch.bfloat16, (n,), "weight")
    nb = adam_staging_bytes(chunk, nslots)
    sp = _host_ptr(staging, torch.uint8, staging.numel() if hasattr(staging, "numel") else staging.size, "staging")
    if (staging.numel() if hasattr(staging, "numel") else staging.size) < nb:
        raise ValueError(f"staging: needs {nb} bytes")
    with torch.cuda.device(grad.device):
        _check(load().situ_adam_stream_step(grad.data_ptr(), weight.data_ptr(),
                                            _host_ptr(master, torch.float32, n, "master"),
                                            _host_ptr(m, torch.bfloat16, n, "m"), _host_ptr(v, torch.bfloat16, n, "v"),
                                            n, ctypes.byref(params), sp, int(chunk), int(nslots), int(nthreads),
                                            _stream_handle(stream, grad.device)))


__all__ = [
    "build", "load", "version", "status_string", "SituGluError",
    "situ_glu_fwd", "situ_glu_bwd_router", "situ_glu_fwd_ptr", "situ_glu_bwd_router_ptr",
    "situ_glu_fwd_save_fp8", "situ_glu_bwd_router_fp8", "FP8_BLOCK", "fp8_scale_blocks",
    "situ_glu_bwd_router_dgrad", "situ_glu_bwd_router_dgrad_wd", "situ_glu_fwd_gateup",
    "situ_and_mul", "selftest_wait_timeout", "AdamParams", "adam_params", "situ_adam_update_host", "situ_adam_stream_step", "adam_staging_bytes",
    "LIB_PATH", "INCLUDE",
]

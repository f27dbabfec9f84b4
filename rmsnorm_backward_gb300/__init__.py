"""LayerNorm / RMSNorm forward and backward on GB300 (sm_103a).

Thin Python binding of the C-ABI library ``libgbnorm.so`` (declared in
``include/gbnorm.h``).  Every step of the computation runs in the library's
CUDA kernels; this module only checks tensor metadata, allocates outputs with
PyTorch when the caller gives none, and passes raw device pointers, sizes and
the current CUDA stream through ctypes.  There is no CPU or PyTorch fallback:
if the library is not built, or a tensor is not on a CUDA device, the call
raises.

Names follow the pages' notation: ``ln_fwd``, ``rms_fwd`` produce ``y`` and
the per-row statistics (``mean``, ``rstd``); ``ln_bwd``, ``rms_bwd`` take
``dy`` and the saved statistics and produce ``dx``, ``dgamma`` (and
``dbeta``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = [
    "GbnError", "GbnOptions", "lib", "library_path", "ln_fwd", "rms_fwd", "ln_bwd", "rms_bwd",
    "ln_bwd_rows", "rms_bwd_rows", "bwd_reduce", "bwd_workspace_bytes", "bwd_plan", "BWD_KERNELS",
    "ln_bwd_host", "rms_bwd_host", "bwd_host_workspace_bytes", "silu_bwd", "gelu_bwd", "REDUCE_MODES", "KERNELS",
    "silu_bwd_host", "gelu_bwd_host",
    "device_error", "status_string", "DTYPE_CODES",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "_lib", "libgbnorm.so")

DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
GBN_OK = 0

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t


class GbnOptions(ctypes.Structure):
    """gbn_options of include/gbnorm.h."""

    _fields_ = [("ld_x", ctypes.c_int64), ("ld_dy", ctypes.c_int64), ("ld_out", ctypes.c_int64),
                ("accumulate", ctypes.c_int), ("grad_dtype", ctypes.c_int), ("reduce_mode", ctypes.c_int),
                ("kernel", ctypes.c_int), ("host_chunk", ctypes.c_int64), ("wait_limit_ns", ctypes.c_int64)]


# reduce_mode values (GBN_REDUCE_* of include/gbnorm.h)
REDUCE_MODES = {"partials": 0, "atomic": 1, "colwalk": 2}
# kernel values (GBN_KERNEL_*): the fastest that applies, the slot-staged
# kernel (never the warp-specialised backward), the plain-load kernel
KERNELS = {"auto": 0, "slot": 1, "plain": 2}


class GbnError(RuntimeError):
    """A libgbnorm call returned a non-zero gbn_status."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    L.gbn_bwd_workspace_bytes.argtypes = [_i64, _i64, _int, _int]
    L.gbn_bwd_workspace_bytes.restype = _sz
    L.ln_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _f, _i64, _i64, _int, _vp]
    L.rms_fwd.argtypes = [_vp, _vp, _vp, _vp, _f, _i64, _i64, _int, _vp]
    L.ln_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f, _i64, _i64, _int, _vp, _sz, _vp]
    L.rms_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _f, _i64, _i64, _int, _vp, _sz, _vp]
    L.ln_bwd_rows.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _vp, _sz, _vp]
    L.rms_bwd_rows.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _vp, _sz, _vp]
    L.gbn_bwd_reduce.argtypes = [_vp, _sz, _i64, _i64, _int, _int, _vp, _vp, _vp]
    opt = ctypes.POINTER(GbnOptions)
    L.ln_fwd_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _f, _i64, _i64, _int, opt, _vp]
    L.rms_fwd_ex.argtypes = [_vp, _vp, _vp, _vp, _f, _i64, _i64, _int, opt, _vp]
    L.ln_bwd_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f, _i64, _i64, _int, _vp, _sz, opt, _vp]
    L.rms_bwd_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _f, _i64, _i64, _int, _vp, _sz, opt, _vp]
    L.gbn_bwd_plan.argtypes = [_i64, _i64, _int, _int, ctypes.POINTER(_int), ctypes.POINTER(_int)]
    L.gbn_bwd_host_workspace_bytes.argtypes = [_i64, _i64, _int, _int]
    L.gbn_bwd_host_workspace_bytes.restype = _sz
    L.ln_bwd_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _vp, _sz, _vp]
    L.rms_bwd_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _vp, _sz, _vp]
    L.gbn_bwd_host_workspace_bytes_ex.argtypes = [_i64, _i64, _int, _int, opt]
    L.gbn_bwd_host_workspace_bytes_ex.restype = _sz
    L.ln_bwd_host_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _vp, _sz, opt, _vp]
    L.rms_bwd_host_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _vp, _sz, opt, _vp]
    L.gbn_act_host_workspace_bytes_ex.argtypes = [_i64, _int, opt]
    L.gbn_act_host_workspace_bytes_ex.restype = _sz
    L.silu_bwd_host_ex.argtypes = [_vp, _vp, _vp, _i64, _int, _vp, _sz, opt, _vp]
    L.gelu_bwd_host_ex.argtypes = [_vp, _vp, _vp, _i64, _int, _vp, _sz, opt, _vp]
    L.gbn_act_host_workspace_bytes.argtypes = [_i64, _int]
    L.gbn_act_host_workspace_bytes.restype = _sz
    L.silu_bwd_host.argtypes = [_vp, _vp, _vp, _i64, _int, _vp, _sz, _vp]
    L.gelu_bwd_host.argtypes = [_vp, _vp, _vp, _i64, _int, _vp, _sz, _vp]
    L.silu_bwd.argtypes = [_vp, _vp, _vp, _i64, _int, _vp]
    L.gelu_bwd.argtypes = [_vp, _vp, _vp, _i64, _int, _vp]
    L.gbn_device_error.argtypes = [_int]
    L.gbn_status_string.argtypes = [_int]
    L.gbn_status_string.restype = ctypes.c_char_p
    for name in ("ln_fwd", "rms_fwd", "ln_bwd", "rms_bwd", "ln_fwd_ex", "rms_fwd_ex", "ln_bwd_ex", "rms_bwd_ex",
                 "ln_bwd_rows", "rms_bwd_rows",
                 "gbn_bwd_reduce", "gbn_bwd_plan", "gbn_device_error", "silu_bwd", "gelu_bwd",
                 "ln_bwd_host", "rms_bwd_host", "silu_bwd_host", "gelu_bwd_host", "ln_bwd_host_ex",
                 "rms_bwd_host_ex", "silu_bwd_host_ex", "gelu_bwd_host_ex"):
        getattr(L, name).restype = _int
    return L


def lib() -> ctypes.CDLL:
    """The loaded libgbnorm.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(library_path):
                    raise RuntimeError(
                        f"libgbnorm.so is not built ({library_path}); run "
                        "`python -m rmsnorm_backward_gb300.build` or __graft_entry__.build()")
                _lib = _declare(ctypes.CDLL(library_path))
    return _lib


def status_string(status: int) -> str:
    return lib().gbn_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != GBN_OK:
        raise GbnError(fn, status)


def _rows(t: torch.Tensor, name: str) -> Tuple[int, int]:
    M, N, _ = _rows_ld(t, name)
    return M, N


def _rows_ld(t: torch.Tensor, name: str) -> Tuple[int, int, int]:
    """(M, N, row stride): a contiguous tensor with N = last dimension, or a
    2-D view whose rows are contiguous (stride(1) == 1, stride(0) >= N)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() < 1:
        raise ValueError(f"{name} must have a feature dimension")
    N = t.shape[-1]
    if t.is_contiguous():
        return (t.numel() // N if N else 0), N, N
    if t.dim() == 2 and t.stride(1) == 1 and t.stride(0) >= N:
        return t.shape[0], N, t.stride(0)
    raise ValueError(f"{name} must be contiguous, or a 2-D view with contiguous rows")


def _same_rows(t: torch.Tensor, ref: torch.Tensor, name: str) -> int:
    """Row stride of t, which must have ref's shape, dtype and device."""
    if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
        raise ValueError(f"{name} must have x's shape, dtype and device")
    return _rows_ld(t, name)[2]


def _code(t: torch.Tensor) -> int:
    try:
        return DTYPE_CODES[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _vec(t: Optional[torch.Tensor], name: str, n: int, dtype: torch.dtype, device) -> None:
    if t is None:
        return
    if t.dtype != dtype or t.numel() != n or not t.is_contiguous() or t.device != device:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of {n} elements on {device}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def bwd_workspace_bytes(M: int, N: int, dtype: torch.dtype, has_beta: bool, device=None) -> int:
    """Workspace bytes the backward needs on ``device`` (default: current)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(lib().gbn_bwd_workspace_bytes(M, N, DTYPE_CODES[dtype], int(has_beta)))


BWD_KERNELS = {0: "bwd_plain_kernel", 1: "bwd_staged_kernel", 2: "bwd_ws_kernel"}


def bwd_plan(M: int, N: int, dtype: torch.dtype, has_beta: bool, device=None) -> Tuple[int, int]:
    """(G, kind): the number of row blocks and the kernel aligned buffers with
    saved statistics take: 2 warp-specialised, 1 slot-staged, 0 plain
    (names in BWD_KERNELS)."""
    G, staged = _int(0), _int(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check("gbn_bwd_plan", lib().gbn_bwd_plan(M, N, DTYPE_CODES[dtype], int(has_beta),
                                                  ctypes.byref(G), ctypes.byref(staged)))
    return G.value, int(staged.value)


def device_error(clear: bool = True, device=None) -> int:
    """Synchronises the device and returns (and by default clears) the kernels' error flag."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(lib().gbn_device_error(int(clear)))


def _options(ld_x: int = 0, ld_dy: int = 0, ld_out: int = 0, accumulate: bool = False, grad_dtype=torch.float32,
             reduce: str = "partials", kernel: str = "auto", host_chunk: int = 0, wait_limit_ns: int = 0):
    return GbnOptions(ld_x, ld_dy, ld_out, int(bool(accumulate)), DTYPE_CODES[grad_dtype], REDUCE_MODES[reduce],
                      KERNELS[kernel], int(host_chunk), int(wait_limit_ns))


def _host_options(host_chunk: int = 0):
    return GbnOptions(0, 0, 0, 0, 0, 0, 0, int(host_chunk), 0)


def ln_fwd(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float, *,
           y: Optional[torch.Tensor] = None, mean: Optional[torch.Tensor] = None,
           rstd: Optional[torch.Tensor] = None, kernel: str = "auto", stream=None):
    """LayerNorm forward over the last dimension. Returns (y, mean, rstd).

    x may be a 2-D view with contiguous rows (any row stride); y likewise.
    kernel: "auto", or "slot" / "plain" to force that kernel (KERNELS)."""
    M, N, ld_x = _rows_ld(x, "x")
    y = torch.empty(x.shape, dtype=x.dtype, device=x.device) if y is None else y
    mean = torch.empty(M, dtype=torch.float32, device=x.device) if mean is None else mean
    rstd = torch.empty(M, dtype=torch.float32, device=x.device) if rstd is None else rstd
    for name, t in (("gamma", gamma), ("beta", beta)):
        _vec(t, name, N, x.dtype, x.device)
    _vec(mean, "mean", M, torch.float32, x.device)
    _vec(rstd, "rstd", M, torch.float32, x.device)
    ld_y = _same_rows(y, x, "y")
    opt = _options(ld_x, N, ld_y, kernel=kernel)
    with torch.cuda.device(x.device):
        _check("ln_fwd", lib().ln_fwd_ex(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(mean), _ptr(rstd),
                                         float(eps), M, N, _code(x), ctypes.byref(opt), _stream(x.device, stream)))
    return y, mean, rstd


def rms_fwd(x: torch.Tensor, gamma: torch.Tensor, eps: float, *, y: Optional[torch.Tensor] = None,
            rstd: Optional[torch.Tensor] = None, kernel: str = "auto", stream=None):
    """RMSNorm forward over the last dimension. Returns (y, rstd)."""
    M, N, ld_x = _rows_ld(x, "x")
    y = torch.empty(x.shape, dtype=x.dtype, device=x.device) if y is None else y
    rstd = torch.empty(M, dtype=torch.float32, device=x.device) if rstd is None else rstd
    _vec(gamma, "gamma", N, x.dtype, x.device)
    _vec(rstd, "rstd", M, torch.float32, x.device)
    ld_y = _same_rows(y, x, "y")
    opt = _options(ld_x, N, ld_y, kernel=kernel)
    with torch.cuda.device(x.device):
        _check("rms_fwd", lib().rms_fwd_ex(_ptr(x), _ptr(gamma), _ptr(y), _ptr(rstd), float(eps), M, N, _code(x),
                                           ctypes.byref(opt), _stream(x.device, stream)))
    return y, rstd


def _bwd_args(dy, x, gamma, stats, dx):
    M, N, ld_x = _rows_ld(x, "x")
    ld_dy = _same_rows(dy, x, "dy")
    _vec(gamma, "gamma", N, x.dtype, x.device)
    for name, t in stats:
        _vec(t, name, M, torch.float32, x.device)
    dx = torch.empty(x.shape, dtype=x.dtype, device=x.device) if dx is None else dx
    ld_dx = _same_rows(dx, x, "dx")
    return M, N, dx, (ld_x, ld_dy, ld_dx)


def _workspace(workspace, M, N, x, ln):
    need = bwd_workspace_bytes(M, N, x.dtype, ln, x.device)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    if workspace.device != x.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on x's device")
    return workspace, workspace.numel() * workspace.element_size()


def _grads(t, name, N, grad_dtype, device, accumulate):
    if t is None:
        return (torch.zeros if accumulate else torch.empty)(N, dtype=grad_dtype, device=device)
    _vec(t, name, N, grad_dtype, device)
    return t


def _recompute_eps(stats, eps):
    """eps for the save-nothing backward (all statistics None), else 0."""
    if all(t is None for t in stats):
        if eps is None:
            raise ValueError("without saved statistics the backward needs eps")
        return float(eps)
    if any(t is None for t in stats):
        raise ValueError("pass all saved statistics or none")
    return 0.0


def ln_bwd(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, mean: Optional[torch.Tensor],
           rstd: Optional[torch.Tensor], *, dx=None, dgamma=None, dbeta=None, workspace=None,
           accumulate: bool = False, grad_dtype=torch.float32, eps: Optional[float] = None,
           reduce: str = "partials", kernel: str = "auto", wait_limit_ns: int = 0, stream=None):
    """LayerNorm backward from the saved mean / rstd. Returns (dx, dgamma, dbeta).

    reduce: "partials" (deterministic, the default), or the measurement
    ablations "atomic" (nondeterministic) and "colwalk".  kernel: "auto", or
    "slot" / "plain" to force that kernel.  wait_limit_ns: the kernels' wait
    limit (0 = two seconds), a diagnostic of the error path.

    With mean = rstd = None nothing was saved: the statistics are formed from
    x with ``eps``.  dgamma / dbeta are float32 unless grad_dtype is x's
    dtype; with accumulate=True this call's sums are added to what they
    hold.  x, dy and dx may be 2-D views with contiguous rows."""
    if grad_dtype not in (torch.float32, x.dtype):
        raise ValueError("grad_dtype must be float32 or x's dtype")
    eps_arg = _recompute_eps((mean, rstd), eps)
    M, N, dx, (ld_x, ld_dy, ld_dx) = _bwd_args(dy, x, gamma, (("mean", mean), ("rstd", rstd)), dx)
    dgamma = _grads(dgamma, "dgamma", N, grad_dtype, x.device, accumulate)
    dbeta = _grads(dbeta, "dbeta", N, grad_dtype, x.device, accumulate)
    workspace, wsb = _workspace(workspace, M, N, x, True)
    opt = _options(ld_x, ld_dy, ld_dx, accumulate, grad_dtype, reduce, kernel, 0, wait_limit_ns)
    with torch.cuda.device(x.device):
        _check("ln_bwd", lib().ln_bwd_ex(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(dx),
                                         _ptr(dgamma), _ptr(dbeta), eps_arg, M, N, _code(x), _ptr(workspace), wsb,
                                         ctypes.byref(opt), _stream(x.device, stream)))
    return dx, dgamma, dbeta


def rms_bwd(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, rstd: Optional[torch.Tensor], *,
            dx=None, dgamma=None, workspace=None, accumulate: bool = False, grad_dtype=torch.float32,
            eps: Optional[float] = None, reduce: str = "partials", kernel: str = "auto", wait_limit_ns: int = 0,
            stream=None):
    """RMSNorm backward from the saved rstd (None: recomputed from x with eps).
    Returns (dx, dgamma); options as for ln_bwd."""
    if grad_dtype not in (torch.float32, x.dtype):
        raise ValueError("grad_dtype must be float32 or x's dtype")
    eps_arg = _recompute_eps((rstd,), eps)
    M, N, dx, (ld_x, ld_dy, ld_dx) = _bwd_args(dy, x, gamma, (("rstd", rstd),), dx)
    dgamma = _grads(dgamma, "dgamma", N, grad_dtype, x.device, accumulate)
    workspace, wsb = _workspace(workspace, M, N, x, False)
    opt = _options(ld_x, ld_dy, ld_dx, accumulate, grad_dtype, reduce, kernel, 0, wait_limit_ns)
    with torch.cuda.device(x.device):
        _check("rms_bwd", lib().rms_bwd_ex(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(dx), _ptr(dgamma),
                                           eps_arg, M, N, _code(x), _ptr(workspace), wsb, ctypes.byref(opt),
                                           _stream(x.device, stream)))
    return dx, dgamma


def ln_bwd_rows(dy, x, gamma, mean, rstd, *, dx=None, workspace, stream=None):
    """Phase 1 of ln_bwd: dx and the per-CTA partial rows in ``workspace``. Returns dx."""
    M, N, dx, lds = _bwd_args(dy, x, gamma, (("mean", mean), ("rstd", rstd)), dx)
    if lds != (N, N, N):
        raise ValueError("the backward phases take contiguous rows")
    workspace, wsb = _workspace(workspace, M, N, x, True)
    with torch.cuda.device(x.device):
        _check("ln_bwd_rows", lib().ln_bwd_rows(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd),
                                                _ptr(dx), M, N, _code(x), _ptr(workspace), wsb,
                                                _stream(x.device, stream)))
    return dx


def rms_bwd_rows(dy, x, gamma, rstd, *, dx=None, workspace, stream=None):
    """Phase 1 of rms_bwd: dx and the per-CTA partial rows in ``workspace``. Returns dx."""
    M, N, dx, lds = _bwd_args(dy, x, gamma, (("rstd", rstd),), dx)
    if lds != (N, N, N):
        raise ValueError("the backward phases take contiguous rows")
    workspace, wsb = _workspace(workspace, M, N, x, False)
    with torch.cuda.device(x.device):
        _check("rms_bwd_rows", lib().rms_bwd_rows(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(dx), M, N,
                                                  _code(x), _ptr(workspace), wsb, _stream(x.device, stream)))
    return dx


def bwd_reduce(workspace: torch.Tensor, M: int, N: int, dtype: torch.dtype, has_beta: bool, *,
               dgamma: torch.Tensor, dbeta: Optional[torch.Tensor] = None, stream=None):
    """Phase 2 of the backward: the fixed-order column sum of the partial rows."""
    dev = workspace.device
    _vec(dgamma, "dgamma", N, torch.float32, dev)
    if has_beta:
        _vec(dbeta, "dbeta", N, torch.float32, dev)
    with torch.cuda.device(dev):
        _check("gbn_bwd_reduce", lib().gbn_bwd_reduce(
            _ptr(workspace), workspace.numel() * workspace.element_size(), M, N, DTYPE_CODES[dtype],
            int(has_beta), _ptr(dgamma), _ptr(dbeta) if has_beta else None, _stream(dev, stream)))


def _act_bwd(fn: str, dy: torch.Tensor, preact: torch.Tensor, dx: Optional[torch.Tensor], stream):
    if not (dy.is_contiguous() and preact.is_contiguous()):
        raise ValueError(f"{fn}: dy and preact must be contiguous")
    if dy.shape != preact.shape or dy.dtype != preact.dtype or dy.device != preact.device:
        raise ValueError(f"{fn}: dy and preact must match in shape, dtype and device")
    code = _code(dy)
    if dx is None:
        dx = torch.empty_like(dy)
    elif not dx.is_contiguous() or dx.shape != dy.shape or dx.dtype != dy.dtype or dx.device != dy.device:
        raise ValueError(f"{fn}: dx must be a contiguous tensor like dy")
    dev = dy.device
    with torch.cuda.device(dev):
        _check(fn, getattr(lib(), fn)(_ptr(dy), _ptr(preact), _ptr(dx), dy.numel(), code, _stream(dev, stream)))
    return dx


def silu_bwd(dy: torch.Tensor, preact: torch.Tensor, *, dx: Optional[torch.Tensor] = None, stream=None):
    """dx = dy * SiLU'(preact), elementwise; ``dx`` may be ``dy`` (in place)."""
    return _act_bwd("silu_bwd", dy, preact, dx, stream)


def gelu_bwd(dy: torch.Tensor, preact: torch.Tensor, *, dx: Optional[torch.Tensor] = None, stream=None):
    """dx = dy * GELU'(preact) (exact erf form), elementwise; ``dx`` may be ``dy``."""
    return _act_bwd("gelu_bwd", dy, preact, dx, stream)


# ---------------------------------------------------------------------------
# backward from host buffers (copies pipelined with the kernels)
# ---------------------------------------------------------------------------
def bwd_host_workspace_bytes(M: int, N: int, dtype: torch.dtype, has_beta: bool, device=None,
                             chunk_rows: int = 0) -> int:
    """Device workspace bytes ``ln_bwd_host`` / ``rms_bwd_host`` need (for
    ``chunk_rows`` rows per chunk; 0 = about 16 MiB of each input)."""
    opt = _host_options(chunk_rows)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(lib().gbn_bwd_host_workspace_bytes_ex(M, N, DTYPE_CODES[dtype], int(has_beta),
                                                         ctypes.byref(opt)))


def _host_args(fn, dy, x, gamma, stats, dx, grads):
    for name, t in (("dy", dy), ("x", x), ("gamma", gamma)) + stats:
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{fn}: {name} must be a contiguous CPU tensor")
    if x.dim() != 2 or dy.shape != x.shape or dy.dtype != x.dtype or gamma.dtype != x.dtype:
        raise ValueError(f"{fn}: dy and x must be [M, N] of one dtype, gamma of that dtype")
    M, N = x.shape
    if gamma.numel() != N:
        raise ValueError(f"{fn}: gamma must have N elements")
    for name, t in stats:
        if t.dtype != torch.float32 or t.numel() != M:
            raise ValueError(f"{fn}: {name} must be float32 with M elements")
    if dx is None:
        dx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    elif dx.device.type != "cpu" or not dx.is_contiguous() or dx.shape != x.shape or dx.dtype != x.dtype:
        raise ValueError(f"{fn}: dx must be a contiguous CPU tensor like x")
    out = []
    for name, g in grads:
        if g is None:
            g = torch.empty(N, dtype=torch.float32, pin_memory=True)
        elif g.device.type != "cpu" or g.dtype != torch.float32 or g.numel() != N or not g.is_contiguous():
            raise ValueError(f"{fn}: {name} must be a contiguous float32 CPU tensor of N elements")
        out.append(g)
    return M, N, dx, out


def _host_workspace(workspace, M, N, dtype, ln, device, chunk_rows):
    need = bwd_host_workspace_bytes(M, N, dtype, ln, device, chunk_rows)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    if workspace.device != torch.device(device) or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a device buffer of at least {need} bytes")
    return workspace, workspace.numel() * workspace.element_size()


def ln_bwd_host(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, mean: torch.Tensor, rstd: torch.Tensor, *,
                dx=None, dgamma=None, dbeta=None, workspace=None, device=None, chunk_rows: int = 0, stream=None):
    """LayerNorm backward with every tensor in host memory (pinned for
    overlap).  Returns (dx, dgamma, dbeta) as CPU tensors, complete once
    ``stream`` is.  chunk_rows: rows per pipeline chunk (0 = about 16 MiB of
    each input)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    M, N, dx, (dgamma, dbeta) = _host_args("ln_bwd_host", dy, x, gamma, (("mean", mean), ("rstd", rstd)), dx,
                                           (("dgamma", dgamma), ("dbeta", dbeta)))
    workspace, wsb = _host_workspace(workspace, M, N, x.dtype, True, device, chunk_rows)
    opt = _host_options(chunk_rows)
    with torch.cuda.device(device):
        _check("ln_bwd_host", lib().ln_bwd_host_ex(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd),
                                                   _ptr(dx), _ptr(dgamma), _ptr(dbeta), M, N, _code(x),
                                                   _ptr(workspace), wsb, ctypes.byref(opt),
                                                   _stream(device, stream)))
    return dx, dgamma, dbeta


def rms_bwd_host(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, rstd: torch.Tensor, *,
                 dx=None, dgamma=None, workspace=None, device=None, chunk_rows: int = 0, stream=None):
    """RMSNorm backward with every tensor in host memory (pinned for
    overlap).  Returns (dx, dgamma) as CPU tensors, complete once ``stream``
    is.  chunk_rows as for ln_bwd_host."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    M, N, dx, (dgamma,) = _host_args("rms_bwd_host", dy, x, gamma, (("rstd", rstd),), dx, (("dgamma", dgamma),))
    workspace, wsb = _host_workspace(workspace, M, N, x.dtype, False, device, chunk_rows)
    opt = _host_options(chunk_rows)
    with torch.cuda.device(device):
        _check("rms_bwd_host", lib().rms_bwd_host_ex(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), _ptr(dx),
                                                     _ptr(dgamma), M, N, _code(x), _ptr(workspace), wsb,
                                                     ctypes.byref(opt), _stream(device, stream)))
    return dx, dgamma


def _act_host(fn: str, dy: torch.Tensor, preact: torch.Tensor, dx, workspace, device, chunk, stream):
    for name, t in (("dy", dy), ("preact", preact)):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{fn}: {name} must be a contiguous CPU tensor")
    if dy.shape != preact.shape or dy.dtype != preact.dtype:
        raise ValueError(f"{fn}: dy and preact must match in shape and dtype")
    code = _code(dy)
    if dx is None:
        dx = torch.empty(dy.shape, dtype=dy.dtype, pin_memory=True)
    elif dx.device.type != "cpu" or not dx.is_contiguous() or dx.shape != dy.shape or dx.dtype != dy.dtype:
        raise ValueError(f"{fn}: dx must be a contiguous CPU tensor like dy")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    opt = _host_options(chunk)
    with torch.cuda.device(device):
        need = int(lib().gbn_act_host_workspace_bytes_ex(dy.numel(), code, ctypes.byref(opt)))
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
        wsb = workspace.numel() * workspace.element_size()
        if workspace.device != device or wsb < need:
            raise ValueError(f"{fn}: workspace must be a device buffer of at least {need} bytes")
        _check(fn, getattr(lib(), fn + "_ex")(_ptr(dy), _ptr(preact), _ptr(dx), dy.numel(), code, _ptr(workspace),
                                              wsb, ctypes.byref(opt), _stream(device, stream)))
    return dx


def silu_bwd_host(dy: torch.Tensor, preact: torch.Tensor, *, dx=None, workspace=None, device=None,
                  chunk: int = 0, stream=None):
    """silu_bwd with dy, preact and dx in host memory (pinned for overlap);
    dx is complete once ``stream`` is.  chunk: elements per pipeline chunk
    (0 = about 16 MiB of each tensor)."""
    return _act_host("silu_bwd_host", dy, preact, dx, workspace, device, chunk, stream)


def gelu_bwd_host(dy: torch.Tensor, preact: torch.Tensor, *, dx=None, workspace=None, device=None,
                  chunk: int = 0, stream=None):
    """gelu_bwd with dy, preact and dx in host memory (pinned for overlap)."""
    return _act_host("gelu_bwd_host", dy, preact, dx, workspace, device, chunk, stream)

"""float64 CPU oracle for the LayerNorm / RMSNorm forward and backward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product path (the
CUDA library and its Python binding) never imports, links or runs it.

The arithmetic lives in ``norm_oracle.c`` (plain loops in double precision,
each function citing the page section it follows); this module only compiles
it with gcc and marshals numpy arrays through ctypes.  Inputs are widened to
float64 here; outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "norm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnorm_oracle.so")
GCC_FLAGS = ["-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11", "-pthread"]

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compiles ``src`` with gcc into the shared library ``out``; returns ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", *GCC_FLAGS, *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


_P = ctypes.POINTER(ctypes.c_double)
_I = ctypes.c_int64


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads the oracle library (building it first if needed)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
        return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.oracle_ln_fwd.argtypes = [_I, _I, _P, _P, _P, ctypes.c_double, _P, _P, _P]
    lib.oracle_rms_fwd.argtypes = [_I, _I, _P, _P, ctypes.c_double, _P, _P]
    lib.oracle_ln_bwd.argtypes = [_I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.oracle_rms_bwd.argtypes = [_I, _I, _P, _P, _P, _P, _P, _P]
    for f in ("oracle_silu_bwd", "oracle_gelu_bwd", "oracle_silu_fwd", "oracle_gelu_fwd"):
        getattr(lib, f).argtypes = [_I, _P, _P, _P][: 4 if f.endswith("bwd") else 3]
    lib.oracle_ln_bwd_threads.argtypes = [_I, _I, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int]
    lib.oracle_rms_bwd_threads.argtypes = [_I, _I, _P, _P, _P, _P, _P, _P, ctypes.c_int]
    lib.oracle_ln_bwd_threads.restype = ctypes.c_int
    lib.oracle_rms_bwd_threads.restype = ctypes.c_int
    for f in ("oracle_ln_fwd", "oracle_rms_fwd", "oracle_ln_bwd", "oracle_rms_bwd", "oracle_silu_bwd",
              "oracle_gelu_bwd", "oracle_silu_fwd", "oracle_gelu_fwd"):
        getattr(lib, f).restype = None
    return lib


def _d(a) -> np.ndarray:
    """Widen to a C-contiguous float64 array (exact for fp16/bf16/fp32 values)."""
    if hasattr(a, "detach"):  # a torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_P)


def _shape(x: np.ndarray) -> Tuple[int, int]:
    if x.ndim != 2:
        raise ValueError("x must be [M, N]")
    return int(x.shape[0]), int(x.shape[1])


def ln_fwd(x, gamma, beta, eps: float, lib: Optional[ctypes.CDLL] = None):
    """LayerNorm forward. Returns (y [M,N], mean [M], rstd [M]), float64."""
    lib = lib or load()
    x, gamma, beta = _d(x), _d(gamma), _d(beta)
    M, N = _shape(x)
    y = np.empty((M, N)); mean = np.empty(M); rstd = np.empty(M)
    lib.oracle_ln_fwd(M, N, _p(x), _p(gamma), _p(beta), float(eps), _p(y), _p(mean), _p(rstd))
    return y, mean, rstd


def rms_fwd(x, gamma, eps: float, lib: Optional[ctypes.CDLL] = None):
    """RMSNorm forward. Returns (y [M,N], rstd [M]), float64."""
    lib = lib or load()
    x, gamma = _d(x), _d(gamma)
    M, N = _shape(x)
    y = np.empty((M, N)); rstd = np.empty(M)
    lib.oracle_rms_fwd(M, N, _p(x), _p(gamma), float(eps), _p(y), _p(rstd))
    return y, rstd


def ln_bwd(dy, x, gamma, mean, rstd, lib: Optional[ctypes.CDLL] = None, threads: int = 1):
    """LayerNorm backward from saved stats. Returns (dx [M,N], dgamma [N], dbeta [N]).

    threads > 1: the timed mode across host threads (row blocks, partial
    sums added in thread order), for the CPU baseline."""
    lib = lib or load()
    dy, x, gamma, mean, rstd = _d(dy), _d(x), _d(gamma), _d(mean).reshape(-1), _d(rstd).reshape(-1)
    M, N = _shape(x)
    dx = np.empty((M, N)); dg = np.empty(N); db = np.empty(N)
    if threads > 1:
        if lib.oracle_ln_bwd_threads(M, N, _p(dy), _p(x), _p(gamma), _p(mean), _p(rstd), _p(dx), _p(dg), _p(db),
                                     threads) != 0:
            raise RuntimeError("oracle_ln_bwd_threads failed")
    else:
        lib.oracle_ln_bwd(M, N, _p(dy), _p(x), _p(gamma), _p(mean), _p(rstd), _p(dx), _p(dg), _p(db))
    return dx, dg, db


def rms_bwd(dy, x, gamma, rstd, lib: Optional[ctypes.CDLL] = None, threads: int = 1):
    """RMSNorm backward from the saved rstd. Returns (dx [M,N], dgamma [N]).

    threads > 1: the timed mode across host threads, as for ln_bwd."""
    lib = lib or load()
    dy, x, gamma, rstd = _d(dy), _d(x), _d(gamma), _d(rstd).reshape(-1)
    M, N = _shape(x)
    dx = np.empty((M, N)); dg = np.empty(N)
    if threads > 1:
        if lib.oracle_rms_bwd_threads(M, N, _p(dy), _p(x), _p(gamma), _p(rstd), _p(dx), _p(dg), threads) != 0:
            raise RuntimeError("oracle_rms_bwd_threads failed")
    else:
        lib.oracle_rms_bwd(M, N, _p(dy), _p(x), _p(gamma), _p(rstd), _p(dx), _p(dg))
    return dx, dg


def act_bwd(kind: str, dy, preact, lib: Optional[ctypes.CDLL] = None) -> np.ndarray:
    """dx = dy * f'(preact) for f = SiLU ("silu") or GELU, erf form ("gelu"); any shape."""
    lib = lib or load()
    dy, preact = _d(dy), _d(preact)
    if dy.shape != preact.shape:
        raise ValueError("dy and preact must have the same shape")
    dx = np.empty_like(dy)
    getattr(lib, f"oracle_{kind}_bwd")(dy.size, _p(dy), _p(preact), _p(dx))
    return dx


def act_fwd(kind: str, x, lib: Optional[ctypes.CDLL] = None) -> np.ndarray:
    """f(x) for f = SiLU or GELU (erf form)."""
    lib = lib or load()
    x = _d(x)
    y = np.empty_like(x)
    getattr(lib, f"oracle_{kind}_fwd")(x.size, _p(x), _p(y))
    return y

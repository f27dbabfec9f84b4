"""Seeded synthetic inputs for the LayerNorm / RMSNorm forward and backward.

This module is shared by the oracle's tests, the GPU parity tests and the
benchmark.  It draws random numbers and rounds them to the storage dtype; it
holds none of the normalisation arithmetic (no means, no variances, no
gradients), so neither the oracle nor the CUDA path depends on the other
through it.

Generator (one documented recipe, used everywhere):

* ``splitmix64`` in counter mode: draw ``i`` of stream ``s`` under seed
  ``seed`` is ``mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` with
  ``key = seed XOR (s * 0xD1B54A32D192ED03)`` and ``mix`` the splitmix64
  finaliser (shifts 30/27/31, multipliers 0xBF58476D1CE4E5B9 and
  0x94D049BB133111EB).
* uniforms on (0, 1): ``((z >> 11) + 0.5) * 2**-53``.
* normals: Box-Muller on uniform pairs (draws ``2i`` and ``2i + 1``),
  ``sqrt(-2 ln u1) * cos(2 pi u2)``.
* every value is formed in float64, rounded to float32 (round to nearest
  even), then to the storage dtype (fp16 / bf16, round to nearest even).
  The oracle receives the storage values widened exactly to float64; the GPU
  receives the same bytes.

The five workloads are the shapes, epsilons and value distributions of the
backward pass studied on the pages ("Norm backward in Triton — the dγ/dβ
reduction", worked numbers: 16384 rows x 4096 features, bf16; "05: Layer
norm", its 1151 x 8192 fp16 check).  Sizes may be overridden to get smaller
cases with the same distributions.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids: one per drawn quantity, so that changing one size does not shift
# another quantity's draws
STREAM_X = 1
STREAM_DY = 2
STREAM_GAMMA = 3
STREAM_BETA = 4
STREAM_ROW_SHIFT = 5
STREAM_ROW_SCALE = 6
STREAM_OUTLIER_COLS = 7
STREAM_PREACT = 8
STREAM_ACT_DY = 9

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of one splitmix64 stream."""
    with np.errstate(over="ignore"):
        key = np.uint64(seed) ^ (np.uint64(stream) * _STREAM_MUL)
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(key + i * _GOLDEN)


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """``n`` float64 uniforms on (0, 1)."""
    out = np.empty(n, dtype=np.float64)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        z = raw_u64(seed, stream, start + c0, c1 - c0)
        out[c0:c1] = ((z >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53
    return out


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` float64 standard normals (Box-Muller, cosine branch)."""
    out = np.empty(n, dtype=np.float64)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        z = raw_u64(seed, stream, 2 * c0, 2 * (c1 - c0))
        u = ((z >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53
        u1, u2 = u[0::2], u[1::2]
        out[c0:c1] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return out


TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def to_storage(values: np.ndarray, dtype: str) -> torch.Tensor:
    """float64 -> float32 (RNE) -> storage dtype (RNE), as a CPU tensor."""
    f32 = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float64).astype(np.float32))
    return f32.to(TORCH_DTYPES[dtype])


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic configuration: op, storage dtype, shape, eps, recipe."""

    name: str
    op: str  # "ln" or "rms"
    dtype: str  # "f32" | "f16" | "bf16"
    M: int
    N: int
    eps: float
    recipe: str  # key into _RECIPES
    seed: int = 0

    @property
    def has_beta(self) -> bool:
        return self.op == "ln"

    def with_shape(self, M: int, N: int, name: Optional[str] = None) -> "Workload":
        return dataclasses.replace(self, M=M, N=N, name=name or f"{self.name}@{M}x{N}")

    def describe(self) -> str:
        return _RECIPE_TEXT[self.recipe]


# the value distributions, one per workload family
_RECIPE_TEXT = {
    "ln_normal": "x~N(0,1); gamma=1+0.1N(0,1); beta=0.1N(0,1); dy~N(0,1)",
    "ln_uniform_affine": "x~N(0,1); gamma~U(0,1); beta~U(0,1); dy=0.1N(0,1)",
    "rms_normal": "x~N(0,1); gamma=1+0.02N(0,1); dy=1e-2N(0,1)",
    "ln_shifted_rows": ("x_r=a_r+s_r*N(0,1), a_r~U(-5,5), s_r=exp(0.5*N(0,1)); "
                        "gamma=1+0.1N(0,1); beta=0.1N(0,1); dy~N(0,1)"),
    "rms_outliers": ("x~N(0,1) with round(1% of N) feature columns (seeded "
                     "permutation) scaled x20; gamma=1+0.05N(0,1); dy=1e-2N(0,1)"),
}


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("ln_f32_64x256", "ln", "f32", 64, 256, 1e-5, "ln_normal"),
        Workload("ln_f16_1151x8192", "ln", "f16", 1151, 8192, 1e-5, "ln_uniform_affine"),
        Workload("rms_bf16_16384x4096", "rms", "bf16", 16384, 4096, 1e-6, "rms_normal"),
        Workload("ln_bf16_65536x1024", "ln", "bf16", 65536, 1024, 1e-5, "ln_shifted_rows"),
        Workload("rms_bf16_8192x16384", "rms", "bf16", 8192, 16384, 1e-6, "rms_outliers"),
    )
}

# the workload the benchmark's headline line is taken on
HEADLINE = "rms_bf16_16384x4096"


def outlier_columns(seed: int, N: int) -> np.ndarray:
    """The round(1% of N) columns scaled x20: the first ones of a seeded permutation."""
    k = int(round(0.01 * N))
    keys = uniform(seed, STREAM_OUTLIER_COLS, N)
    return np.sort(np.argsort(keys, kind="stable")[:k])


def _x_values(w: Workload) -> np.ndarray:
    M, N = w.M, w.N
    x = normal(w.seed, STREAM_X, M * N).reshape(M, N)
    if w.recipe == "ln_shifted_rows":
        a = -5.0 + 10.0 * uniform(w.seed, STREAM_ROW_SHIFT, M)
        s = np.exp(0.5 * normal(w.seed, STREAM_ROW_SCALE, M))
        x = a[:, None] + s[:, None] * x
    elif w.recipe == "rms_outliers":
        x[:, outlier_columns(w.seed, N)] *= 20.0
    return x


def _gamma_beta_values(w: Workload):
    N = w.N
    g = normal(w.seed, STREAM_GAMMA, N)
    b = normal(w.seed, STREAM_BETA, N)
    if w.recipe in ("ln_normal", "ln_shifted_rows"):
        return 1.0 + 0.1 * g, 0.1 * b
    if w.recipe == "ln_uniform_affine":
        return uniform(w.seed, STREAM_GAMMA, N), uniform(w.seed, STREAM_BETA, N)
    if w.recipe == "rms_normal":
        return 1.0 + 0.02 * g, None
    if w.recipe == "rms_outliers":
        return 1.0 + 0.05 * g, None
    raise KeyError(w.recipe)


def _dy_scale(w: Workload) -> float:
    return {"ln_normal": 1.0, "ln_uniform_affine": 0.1, "rms_normal": 1e-2,
            "ln_shifted_rows": 1.0, "rms_outliers": 1e-2}[w.recipe]


def make_inputs(w: Workload) -> Dict[str, torch.Tensor]:
    """Storage-dtype CPU tensors ``x``, ``dy`` [M, N], ``gamma`` [N], ``beta`` [N] (LN only)."""
    out = {
        "x": to_storage(_x_values(w), w.dtype),
        "dy": to_storage(_dy_scale(w) * normal(w.seed, STREAM_DY, w.M * w.N).reshape(w.M, w.N), w.dtype),
    }
    g, b = _gamma_beta_values(w)
    out["gamma"] = to_storage(g, w.dtype)
    if w.has_beta:
        out["beta"] = to_storage(b, w.dtype)
    return out


def exact_double(t: torch.Tensor) -> np.ndarray:
    """Storage values widened exactly to float64 (every fp16/bf16/fp32 value is a double)."""
    return t.detach().to("cpu", torch.float64).numpy()


def bwd_min_bytes(op: str, dtype: str, M: int, N: int) -> int:
    """Algorithmic HBM bytes of one backward pass.

    Reads x and dy (M*N storage elements each), gamma (N), the saved fp32
    statistics (rstd, plus mean for LayerNorm: 4 bytes per row each); writes dx
    (M*N), dgamma and, for LayerNorm, dbeta (N fp32 each).  The [G, N] partial
    workspace is overhead, not algorithmic traffic.
    """
    es = ELEM_BYTES[dtype]
    nstat = 2 if op == "ln" else 1
    ngrad = 2 if op == "ln" else 1
    return 3 * M * N * es + N * es + 4 * nstat * M + 4 * ngrad * N


def fwd_min_bytes(op: str, dtype: str, M: int, N: int) -> int:
    """Algorithmic HBM bytes of one forward pass: read x, gamma (and beta); write y and the stats."""
    es = ELEM_BYTES[dtype]
    nstat = 2 if op == "ln" else 1
    nparam = 2 if op == "ln" else 1
    return 2 * M * N * es + nparam * N * es + 4 * nstat * M


# ---------------------------------------------------------------------------
# activation backward inputs: dy and the saved pre-activation of an MLP's
# SiLU / GELU ("Norm backward in Triton", section "Activation backward")
# ---------------------------------------------------------------------------
ACT_RECIPE = "preact = 2 N(0,1) (both tails and the zeros of f' are covered); dy = N(0,1)"


@dataclasses.dataclass(frozen=True)
class ActWorkload:
    """dx = dy * f'(preact) over an M x N activation tensor (stored contiguous)."""

    name: str
    kind: str  # "silu" | "gelu"
    dtype: str
    M: int
    N: int
    seed: int = 0

    @property
    def n(self) -> int:
        return self.M * self.N

    def with_shape(self, M: int, N: int) -> "ActWorkload":
        return dataclasses.replace(self, M=M, N=N, name=f"{self.name}@{M}x{N}")


ACT_WORKLOADS: Dict[str, ActWorkload] = {
    a.name: a
    for a in (
        ActWorkload("silu_bf16_16384x4096", "silu", "bf16", 16384, 4096),
        ActWorkload("gelu_bf16_16384x4096", "gelu", "bf16", 16384, 4096),
    )
}


def make_act_inputs(a: ActWorkload) -> Dict[str, torch.Tensor]:
    """Storage-dtype CPU tensors ``dy`` and ``preact`` of shape [M, N]."""
    return {
        "dy": to_storage(normal(a.seed, STREAM_ACT_DY, a.n).reshape(a.M, a.N), a.dtype),
        "preact": to_storage(2.0 * normal(a.seed, STREAM_PREACT, a.n).reshape(a.M, a.N), a.dtype),
    }


def act_min_bytes(dtype: str, n: int) -> int:
    """Algorithmic HBM bytes of one activation backward: read dy and preact, write dx."""
    return 3 * n * ELEM_BYTES[dtype]

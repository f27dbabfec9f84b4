"""Parity rules between the CUDA path and the float64 oracle.

The stated bars:
  * fp32 outputs: relative error <= 1e-5;
  * fp16 / bf16 outputs (y, dx): error <= 2 ulp of the output dtype relative
    to the oracle's value rounded to that dtype (round to nearest even);
  * dgamma / dbeta: |err| <= 1e-3 * (1 + |ref|).

Reading for values near zero.  y (with beta) and dx are differences of O(1)
terms and can be arbitrarily close to zero, where no float32 computation can
be relatively accurate.  Each row therefore has a term scale ``s`` (the
largest magnitude among the summands that form an output of that row), and
a float32 noise allowance A.  For float32 outputs ``A = 2**-21 * s`` (8
float32 unit roundoffs u of the term scale): the largest errors measured on
a GB300 over LayerNorm and RMSNorm at N = 256 ... 65536, every kernel, are
about 3.5u (y) and 3u (dx end to end), so A leaves a margin of about 2x and a
3x accuracy regression fails.  For fp16 / bf16 outputs ``A = 2**-18 * s`` (64u):
there A only matters where the value is below about 2**-11 * s, where one
output ulp is already of the order of the float32 noise.  An element passes
if its error is within the stated bar OR within A:
  * fp32:        |got - ref| <= max(1e-5 * |ref|, A)
  * fp16 / bf16: |got - R(ref)| <= max(2 * ulp(R(ref)), A)
The strict per-element counts (without A) are reported alongside.

Term scales, with m_j = (|x_j| + |mean|) * rstd the magnitude of the float32
quantities xhat_j is formed from (x*rstd and mean*rstd; for RMSNorm mean = 0
and m_j = |xhat_j|): LayerNorm rows with a large mean next to their spread
lose the mean's float32 rounding to the cancellation in x - mean, so their
noise scales with |mean| * rstd, not with |xhat|.
  * dx: rstd * max_j (|dyhat_j| + mean_k |dyhat_k| [LayerNorm] + m_j * mean_k |dyhat_k| m_k)
  * y:  max_j (|gamma_j| m_j + |beta_j|)
  * mean: mean_j |x_j|;  rstd: none (it is a quotient of positive sums)
"""
from __future__ import annotations

import dataclasses

import numpy as np

A_EXP = {"f32": -21, "f16": -18, "bf16": -18}
SIGNIF_BITS = {"f32": 24, "f16": 11, "bf16": 8}
MIN_QUANTUM = {"f32": 2.0 ** -149, "f16": 2.0 ** -24, "bf16": 2.0 ** -133}


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of ``dtype`` values at |v| (the quantum of the binade of v)."""
    p = SIGNIF_BITS[dtype]
    _, e = np.frexp(np.abs(v))
    q = np.ldexp(np.ones_like(v, dtype=np.float64), e - p)
    return np.maximum(q, MIN_QUANTUM[dtype])


def round_to(v: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> nearest ``dtype`` value (ties to even), returned as float64."""
    q = ulp(v, dtype)
    return np.round(v / q) * q


@dataclasses.dataclass
class Report:
    name: str
    n: int
    n_fail: int
    n_strict_fail: int
    worst: float  # worst error / allowed
    worst_index: tuple
    worst_u: float = 0.0  # worst error in float32 unit roundoffs of the row's term scale (2**-24 * s)

    def ok(self) -> bool:
        return self.n_fail == 0

    def __str__(self) -> str:
        return (f"{self.name}: {self.n_fail}/{self.n} beyond tolerance "
                f"({self.n_strict_fail} beyond the strict bar), worst err/allowed {self.worst:.3g} "
                f"at {self.worst_index}, worst err {self.worst_u:.3g} u*s")


def check_elementwise(name: str, got: np.ndarray, ref: np.ndarray, dtype: str, scale_row: np.ndarray,
                      abs_floor=0.0, a_exp=None) -> Report:
    """got, ref: [M, N] (got already widened to float64); scale_row: [M];
    abs_floor: an extra absolute allowance (scalar or broadcastable to [M, N]);
    a_exp: the noise allowance's exponent (A = 2**a_exp * s), default A_EXP[dtype]."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    A = np.ldexp(np.asarray(scale_row, dtype=np.float64), A_EXP[dtype] if a_exp is None else a_exp)[:, None]
    if dtype == "f32":
        strict = 1e-5 * np.abs(ref)
        err = np.abs(got - ref)
    else:
        R = round_to(ref, dtype)
        strict = 2.0 * ulp(R, dtype)
        err = np.abs(got - R)
    allowed = np.maximum(np.maximum(strict, A), abs_floor)
    bad = ~(err <= allowed)  # NaN counts as bad
    ratio = np.where(allowed > 0, err / np.where(allowed > 0, allowed, 1), np.where(err > 0, np.inf, 0))
    ratio = np.where(np.isnan(ratio), np.inf, ratio)
    idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape) if ratio.size else ()
    s64 = np.ldexp(np.asarray(scale_row, dtype=np.float64), -24)[:, None]
    eu = np.where(s64 > 0, err / np.where(s64 > 0, s64, 1), 0.0)
    return Report(name, int(got.size), int(bad.sum()), int((~(err <= strict)).sum()),
                  float(ratio.max()) if ratio.size else 0.0, tuple(int(i) for i in idx),
                  float(np.nanmax(eu)) if eu.size else 0.0)


def check_stat(name: str, got: np.ndarray, ref: np.ndarray, floor: np.ndarray = None) -> Report:
    """fp32 per-row statistic against float64: relative 1e-5, floored at A of ``floor``."""
    got = np.asarray(got, dtype=np.float64)[:, None]
    ref = np.asarray(ref, dtype=np.float64)[:, None]
    fl = np.zeros(ref.shape[0]) if floor is None else np.asarray(floor, dtype=np.float64)
    return check_elementwise(name, got, ref, "f32", fl)


def check_param_grad(name: str, got: np.ndarray, ref: np.ndarray) -> Report:
    """dgamma / dbeta: |err| <= 1e-3 * (1 + |ref|)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    allowed = 1e-3 * (1.0 + np.abs(ref))
    bad = ~(err <= allowed)
    ratio = np.where(np.isnan(err), np.inf, err / allowed)
    return Report(name, int(got.size), int(bad.sum()), int(bad.sum()),
                  float(ratio.max()) if ratio.size else 0.0,
                  (int(np.argmax(ratio)),) if ratio.size else ())


def dx_scale(op: str, dy, x, gamma, mean, rstd, chunk: int = 1024) -> np.ndarray:
    """Per-row term scale of dx (float64 inputs), computed in row chunks."""
    M = x.shape[0]
    out = np.empty(M)
    for r0 in range(0, M, chunk):
        r1 = min(M, r0 + chunk)
        rs = rstd[r0:r1, None]
        m = (np.abs(x[r0:r1]) + np.abs(mean[r0:r1, None])) * rs if op == "ln" else np.abs(x[r0:r1]) * rs
        dyhat = dy[r0:r1] * gamma[None, :]
        t = np.abs(dyhat) + m * np.mean(np.abs(dyhat) * m, axis=1, keepdims=True)
        if op == "ln":
            t = t + np.mean(np.abs(dyhat), axis=1, keepdims=True)
        out[r0:r1] = rs[:, 0] * t.max(axis=1)
    return out


def y_scale(op: str, x, gamma, beta, mean, rstd, chunk: int = 1024) -> np.ndarray:
    M = x.shape[0]
    out = np.empty(M)
    for r0 in range(0, M, chunk):
        r1 = min(M, r0 + chunk)
        rs = rstd[r0:r1, None]
        m = (np.abs(x[r0:r1]) + np.abs(mean[r0:r1, None])) * rs if op == "ln" else np.abs(x[r0:r1]) * rs
        t = np.abs(gamma[None, :]) * m
        if op == "ln":
            t = t + np.abs(beta)[None, :]
        out[r0:r1] = t.max(axis=1)
    return out


def check_activation(name: str, got, ref, dtype: str, kind: str, dy, preact) -> Report:
    """dx = dy * f'(preact), elementwise (all arrays flat, float64).

    The term scale of an element is |dy| times the sum of the magnitudes of the
    terms that form f': SiLU  sigma(x) (1 + |x| (1 - sigma(x)));  GELU
    Phi(x) + |x| phi(x).  The A floor (2**-18 * s for every dtype) covers the
    cancellation at the zeros of f'.  An extra absolute floor 2**-149 (1 + |dy| (1 + |x|)) covers a float32
    intermediate that is subnormal (e^-|x| or phi(x) far in the tail, whose
    absolute error is one subnormal quantum, scaled by the factors after it).
    """
    from scipy.special import expit, ndtr

    x = np.asarray(preact, dtype=np.float64).reshape(-1)
    d = np.abs(np.asarray(dy, dtype=np.float64).reshape(-1))
    ax = np.abs(x)
    if kind == "silu":
        sg = expit(x)
        t = sg * (1.0 + ax * expit(-x))
    else:
        t = ndtr(x) + ax * np.exp(-0.5 * np.minimum(ax, 40.0) ** 2) / np.sqrt(2.0 * np.pi)
    scale = d * t
    floor = 2.0 ** -149 * (1.0 + d * (1.0 + ax))
    return check_elementwise(name, np.asarray(got, dtype=np.float64).reshape(-1, 1),
                             np.asarray(ref, dtype=np.float64).reshape(-1, 1), dtype, scale,
                             floor.reshape(-1, 1), a_exp=-18)

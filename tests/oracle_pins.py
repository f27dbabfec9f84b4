"""Checks that pin the float64 oracle to facts other than itself.

Each ``pin_*`` function takes a loaded oracle library (the real one, or a copy
with a planted mistake) and raises ``AssertionError`` if the oracle disagrees
with what the pages and the mathematics fix:

* ``pin_finite_differences``: the backward equals the numerical derivative of
  L = sum(dy * y) taken through the oracle's own forward (a five-point
  central stencil), for x, gamma and beta, on tiny shapes.
* ``pin_sympy_exact``: the backward equals the exact symbolic derivative of
  the forward's definition (page "Norm backward in Triton — the dγ/dβ
  reduction", section "The gradients"), built and differentiated by sympy and
  evaluated at rational points; the forward equals the definition evaluated
  exactly.
* ``pin_torch_fp64``: forward and backward equal torch's CPU float64
  layer_norm / rms_norm with autograd (a library special case).
* ``pin_invariants``: sum_j dx = 0 for LayerNorm (any eps); sum_j xhat*dx = 0
  at eps = 0 (both norms); LayerNorm's translation invariance and, at eps = 0,
  scale invariance; dx linear in dy; a constant row gives xhat = 0, y = beta
  and dx = rstd*(dyhat - mean(dyhat)); N = 2, eps = 0 gives xhat = +-1.
* ``pin_rms_is_ln_without_mean``: on rows of zero mean with dy*gamma of zero
  mean, LayerNorm's y - beta, dx and dgamma equal RMSNorm's.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

import oracle
import workloads as wl


def _rand(seed, stream, shape, scale=1.0, shift=0.0):
    n = int(np.prod(shape))
    return shift + scale * wl.normal(seed, stream, n).reshape(shape)


def _small_case(seed, M, N, op):
    x = _rand(seed, 11, (M, N))
    dy = _rand(seed, 12, (M, N))
    g = _rand(seed, 13, (N,), 0.3, 1.0)
    b = _rand(seed, 14, (N,), 0.3) if op == "ln" else None
    return x, dy, g, b


def _loss(lib, op, x, g, b, dy, eps):
    if op == "ln":
        y, _, _ = oracle.ln_fwd(x, g, b, eps, lib=lib)
    else:
        y, _ = oracle.rms_fwd(x, g, eps, lib=lib)
    return float(np.sum(dy * y))


def _analytic(lib, op, x, g, b, dy, eps):
    if op == "ln":
        _, mean, rstd = oracle.ln_fwd(x, g, b, eps, lib=lib)
        dx, dg, db = oracle.ln_bwd(dy, x, g, mean, rstd, lib=lib)
        return dx, dg, db
    _, rstd = oracle.rms_fwd(x, g, eps, lib=lib)
    dx, dg = oracle.rms_bwd(dy, x, g, rstd, lib=lib)
    return dx, dg, None


def _fd(f, a, h):
    """Five-point central difference of scalar f w.r.t. each element of a."""
    out = np.empty_like(a)
    flat = a.reshape(-1)
    o = out.reshape(-1)
    for i in range(flat.size):
        v = flat[i]
        vals = []
        for k in (2, 1, -1, -2):
            flat[i] = v + k * h
            vals.append(f())
        flat[i] = v
        o[i] = (-vals[0] + 8 * vals[1] - 8 * vals[2] + vals[3]) / (12 * h)
    return out


def _close(got, want, rtol, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(want))) if want.size else 1.0)
    err = float(np.max(np.abs(got - want))) if want.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err <= rtol * scale, f"{what}: max err {err:.3e} > {rtol:.1e} * {scale:.3e}"


FD_SHAPES = [(1, 1), (1, 2), (3, 5), (2, 8), (1, 33)]


def pin_finite_differences(lib, shapes=FD_SHAPES, eps_list=(1e-5, 0.3)):
    for op in ("ln", "rms"):
        for (M, N) in shapes:
            for eps in eps_list:
                x, dy, g, b = _small_case(7 * M + N, M, N, op)
                dx, dg, db = _analytic(lib, op, x, g, b, dy, eps)
                f = lambda: _loss(lib, op, x, g, b, dy, eps)  # noqa: E731
                tag = f"{op} M={M} N={N} eps={eps}"
                _close(dx, _fd(f, x, 1e-4), 1e-7, f"FD dx {tag}")
                _close(dg, _fd(f, g, 1e-4), 1e-7, f"FD dgamma {tag}")
                if op == "ln":
                    _close(db, _fd(f, b, 1e-4), 1e-7, f"FD dbeta {tag}")


def pin_sympy_exact(lib):
    import sympy as sp

    cases = [
        ("ln", [Fraction(1, 2), Fraction(-3, 4), Fraction(2, 1)], Fraction(1, 10)),
        ("ln", [Fraction(0), Fraction(1), Fraction(2), Fraction(-5, 3)], Fraction(0)),
        ("rms", [Fraction(1, 2), Fraction(-3, 4), Fraction(2, 1)], Fraction(1, 10)),
        ("rms", [Fraction(3), Fraction(-1), Fraction(1, 4), Fraction(7, 5)], Fraction(0)),
    ]
    for op, xv, epsv in cases:
        N = len(xv)
        xs = sp.symbols(f"x0:{N}")
        gs = sp.symbols(f"g0:{N}")
        bs = sp.symbols(f"b0:{N}")
        dyv = [sp.Rational(3 * j - 2, 5) for j in range(N)]
        gv = [sp.Rational(7 + j, 8) for j in range(N)]
        bv = [sp.Rational(1 - 2 * j, 9) for j in range(N)]
        eps = sp.Rational(epsv.numerator, epsv.denominator)
        if op == "ln":
            mu = sum(xs) / N
            var = sum((xi - mu) ** 2 for xi in xs) / N
            sigma = sp.sqrt(var + eps)
            ys = [gs[j] * (xs[j] - mu) / sigma + bs[j] for j in range(N)]
        else:
            sigma = sp.sqrt(sum(xi ** 2 for xi in xs) / N + eps)
            ys = [gs[j] * xs[j] / sigma for j in range(N)]
        L = sum(dyv[j] * ys[j] for j in range(N))
        subs = {xs[j]: sp.Rational(xv[j].numerator, xv[j].denominator) for j in range(N)}
        subs.update({gs[j]: gv[j] for j in range(N)})
        subs.update({bs[j]: bv[j] for j in range(N)})
        ev = lambda e: float(sp.N(e.subs(subs), 40))  # noqa: E731
        y_ex = np.array([[ev(yj) for yj in ys]])
        dx_ex = np.array([[ev(sp.diff(L, xs[i])) for i in range(N)]])
        dg_ex = np.array([ev(sp.diff(L, gs[i])) for i in range(N)])
        x = np.array([[float(v) for v in xv]])
        dy = np.array([[float(v) for v in dyv]])
        g = np.array([float(v) for v in gv])
        b = np.array([float(v) for v in bv])
        tag = f"{op} N={N} eps={epsv}"
        if op == "ln":
            y, mean, rstd = oracle.ln_fwd(x, g, b, float(eps), lib=lib)
            dx, dg, db = oracle.ln_bwd(dy, x, g, mean, rstd, lib=lib)
            db_ex = np.array([ev(sp.diff(L, bs[i])) for i in range(N)])
            _close(db, db_ex, 1e-13, f"sympy dbeta {tag}")
            _close(rstd, [ev(1 / sigma)], 1e-13, f"sympy rstd {tag}")
            _close(mean, [ev(mu)], 1e-13, f"sympy mean {tag}")
        else:
            y, rstd = oracle.rms_fwd(x, g, float(eps), lib=lib)
            dx, dg = oracle.rms_bwd(dy, x, g, rstd, lib=lib)
            _close(rstd, [ev(1 / sigma)], 1e-13, f"sympy rstd {tag}")
        _close(y, y_ex, 1e-13, f"sympy y {tag}")
        _close(dx, dx_ex, 1e-13, f"sympy dx {tag}")
        _close(dg, dg_ex, 1e-13, f"sympy dgamma {tag}")


def pin_torch_fp64(lib, shapes=((16, 100), (3, 7), (5, 1), (2, 512))):
    import torch
    import torch.nn.functional as F

    for (M, N) in shapes:
        for op in ("ln", "rms"):
            for eps in (1e-5, 0.05):
                x, dy, g, b = _small_case(M * 1000 + N, M, N, op)
                xt = torch.tensor(x, requires_grad=True)
                gt = torch.tensor(g, requires_grad=True)
                tag = f"{op} {M}x{N} eps={eps}"
                if op == "ln":
                    bt = torch.tensor(b, requires_grad=True)
                    yt = F.layer_norm(xt, (N,), gt, bt, eps)
                    _, mt, rt = torch.ops.aten.native_layer_norm(xt.detach(), [N], gt.detach(), bt.detach(), eps)
                else:
                    yt = F.rms_norm(xt, (N,), gt, eps)
                yt.backward(torch.tensor(dy))
                if op == "ln":
                    y, mean, rstd = oracle.ln_fwd(x, g, b, eps, lib=lib)
                    dx, dg, db = oracle.ln_bwd(dy, x, g, mean, rstd, lib=lib)
                    _close(mean, mt.reshape(-1).numpy(), 1e-12, f"torch mean {tag}")
                    _close(rstd, rt.reshape(-1).numpy(), 1e-12, f"torch rstd {tag}")
                    _close(db, bt.grad.numpy(), 1e-12, f"torch dbeta {tag}")
                else:
                    y, rstd = oracle.rms_fwd(x, g, eps, lib=lib)
                    dx, dg = oracle.rms_bwd(dy, x, g, rstd, lib=lib)
                _close(y, yt.detach().numpy(), 1e-12, f"torch y {tag}")
                _close(dx, xt.grad.numpy(), 1e-12, f"torch dx {tag}")
                _close(dg, gt.grad.numpy(), 1e-12, f"torch dgamma {tag}")


def pin_invariants(lib):
    M, N = 6, 37
    x, dy, g, b = _small_case(99, M, N, "ln")
    for eps in (1e-5, 0.5):
        y, mean, rstd = oracle.ln_fwd(x, g, b, eps, lib=lib)
        dx, dg, db = oracle.ln_bwd(dy, x, g, mean, rstd, lib=lib)
        # sum_j dx = 0 for LayerNorm, any eps (sum of xhat is 0)
        _close(dx.sum(axis=1), np.zeros(M), 1e-13, f"LN sum dx eps={eps}")
        # translation invariance of LayerNorm
        y2, _, _ = oracle.ln_fwd(x + 3.25, g, b, eps, lib=lib)
        _close(y2, y, 1e-12, f"LN translation y eps={eps}")
        _, m2, r2 = oracle.ln_fwd(x + 3.25, g, b, eps, lib=lib)
        dx2, _, _ = oracle.ln_bwd(dy, x + 3.25, g, m2, r2, lib=lib)
        _close(dx2, dx, 1e-12, f"LN translation dx eps={eps}")
        # dx linear in dy
        dyb = _rand(5, 21, (M, N))
        dxa, dga, dba = oracle.ln_bwd(2.0 * dy - 0.5 * dyb, x, g, mean, rstd, lib=lib)
        dxb, dgb, dbb = oracle.ln_bwd(dyb, x, g, mean, rstd, lib=lib)
        _close(dxa, 2.0 * dx - 0.5 * dxb, 1e-13, "LN dx linear in dy")
        _close(dga, 2.0 * dg - 0.5 * dgb, 1e-13, "LN dgamma linear in dy")
        _close(dba, 2.0 * db - 0.5 * dbb, 1e-13, "LN dbeta linear in dy")
    # eps = 0: sum_j xhat*dx = 0 and scale invariance, both norms
    y, mean, rstd = oracle.ln_fwd(x, g, b, 0.0, lib=lib)
    dx, _, _ = oracle.ln_bwd(dy, x, g, mean, rstd, lib=lib)
    xhat = (x - mean[:, None]) * rstd[:, None]
    _close((xhat * dx).sum(axis=1), np.zeros(M), 1e-12, "LN sum xhat*dx (eps=0)")
    _close((xhat ** 2).mean(axis=1), np.ones(M), 1e-13, "LN mean xhat^2 = 1 (eps=0)")
    y3, m3, r3 = oracle.ln_fwd(4.0 * x, g, b, 0.0, lib=lib)
    _close(y3, y, 1e-12, "LN scale invariance y")
    dx3, _, _ = oracle.ln_bwd(dy, 4.0 * x, g, m3, r3, lib=lib)
    _close(4.0 * dx3, dx, 1e-12, "LN scale dx(a x) = dx(x)/a")
    yr, rr = oracle.rms_fwd(x, g, 0.0, lib=lib)
    dxr, _ = oracle.rms_bwd(dy, x, g, rr, lib=lib)
    xhr = x * rr[:, None]
    _close((xhr * dxr).sum(axis=1), np.zeros(M), 1e-12, "RMS sum xhat*dx (eps=0)")
    _close((xhr ** 2).mean(axis=1), np.ones(M), 1e-13, "RMS mean xhat^2 = 1 (eps=0)")
    yr3, rr3 = oracle.rms_fwd(4.0 * x, g, 0.0, lib=lib)
    _close(yr3, yr, 1e-12, "RMS scale invariance y")
    dxr3, _ = oracle.rms_bwd(dy, 4.0 * x, g, rr3, lib=lib)
    _close(4.0 * dxr3, dxr, 1e-12, "RMS scale dx(a x) = dx(x)/a")
    # constant rows: var = 0, xhat = 0, y = beta, rstd = 1/sqrt(eps)
    eps = 1e-3
    xc = np.full((2, N), 1.75)
    yc, mc, rc = oracle.ln_fwd(xc, g, b, eps, lib=lib)
    _close(yc, np.broadcast_to(b, (2, N)), 1e-13, "LN constant row y = beta")
    _close(rc, np.full(2, 1.0 / np.sqrt(eps)), 1e-13, "LN constant row rstd")
    dxc, _, _ = oracle.ln_bwd(dy[:2], xc, g, mc, rc, lib=lib)
    dyh = dy[:2] * g
    _close(dxc, rc[:, None] * (dyh - dyh.mean(axis=1, keepdims=True)), 1e-12,
           "LN constant row dx = rstd*(dyhat - mean(dyhat))")
    # N = 1: LayerNorm output is beta and dx is 0
    y1, m1, r1 = oracle.ln_fwd(x[:, :1], g[:1], b[:1], 1e-5, lib=lib)
    _close(y1, np.broadcast_to(b[:1], (M, 1)), 1e-13, "LN N=1 y = beta")
    dx1, _, _ = oracle.ln_bwd(dy[:, :1], x[:, :1], g[:1], m1, r1, lib=lib)
    _close(dx1, np.zeros((M, 1)), 1e-13, "LN N=1 dx = 0")
    # N = 2, eps = 0: xhat = +-1, so y = +-gamma + beta
    x2 = np.array([[0.25, -1.5], [3.0, 7.0]])
    y2, _, _ = oracle.ln_fwd(x2, g[:2], b[:2], 0.0, lib=lib)
    want = np.array([[g[0] + b[0], -g[1] + b[1]], [-g[0] + b[0], g[1] + b[1]]])
    _close(y2, want, 1e-13, "LN N=2 closed form")
    # M = 0: the per-feature sums are zero
    _, dg0, db0 = oracle.ln_bwd(np.zeros((0, N)), np.zeros((0, N)), g, np.zeros(0), np.zeros(0), lib=lib)
    _close(dg0, np.zeros(N), 0.0, "LN M=0 dgamma")
    _close(db0, np.zeros(N), 0.0, "LN M=0 dbeta")


def pin_rms_is_ln_without_mean(lib):
    M, N = 4, 24
    half = _rand(3, 31, (M, N // 2))
    x = np.empty((M, N))
    x[:, 0::2], x[:, 1::2] = half, -half  # rows of exactly zero mean
    dyh = _rand(3, 32, (M, N // 2))
    dy = np.empty((M, N))
    dy[:, 0::2], dy[:, 1::2] = dyh, -dyh
    g = np.ones(N)  # so dyhat = dy has zero row mean too
    b = np.zeros(N)
    for eps in (1e-5, 0.2):
        yl, ml, rl = oracle.ln_fwd(x, g, b, eps, lib=lib)
        yr, rr = oracle.rms_fwd(x, g, eps, lib=lib)
        _close(ml, np.zeros(M), 1e-15, "zero-mean rows")
        _close(yl, yr, 1e-14, f"LN y = RMS y on zero-mean rows eps={eps}")
        _close(rl, rr, 1e-14, f"LN rstd = RMS rstd eps={eps}")
        dxl, dgl, _ = oracle.ln_bwd(dy, x, g, ml, rl, lib=lib)
        dxr, dgr = oracle.rms_bwd(dy, x, g, rr, lib=lib)
        _close(dxl, dxr, 1e-14, f"LN dx = RMS dx eps={eps}")
        _close(dgl, dgr, 1e-14, f"LN dgamma = RMS dgamma eps={eps}")


ALL_PINS = (pin_finite_differences, pin_sympy_exact, pin_torch_fp64, pin_invariants,
            pin_rms_is_ln_without_mean)


def pin_activation(lib):
    """SiLU / GELU backward: finite differences of the forward, exact values,
    limits, and torch float64 autograd."""
    import torch
    import torch.nn.functional as F

    x = np.concatenate([np.linspace(-12, 12, 97), wl.normal(4, 51, 200) * 3])
    dy = wl.normal(4, 52, x.size)
    for kind in ("silu", "gelu"):
        dx = oracle.act_bwd(kind, dy, x, lib=lib)
        # five-point finite differences of the forward, elementwise
        h = 1e-3
        f = lambda t: oracle.act_fwd(kind, t, lib=lib)  # noqa: E731
        fd = (-f(x + 2 * h) + 8 * f(x + h) - 8 * f(x - h) + f(x - 2 * h)) / (12 * h)
        _close(dx, dy * fd, 1e-9, f"FD {kind}")
        # torch autograd in float64
        xt = torch.tensor(x, requires_grad=True)
        (F.silu(xt) if kind == "silu" else F.gelu(xt)).backward(torch.tensor(dy))
        _close(dx, xt.grad.numpy(), 1e-13, f"torch {kind}")
        # f'(0) = 1/2 for both; f' -> 1 for large x, -> 0 for very negative x
        one = np.ones(1)
        _close(oracle.act_bwd(kind, one, np.zeros(1), lib=lib), [0.5], 1e-15, f"{kind}'(0)")
        _close(oracle.act_bwd(kind, one, np.array([40.0]), lib=lib), [1.0], 1e-12, f"{kind}'(+inf)")
        _close(oracle.act_bwd(kind, one, np.array([-40.0]), lib=lib), [0.0], 1e-12, f"{kind}'(-inf)")
    # lower tails, relative to closed forms that use neither erf nor the oracle's sigma:
    # GELU'(x) = phi(x) (Phi(x) / phi(x) - |x|), with Mills' ratio Phi(x) / phi(x)
    # = (1/|x|) sum_k (-1)^k (2k-1)!! / x^(2k) (asymptotic; summed to its smallest term)
    for t in (-9.0, -12.0, -16.0, -20.0, -25.0, -30.0, -35.0):
        term, mills, k = 1.0, 0.0, 0
        while True:
            mills += term
            nxt = -term * (2 * k + 1) / (t * t)
            if abs(nxt) >= abs(term) or abs(nxt) < 1e-18:
                break
            term, k = nxt, k + 1
        pdf = np.exp(-0.5 * t * t) / np.sqrt(2.0 * np.pi)
        want = pdf * (mills / abs(t) - abs(t))
        got = oracle.act_bwd("gelu", np.ones(1), np.array([t]), lib=lib)[0]
        assert abs(got - want) <= 1e-12 * abs(want), ("GELU' lower tail", t, got, want)
        # sigma(x) = e^x - e^(2x) + O(e^(3x)) gives, as x -> -inf,
        # SiLU'(x) = e^x (1 + x) - e^(2x) (1 + 2x) + O(x e^(3x))
        want = np.exp(t) * (1.0 + t) - np.exp(2.0 * t) * (1.0 + 2.0 * t)
        got = oracle.act_bwd("silu", np.ones(1), np.array([t]), lib=lib)[0]
        assert abs(got - want) <= 1e-7 * abs(want), ("SiLU' lower tail", t, got, want)
    # SiLU has its minimum at x* = -1.27846454276107..., where 1 + x*(1 - sigma(x*)) = 0:
    # its derivative vanishes there
    m = oracle.act_bwd("silu", np.ones(1), np.array([-1.2784645427610738]), lib=lib)[0]
    assert abs(m) < 1e-12, m


ALL_PINS = ALL_PINS + (pin_activation,)

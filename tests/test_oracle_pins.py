"""The float64 oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle
import oracle_pins as pins
import numpy as np
import workloads as wl


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


def test_finite_differences(lib):
    pins.pin_finite_differences(lib)


def test_sympy_exact_derivative(lib):
    pytest.importorskip("sympy")
    pins.pin_sympy_exact(lib)


def test_torch_fp64_cross_check(lib):
    pins.pin_torch_fp64(lib)


def test_invariants_and_closed_forms(lib):
    pins.pin_invariants(lib)


def test_rms_is_ln_without_the_mean(lib):
    pins.pin_rms_is_ln_without_mean(lib)


def test_activation_backward(lib):
    pins.pin_activation(lib)


def test_threaded_timing_mode_equals_the_single_thread_oracle():
    """The CPU baseline's threaded mode runs the same per-row loops on row
    blocks: dx bit for bit, dgamma / dbeta up to the grouping of the sums."""
    lib = oracle.load()
    for op, M, N, th in (("rms", 37, 65, 4), ("ln", 50, 33, 7), ("ln", 3, 8, 16)):
        x = wl.normal(11, 1, M * N).reshape(M, N) * 2 + 0.5
        dy = wl.normal(11, 2, M * N).reshape(M, N)
        g = 1 + 0.1 * wl.normal(11, 3, N)
        if op == "ln":
            _, mean, rstd = oracle.ln_fwd(x, g, np.zeros(N), 1e-5, lib=lib)
            a = oracle.ln_bwd(dy, x, g, mean, rstd, lib=lib)
            b = oracle.ln_bwd(dy, x, g, mean, rstd, lib=lib, threads=th)
        else:
            _, rstd = oracle.rms_fwd(x, g, 1e-6, lib=lib)
            a = oracle.rms_bwd(dy, x, g, rstd, lib=lib)
            b = oracle.rms_bwd(dy, x, g, rstd, lib=lib, threads=th)
        assert np.array_equal(a[0], b[0])
        for u, v in zip(a[1:], b[1:]):
            np.testing.assert_allclose(v, u, rtol=1e-13, atol=1e-13)

"""The float64 oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle
import oracle_pins as pins


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

"""Plants plausible mistakes in copies of the oracle and checks the pins catch each one.

Every mutant is a text edit of ``oracle/norm_oracle.c`` compiled into a
temporary library on the CPU; the real oracle is untouched.
"""
import os

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "norm_oracle.c")

# (name, text to find, replacement, occurrence index)
MUTANTS = [
    ("ln dx drops mean(dyhat)", "dyhat - mean_dyhat - xhat", "dyhat - xhat", 0),
    ("ln dx sign of xhat term", "rs * (dyhat - mean_dyhat - xhat * mean_dyhat_xhat)",
     "rs * (dyhat - mean_dyhat + xhat * mean_dyhat_xhat)", 0),
    ("rms dx sign of xhat term", "rs * (dyhat - xhat * mean_dyhat_xhat)",
     "rs * (dyhat + xhat * mean_dyhat_xhat)", 0),
    ("rms dx missing rstd factor", "dx[r * N + j] = rs * (dyhat - xhat", "dx[r * N + j] = (dyhat - xhat", 0),
    ("unbiased variance", "const double var = sq / (double)N;", "const double var = sq / (double)(N + 1);", 0),
    ("eps outside the root", "1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)", 0),
    ("rms eps dropped", "1.0 / sqrt(ms + eps)", "1.0 / sqrt(ms)", 0),
    ("ln mean not divided by N", "const double mu = sum / (double)N;", "const double mu = sum / (double)(N + 1);", 0),
    ("ln dgamma without xhat", "dgamma[j] += dyr[j] * xhat;\n            dbeta", "dgamma[j] += dyr[j];\n            dbeta", 0),
    ("rms dgamma uses dyhat", "dgamma[j] += dyr[j] * xhat;\n        }\n    }\n}\n",
     "dgamma[j] += dyr[j] * gamma[j] * xhat;\n        }\n    }\n}\n", 0),
    ("ln dbeta uses dyhat", "dbeta[j] += dyr[j];", "dbeta[j] += dyr[j] * gamma[j];", 0),
    ("rms wrong row stride", "const double *xr = x + r * N;\n        const double *dyr = dy + r * N;\n        const double rs = rstd[r];\n        double s2",
     "const double *xr = x + r;\n        const double *dyr = dy + r * N;\n        const double rs = rstd[r];\n        double s2", 0),
    ("ln gamma index transposed", "const double dyhat = dyr[j] * gamma[j];\n            s1",
     "const double dyhat = dyr[j] * gamma[r % N];\n            s1", 0),
    ("ln y missing beta", "y[r * N + j] = gamma[j] * xhat + beta[j];", "y[r * N + j] = gamma[j] * xhat;", 0),
    ("silu derivative missing the x term", "dx[i] = dy[i] * (s * (1.0 + x * (1.0 - s)));", "dx[i] = dy[i] * s;", 0),
    ("gelu derivative missing the pdf term", "dx[i] = dy[i] * (cdf + x * pdf);", "dx[i] = dy[i] * cdf;", 0),
    ("gelu erfc argument unscaled", "const double cdf = 0.5 * erfc(-x * inv_sqrt2);", "const double cdf = 0.5 * erfc(-x);", 0),
    ("gelu distribution function through 1 + erf (lower-tail cancellation)",
     "const double cdf = 0.5 * erfc(-x * inv_sqrt2);", "const double cdf = 0.5 * (1.0 + erf(x * inv_sqrt2));", 0),
    ("ln c2 divided by N-1", "const double mean_dyhat_xhat = s2 / (double)N;\n        for (int64_t j = 0; j < N; ++j) {\n            const double xhat = (xr[j] - mu) * rs;",
     "const double mean_dyhat_xhat = s2 / (double)(N + 1);\n        for (int64_t j = 0; j < N; ++j) {\n            const double xhat = (xr[j] - mu) * rs;", 0),
]


def _mutate(text, find, repl, occ):
    idx = -1
    for _ in range(occ + 1):
        idx = text.index(find, idx + 1)
    return text[:idx] + repl + text[idx + len(find):]


@pytest.mark.parametrize("name,find,repl,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, find, repl, occ):
    text = open(SRC).read()
    assert find in text, f"mutation site for '{name}' not found"
    src = tmp_path / "mutant.c"
    src.write_text(_mutate(text, find, repl, occ))
    lib = oracle.load(oracle.build(str(src), str(tmp_path / "libmutant.so")))
    caught = []
    for pin in pins.ALL_PINS:
        if pin is pins.pin_sympy_exact:
            try:
                import sympy  # noqa: F401
            except ImportError:
                continue
        try:
            pin(lib)
        except (AssertionError, FloatingPointError, ValueError, ZeroDivisionError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"

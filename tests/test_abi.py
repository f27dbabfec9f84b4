"""The C-ABI library: it builds, loads, exports every symbol the header
declares, and rejects bad arguments on the host (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbnorm.h")


@pytest.fixture(scope="module")
def lib():
    from rmsnorm_backward_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("ln_fwd", "ln_bwd", "rms_fwd", "rms_bwd", "gbn_bwd_workspace_bytes", "gbn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libgbnorm.so does not export {name}"


def test_status_strings(lib):
    lib.gbn_status_string.restype = ctypes.c_char_p
    lib.gbn_status_string.argtypes = [ctypes.c_int]
    assert lib.gbn_status_string(0) == b"ok"
    assert b"workspace" in lib.gbn_status_string(4)
    assert lib.gbn_status_string(99) == b"unknown status"


def test_host_side_argument_checks(lib):
    import rmsnorm_backward_gb300 as gbn
    L = gbn._declare(ctypes.CDLL(gbn.build.LIB if hasattr(gbn, "build") else gbn.library_path))
    p = ctypes.c_void_p(16)
    # null pointers with rows to process
    assert L.ln_fwd(None, p, p, p, p, p, 1e-5, 4, 8, 2, None) == 1
    assert L.rms_fwd(p, None, p, p, 1e-5, 4, 8, 2, None) == 1
    assert L.rms_bwd(p, p, p, p, p, None, 0.0, 4, 8, 2, p, 1 << 20, None) == 1
    assert L.ln_bwd(p, p, p, p, p, p, p, None, 0.0, 4, 8, 2, p, 1 << 20, None) == 1
    # unknown dtype, bad sizes, bad eps
    assert L.rms_fwd(p, p, p, p, 1e-5, 4, 8, 7, None) == 2
    assert L.rms_fwd(p, p, p, p, 1e-5, -1, 8, 2, None) == 1
    assert L.rms_fwd(p, p, p, p, 1e-5, 4, 0, 2, None) == 1
    assert L.rms_fwd(p, p, p, p, -1.0, 4, 8, 2, None) == 1
    assert L.rms_fwd(p, p, p, p, float("nan"), 4, 8, 2, None) == 1
    assert L.rms_fwd(p, p, p, p, 1e-5, 4, (1 << 24) + 1, 2, None) == 1
    # nothing to do
    assert L.rms_fwd(None, None, None, None, 1e-5, 0, 8, 2, None) == 0
    assert L.gbn_bwd_workspace_bytes(0, 8, 2, 0) == 0
    assert L.gbn_bwd_workspace_bytes(4, 8, 9, 0) == 0


def test_activation_host_checks(lib):
    import rmsnorm_backward_gb300 as gbn
    L = gbn._declare(ctypes.CDLL(gbn.library_path))
    p = ctypes.c_void_p(16)
    for fn in (L.silu_bwd, L.gelu_bwd):
        assert fn(p, p, p, 0, 2, None) == 0       # empty: no-op, no device needed
        assert fn(None, p, p, 8, 2, None) == 1    # null pointer
        assert fn(p, p, None, 8, 2, None) == 1
        assert fn(p, p, p, -1, 2, None) == 1      # negative size
        assert fn(p, p, p, 8, 5, None) == 2       # unknown dtype


def test_host_buffer_entry_checks(lib):
    import rmsnorm_backward_gb300 as gbn
    L = gbn._declare(ctypes.CDLL(gbn.library_path))
    p = ctypes.c_void_p(16)
    assert L.rms_bwd_host(None, p, p, p, p, p, 4, 8, 2, p, 1 << 20, None) == 1     # null input
    assert L.rms_bwd_host(p, p, p, p, p, None, 4, 8, 2, p, 1 << 20, None) == 1     # null dgamma
    assert L.rms_bwd_host(p, p, p, p, p, p, 4, 8, 7, p, 1 << 20, None) == 2        # dtype
    assert L.rms_bwd_host(p, p, p, p, p, p, -1, 8, 2, p, 1 << 20, None) == 1       # M < 0
    assert L.ln_bwd_host(p, p, p, None, p, p, p, p, 4, 8, 2, p, 1 << 20, None) == 1  # LayerNorm without mean
    assert L.ln_bwd_host(p, p, p, p, p, p, p, None, 4, 8, 2, p, 1 << 20, None) == 1  # LayerNorm without dbeta


def test_activation_host_entry_checks(lib):
    import rmsnorm_backward_gb300 as gbn
    L = gbn._declare(ctypes.CDLL(gbn.library_path))
    p = ctypes.c_void_p(16)
    for fn in (L.silu_bwd_host, L.gelu_bwd_host):
        assert fn(p, p, p, 0, 2, p, 1 << 20, None) == 0      # empty: no-op
        assert fn(None, p, p, 8, 2, p, 1 << 20, None) == 1   # null input
        assert fn(p, p, p, 8, 2, None, 1 << 20, None) == 1   # no workspace
        assert fn(p, p, p, -1, 2, p, 1 << 20, None) == 1     # negative size
        assert fn(p, p, p, 8, 9, p, 1 << 20, None) == 2      # unknown dtype


def test_option_fields_are_checked_on_the_host(lib):
    """gbn_options: an unknown kernel, a negative wait limit, a host chunk on
    a device call, or a device-call field on a host-buffer call are
    GBN_EINVAL before anything is enqueued (no GPU needed)."""
    import rmsnorm_backward_gb300 as gbn
    L = gbn._declare(ctypes.CDLL(gbn.library_path))
    p = ctypes.c_void_p(16)

    def opt(**kw):
        o = gbn.GbnOptions()
        for k, v in kw.items():
            setattr(o, k, v)
        return ctypes.byref(o)

    assert ctypes.sizeof(gbn.GbnOptions) == 56 and gbn.GbnOptions.host_chunk.offset == 40
    for bad in (opt(kernel=3), opt(kernel=-1), opt(wait_limit_ns=-1), opt(host_chunk=64)):
        assert L.rms_bwd_ex(p, p, p, p, p, p, 0.0, 4, 8, 2, p, 1 << 20, bad, None) == 1
        assert L.rms_fwd_ex(p, p, p, p, 1e-5, 4, 8, 2, bad, None) == 1
    for bad in (opt(ld_x=8), opt(accumulate=1), opt(grad_dtype=2), opt(reduce_mode=1), opt(host_chunk=-1),
                opt(kernel=7)):
        assert L.rms_bwd_host_ex(p, p, p, p, p, p, 4, 8, 2, p, 1 << 20, bad, None) == 1
        assert L.ln_bwd_host_ex(p, p, p, p, p, p, p, p, 4, 8, 2, p, 1 << 20, bad, None) == 1
        assert L.silu_bwd_host_ex(p, p, p, 8, 2, p, 1 << 20, bad, None) == 1
        assert L.gbn_bwd_host_workspace_bytes_ex(4, 8, 2, 0, bad) == 0
        assert L.gbn_act_host_workspace_bytes_ex(8, 2, bad) == 0


def test_library_reads_no_environment():
    """No knob of the environment reaches the library: which kernel runs
    and the summation order of dgamma / dbeta depend only on the call."""
    csrc = os.path.join(ROOT, "rmsnorm_backward_gb300", "csrc")
    for name in os.listdir(csrc):
        text = open(os.path.join(csrc, name)).read()
        assert "getenv" not in text, f"{name} reads the environment"

"""rms_bwd_noalloc: the RMSNorm backward for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the backward (inside an
allocator callback, under a device-memory budget fixed up front, in loops
that cannot take a cudaMalloc's implicit synchronisation); rms_bwd_noalloc
keeps rms_bwd's partial rows in the library's own
static device array instead of a caller workspace.  These tests call it
through the C ABI and hold it to rms_bwd's output with the parity tolerance
of the other tests, on two calls in a row (the second call starts from the
first call's leftover scratch contents).  This file sorts last so that a
failure here cannot hide another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import rmsnorm_backward_gb300 as gbn
import tolerance as tol
import workloads as wl

pytestmark = pytest.mark.gpu

_vp, _i64, _int, _f = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float


def _entry():
    fn = gbn.lib().rms_bwd_noalloc
    fn.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _f, _i64, _i64, _int, _vp]
    fn.restype = _int
    return fn


def _call(fn, dy, x, g, rstd, dx, dg):
    M, N = x.shape
    return fn(dy.data_ptr(), x.data_ptr(), g.data_ptr(), rstd.data_ptr(), dx.data_ptr(), dg.data_ptr(), 0.0,
              M, N, gbn.DTYPE_CODES[x.dtype], torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,M", [("rms_bf16_16384x4096", None), ("rms_bf16_8192x16384", 1000),
                                    ("rms_bf16_16384x4096", 37)])
def test_noalloc_matches_rms_bwd_on_two_calls_in_a_row(name, M):
    w = wl.WORKLOADS[name]
    w = w.with_shape(M or w.M, w.N)
    d = {k: v.cuda() for k, v in wl.make_inputs(w).items()}
    y, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
    dx_ref, dg_ref = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd)
    fn = _entry()
    x64 = wl.exact_double(d["x"].cpu())
    scale = tol.dx_scale("rms", wl.exact_double(d["dy"].cpu()), x64, wl.exact_double(d["gamma"].cpu()),
                         np.zeros(w.M), wl.exact_double(rstd.cpu()))
    for call in range(2):
        dx = torch.full_like(d["x"], float("nan"))
        dg = torch.full((w.N,), float("nan"), device="cuda")
        assert _call(fn, d["dy"], d["x"], d["gamma"], rstd, dx, dg) == 0
        torch.cuda.synchronize()
        r_dx = tol.check_elementwise(f"dx call {call}", wl.exact_double(dx.cpu()),
                                     wl.exact_double(dx_ref.cpu()), w.dtype, scale)
        r_dg = tol.check_param_grad(f"dgamma call {call}", dg.cpu().double().numpy(),
                                    dg_ref.cpu().double().numpy())
        assert r_dx.ok() and r_dg.ok(), f"{r_dx}\n{r_dg}"
    assert gbn.device_error() == 0


def test_noalloc_refuses_problems_beyond_its_scratch():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = 32768
    assert gbn.bwd_workspace_bytes(sms, N, torch.bfloat16, False) > (16 << 20)
    x = torch.zeros(sms, N, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(sms, dtype=torch.float32, device="cuda")
    dx = torch.empty_like(x)
    dg = torch.empty(N, dtype=torch.float32, device="cuda")
    assert _call(_entry(), x, x, g, rstd, dx, dg) == 7
    assert "static scratch" in gbn.status_string(7)
    torch.cuda.synchronize()

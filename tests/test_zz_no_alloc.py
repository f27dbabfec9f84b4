"""rms_bwd_noalloc: the RMSNorm backward for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the backward (inside an
allocator callback, under a device-memory budget fixed up front, in loops
that cannot take a cudaMalloc's implicit synchronisation); rms_bwd_noalloc
keeps rms_bwd's partial rows in the library's own static device array
instead of a caller workspace.  These tests call it through the C ABI and
hold it to rms_bwd's output bit for bit (both run the same kernels with the
same row blocks and the same column-reduce order), on two calls in a row
(the second call starts from the first call's leftover scratch contents),
with saved rstd and without it (rstd recomputed from x with eps).  The
outputs sit between sentinel bands that must come back unchanged.  This
file sorts last so that a failure here cannot hide another test's result.
"""
import ctypes
import dataclasses

import pytest
import torch

import guards
import rmsnorm_backward_gb300 as gbn
import workloads as wl

pytestmark = pytest.mark.gpu

_vp, _i64, _int, _f = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float


def _entry():
    fn = gbn.lib().rms_bwd_noalloc
    fn.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _f, _i64, _i64, _int, _vp]
    fn.restype = _int
    return fn


def _call(fn, dy, x, g, rstd, dx, dg, eps=0.0):
    M, N = x.shape
    return fn(dy.data_ptr(), x.data_ptr(), g.data_ptr(), None if rstd is None else rstd.data_ptr(),
              dx.data_ptr(), dg.data_ptr(), eps, M, N, gbn.DTYPE_CODES[x.dtype],
              torch.cuda.current_stream().cuda_stream)


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("name,M,dtype", [("rms_bf16_16384x4096", None, "bf16"),
                                          ("rms_bf16_8192x16384", 1000, "bf16"),
                                          ("rms_bf16_16384x4096", 37, "bf16"),
                                          ("rms_bf16_16384x4096", 500, "f16"),
                                          ("rms_bf16_16384x4096", 300, "f32")])
@pytest.mark.parametrize("saved", [True, False])
def test_noalloc_matches_rms_bwd_on_two_calls_in_a_row(name, M, dtype, saved):
    w = wl.WORKLOADS[name]
    w = dataclasses.replace(w.with_shape(M or w.M, w.N), dtype=dtype)
    d = {k: v.cuda() for k, v in wl.make_inputs(w).items()}
    _, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
    if not saved:
        rstd = None
    dx_ref, dg_ref = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd, eps=None if saved else w.eps)
    fn = _entry()
    for call in range(2):
        g = guards.Guarded("cuda")
        dx = g.empty(tuple(d["x"].shape), d["x"].dtype, "dx")
        dg = g.empty((w.N,), torch.float32, "dgamma")
        assert _call(fn, d["dy"], d["x"], d["gamma"], rstd, dx, dg, 0.0 if saved else w.eps) == 0
        torch.cuda.synchronize()
        g.check()
        assert torch.equal(_bits(dx), _bits(dx_ref)), f"dx differs from rms_bwd on call {call}"
        assert torch.equal(_bits(dg), _bits(dg_ref)), f"dgamma differs from rms_bwd on call {call}"
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

"""The save-nothing backward (no saved statistics: the kernels form each row's
mean and rstd from x with eps) against the float64 oracle (needs a GPU)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_backward_gb300 as gbn
import tolerance as tol
import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [  # (workload family, dtype, M, N): staged kernels, then plain-load ones (N not 16-byte)
    ("rms_bf16_16384x4096", "bf16", 700, 4096),
    ("ln_bf16_65536x1024", "bf16", 700, 1024),
    ("ln_f16_1151x8192", "f16", 300, 8192),
    ("rms_bf16_8192x16384", "bf16", 200, 16384),
    ("ln_f32_64x256", "f32", 64, 256),
    ("ln_bf16_65536x1024", "bf16", 300, 1000),
    ("rms_bf16_16384x4096", "f32", 100, 333),
    # rows with large means next to their spread, in float32: the
    # statistics formed inside the kernels must not lose the variance to
    # cancellation
    ("ln_bf16_65536x1024", "f32", 300, 1024),
    ("ln_bf16_65536x1024", "f32", 200, 2000),
    ("ln_bf16_65536x1024", "bf16", 153, 16384),
    # RMSNorm with x held as raw vectors, the last vectors of a row unowned
    ("rms_bf16_8192x16384", "bf16", 100, 16000),
]


@pytest.mark.parametrize("family,dtype,M,N", CASES)
def test_backward_without_saved_statistics(family, dtype, M, N):
    _check_recompute(family, dtype, M, N)


@pytest.mark.parametrize("dtype,N", [("f32", 1024), ("bf16", 1024), ("f32", 4096)])
def test_backward_without_saved_statistics_outlier_first_column(dtype, N):
    """Column 0 of every row far from the rest (an outlier channel at the
    first feature): the statistics formed inside the kernels (the mean
    first, then the centred sums) keep their accuracy."""
    def bend(inp):
        inp["x"][:, 0] = inp["x"][:, 0] * 64 + 300
    _check_recompute("ln_bf16_65536x1024", dtype, 300, N, bend)


def _check_recompute(family, dtype, M, N, bend=None):
    w = dataclasses.replace(wl.WORKLOADS[family], dtype=dtype, M=M, N=N, name=f"{family}-{dtype}-{M}x{N}")
    inp = wl.make_inputs(w)
    if bend is not None:
        bend(inp)
    d = {k: v.cuda() for k, v in inp.items()}
    x, dy, g = (wl.exact_double(inp[k]) for k in ("x", "dy", "gamma"))
    if w.op == "ln":
        _, mean_o, rstd_o = oracle.ln_fwd(x, g, wl.exact_double(inp["beta"]), w.eps)
        dx_o, dg_o, db_o = oracle.ln_bwd(dy, x, g, mean_o, rstd_o)
        dx, dg, db = gbn.ln_bwd(d["dy"], d["x"], d["gamma"], None, None, eps=w.eps)
        _, mean, rstd = gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps)
        dx_s, dg_s, db_s = gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean, rstd)
        grads = [("dgamma", dg, dg_o), ("dbeta", db, db_o)]
    else:
        mean_o = np.zeros(M)
        _, rstd_o = oracle.rms_fwd(x, g, w.eps)
        dx_o, dg_o = oracle.rms_bwd(dy, x, g, rstd_o)
        dx, dg = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], None, eps=w.eps)
        _, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
        dx_s, dg_s = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd)
        grads = [("dgamma", dg, dg_o)]
    torch.cuda.synchronize()
    scale = tol.dx_scale(w.op, dy, x, g, mean_o, rstd_o)
    reps = [tol.check_elementwise("dx", wl.exact_double(dx.cpu()), dx_o, dtype, scale),
            tol.check_elementwise("dx vs saved-stats path", wl.exact_double(dx.cpu()),
                                  wl.exact_double(dx_s.cpu()), dtype, scale)]
    reps += [tol.check_param_grad(n, got.cpu().double().numpy(), ref) for n, got, ref in grads]
    assert all(r.ok() for r in reps), "\n".join(map(str, reps))
    assert gbn.device_error() == 0


def test_partial_statistics_are_rejected():
    x = torch.zeros(4, 64, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(64, device="cuda", dtype=torch.bfloat16)
    r = torch.ones(4, device="cuda")
    with pytest.raises(ValueError):
        gbn.ln_bwd(x, x, g, None, r, eps=1e-5)
    with pytest.raises(ValueError):
        gbn.rms_bwd(x, x, g, None)  # no eps
    L = gbn.lib()
    ws = torch.empty(gbn.bwd_workspace_bytes(4, 64, torch.bfloat16, True), dtype=torch.uint8, device="cuda")
    dg = torch.empty(64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # only one of mean / rstd, or a bad eps: GBN_EINVAL
    assert L.ln_bwd(x.data_ptr(), x.data_ptr(), g.data_ptr(), None, r.data_ptr(), x.data_ptr(), dg.data_ptr(),
                    dg.data_ptr(), 1e-5, 4, 64, 2, ws.data_ptr(), ws.numel(), s) == 1
    assert L.rms_bwd(x.data_ptr(), x.data_ptr(), g.data_ptr(), None, x.data_ptr(), dg.data_ptr(), -1.0, 4, 64, 2,
                     ws.data_ptr(), ws.numel(), s) == 1
    # the phase API needs the statistics
    assert L.rms_bwd_rows(x.data_ptr(), x.data_ptr(), g.data_ptr(), None, x.data_ptr(), 4, 64, 2, ws.data_ptr(),
                          ws.numel(), s) == 1
    torch.cuda.synchronize()

"""gbn_options: strided rows, accumulation into dgamma / dbeta and their cast
to the parameter dtype, against the float64 oracle (needs a GPU)."""
import ctypes

import numpy as np
import pytest
import torch

import gpu_parity
import oracle
import rmsnorm_backward_gb300 as gbn
import tolerance as tol
import workloads as wl

pytestmark = pytest.mark.gpu


def _strided(t: torch.Tensor, extra: int):
    """t (2-D, on the CPU) copied into the first columns of a wider CUDA
    buffer whose other columns hold NaN.  Returns (view, buffer)."""
    M, N = t.shape
    buf = torch.full((M, N + extra), float("nan"), dtype=t.dtype, device="cuda")
    buf[:, :N] = t.cuda()
    return buf[:, :N], buf


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("extra", [64, 3])  # 64: 16-byte rows (staged kernels); 3: plain kernels
def test_strided_rows(op, extra):
    base = wl.WORKLOADS["ln_bf16_65536x1024" if op == "ln" else "rms_bf16_16384x4096"]
    w = base.with_shape(700, 1024)
    inp = wl.make_inputs(w)
    (x, xb), (dy, dyb) = _strided(inp["x"], extra), _strided(inp["dy"], extra)
    assert x.stride(0) == 1024 + extra
    y, yb = _strided(torch.zeros_like(inp["x"]), extra + 8)
    dx, dxb = _strided(torch.zeros_like(inp["x"]), extra + 16)
    g = inp["gamma"].cuda()
    if op == "ln":
        b = inp["beta"].cuda()
        _, mean, rstd = gbn.ln_fwd(x, g, b, w.eps, y=y)
        _, dg, db = gbn.ln_bwd(dy, x, g, mean, rstd, dx=dx)
        got = dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)
    else:
        _, rstd = gbn.rms_fwd(x, g, w.eps, y=y)
        _, dg = gbn.rms_bwd(dy, x, g, rstd, dx=dx)
        got = dict(y=y, rstd=rstd, dx=dx, dgamma=dg)
    got = {k: v.cpu().contiguous() for k, v in got.items()}
    reps = gpu_parity.compare(w, inp, got)
    assert all(r.ok() for r in reps), "\n".join(map(str, reps))
    # nothing was written into the rows' padding, nor into the inputs
    N = w.N
    for name, buf in (("x", xb), ("dy", dyb), ("y", yb), ("dx", dxb)):
        assert torch.isnan(buf[:, N:]).all(), f"{name}: the row padding was written"
    assert torch.equal(xb[:, :N].cpu(), inp["x"]) and torch.equal(dyb[:, :N].cpu(), inp["dy"])
    assert gbn.device_error() == 0


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [2048, 4096])  # the slot and the warp-specialised rows kernel
def test_accumulate_and_grad_dtype(op, grad_dtype, N):
    base = wl.WORKLOADS["ln_bf16_65536x1024" if op == "ln" else "rms_bf16_16384x4096"]
    w = base.with_shape(900, N)
    inp = wl.make_inputs(w)
    d = {k: v.cuda() for k, v in inp.items()}
    gdt = wl.TORCH_DTYPES[grad_dtype]
    if op == "ln":
        _, mean, rstd = gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps)
        _, dg_o, db_o = oracle.ln_bwd(inp["dy"], inp["x"], inp["gamma"], mean.cpu(), rstd.cpu())
    else:
        _, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
        _, dg_o = oracle.rms_bwd(inp["dy"], inp["x"], inp["gamma"], rstd.cpu())
    prev = wl.to_storage(50.0 * wl.normal(9, 77, w.N), grad_dtype).cuda()
    for acc in (False, True):
        dg = prev.clone()
        db = prev.clone()
        if op == "ln":
            gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean, rstd, dgamma=dg, dbeta=db, accumulate=acc,
                       grad_dtype=gdt)
            pairs = [("dgamma", dg, dg_o), ("dbeta", db, db_o)]
        else:
            gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd, dgamma=dg, accumulate=acc, grad_dtype=gdt)
            pairs = [("dgamma", dg, dg_o)]
        old = wl.exact_double(prev.cpu())
        for name, got, ref in pairs:
            want = ref + old if acc else ref
            g64 = wl.exact_double(got.cpu())
            if grad_dtype == "f32":
                r = tol.check_param_grad(f"{name} acc={acc}", g64, want)
            else:
                # the sum is rounded once to the parameter dtype: 2 ulp of it,
                # or the fp32 parameter-gradient bar, whichever is looser
                R = tol.round_to(want, grad_dtype)
                err = np.abs(g64 - R)
                ok = err <= np.maximum(2 * tol.ulp(R, grad_dtype), 1e-3 * (1 + np.abs(want)))
                assert ok.all(), f"{name} acc={acc}: worst {err.max():.3g}"
                continue
            assert r.ok(), str(r)
    assert gbn.device_error() == 0


def test_accumulate_with_no_rows_keeps_the_buffers():
    x = torch.empty(0, 256, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(256, device="cuda", dtype=torch.bfloat16)
    rstd = torch.empty(0, device="cuda")
    dg = torch.full((256,), 3.0, device="cuda")
    gbn.rms_bwd(x, x, g, rstd, dgamma=dg, accumulate=True)
    torch.cuda.synchronize()
    assert torch.all(dg == 3.0)


def test_option_errors():
    L = gbn.lib()
    x = torch.zeros(8, 64, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(64, device="cuda", dtype=torch.bfloat16)
    y = torch.empty_like(x)
    r = torch.empty(8, device="cuda")
    bad_ld = gbn.GbnOptions(32, 0, 0, 0, 0, 0)      # stride below N
    bad_acc = gbn.GbnOptions(0, 0, 0, 2, 0, 0)      # accumulate not 0/1
    bad_dt = gbn.GbnOptions(0, 0, 0, 0, 1, 0)       # fp16 grads for bf16 parameters
    s = torch.cuda.current_stream().cuda_stream
    assert L.rms_fwd_ex(x.data_ptr(), g.data_ptr(), y.data_ptr(), r.data_ptr(), 1e-6, 8, 64, 2,
                        ctypes.byref(bad_ld), s) == 1
    ws = torch.empty(gbn.bwd_workspace_bytes(8, 64, torch.bfloat16, False), dtype=torch.uint8, device="cuda")
    dg = torch.empty(64, device="cuda")
    bad_mode = gbn.GbnOptions(0, 0, 0, 0, 0, 7)     # unknown reduce mode
    bad_mode_dt = gbn.GbnOptions(0, 0, 0, 0, 2, 1)  # atomic reduce into bf16 grads
    for opt, code in ((bad_acc, 1), (bad_dt, 2), (bad_mode, 1), (bad_mode_dt, 2)):
        assert L.rms_bwd_ex(x.data_ptr(), x.data_ptr(), g.data_ptr(), r.data_ptr(), y.data_ptr(), dg.data_ptr(),
                            0.0, 8, 64, 2, ws.data_ptr(), ws.numel(), ctypes.byref(opt), s) == code
    with pytest.raises(ValueError):
        gbn.rms_bwd(x, x, g, r, grad_dtype=torch.float16)
    torch.cuda.synchronize()

"""The warp-specialised backward (producer, sum and output warps) at the edges
of its shapes: every dtype and row width it serves, few rows (fewer than its
stages, than its sum warps, than the CTAs), with saved statistics and
without (the save-nothing variant), and the slot kernel it replaces on the
same shapes (needs a GPU)."""
import dataclasses

import pytest
import torch

import numpy as np

import gpu_parity
import oracle
import rmsnorm_backward_gb300 as gbn
import tolerance as tol
import workloads as wl

pytestmark = pytest.mark.gpu

BASE = {"ln": wl.WORKLOADS["ln_bf16_65536x1024"], "rms": wl.WORKLOADS["rms_bf16_16384x4096"]}
# (dtype, N) the kernel serves: 16 output warps of 1 or 2 vectors a lane
SHAPES = [("bf16", 4096), ("f16", 8192), ("f32", 2048), ("f32", 4096)]


def _w(op, dtype, M, N):
    return dataclasses.replace(BASE[op], dtype=dtype, M=M, N=N, name=f"{op}_{dtype}_{M}x{N}")


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("dtype,N", SHAPES)
@pytest.mark.parametrize("M", [1, 3, 6, 151, 153, 700])
def test_parity(op, dtype, N, M):
    w = _w(op, dtype, M, N)
    G, kind = gbn.bwd_plan(M, N, wl.TORCH_DTYPES[dtype], op == "ln")
    assert kind == 2, f"{w.name} does not take the warp-specialised kernel"
    gpu_parity.assert_parity(w)


@pytest.mark.parametrize("op", ["ln", "rms"])
def test_deterministic_and_slot_kernel_agrees(op):
    w = _w(op, "bf16", 999, 4096)
    inp = wl.make_inputs(w)
    runs = [gpu_parity.run_gpu(w, inp) for _ in range(3)]
    for r in runs[1:]:
        for k in ("dx", "dgamma") + (("dbeta",) if op == "ln" else ()):
            assert torch.equal(r[k], runs[0][k]), k
    # the slot kernel on the same shape passes the same parity checks
    gpu_parity.assert_parity(w, inp, kernel="slot")


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("dtype,N", SHAPES)
@pytest.mark.parametrize("M", [1, 5, 153, 700])
def test_save_nothing(op, dtype, N, M):
    """No saved statistics: the sum warps form each row's mean (LayerNorm,
    exchanged among them) and the sums that give rstd."""
    w = _w(op, dtype, M, N)
    inp = wl.make_inputs(w)
    x, dy, g = (wl.exact_double(inp[k]) for k in ("x", "dy", "gamma"))
    d = {k: v.cuda() for k, v in inp.items()}
    if op == "ln":
        _, mean_o, rstd_o = oracle.ln_fwd(x, g, wl.exact_double(inp["beta"]), w.eps)
        dx_o, dg_o, db_o = oracle.ln_bwd(dy, x, g, mean_o, rstd_o)
        dx, dg, db = gbn.ln_bwd(d["dy"], d["x"], d["gamma"], None, None, eps=w.eps)
        grads = [("dgamma", dg, dg_o), ("dbeta", db, db_o)]
    else:
        mean_o = np.zeros(M)
        _, rstd_o = oracle.rms_fwd(x, g, w.eps)
        dx_o, dg_o = oracle.rms_bwd(dy, x, g, rstd_o)
        dx, dg = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], None, eps=w.eps)
        grads = [("dgamma", dg, dg_o)]
    torch.cuda.synchronize()
    scale = tol.dx_scale(op, dy, x, g, mean_o, rstd_o)
    reps = [tol.check_elementwise("dx", wl.exact_double(dx.cpu()), dx_o, dtype, scale)]
    reps += [tol.check_param_grad(n, got.cpu().double().numpy(), ref) for n, got, ref in grads]
    assert all(r.ok() for r in reps), "\n".join(map(str, reps))
    assert gbn.device_error() == 0


def test_shapes_it_does_not_take():
    # rows that leave fewer than 16 output warps, or need 4 vectors a lane
    for N, dtype in ((1024, torch.bfloat16), (2048, torch.bfloat16), (16384, torch.bfloat16), (512, torch.float32)):
        assert gbn.bwd_plan(4096, N, dtype, False)[1] == 1

"""Runs the CUDA path and the oracle on the same seeded inputs and compares.

Used by the ``-m gpu`` tests and by ``__graft_entry__.smoke()``.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np
import torch

import guards
import oracle
import rmsnorm_backward_gb300 as gbn
import tolerance as tol
import workloads as wl


def run_gpu(w: wl.Workload, inputs: Dict[str, torch.Tensor], device="cuda", kernel: str = "auto",
            ws_misalign: int = 0):
    """Forward then backward on the GPU. Returns CPU tensors.

    Every input, output and the workspace sit between sentinel bands
    (tests/guards.py); after the calls the bands and the inputs are checked
    unchanged.  kernel: "auto", or "slot" / "plain" to force that kernel."""
    g = guards.Guarded(device)
    d = {k: g.copy_in(v, k) for k, v in inputs.items()}
    M, N = w.M, w.N
    tdt = wl.TORCH_DTYPES[w.dtype]
    ln = w.op == "ln"
    y = g.empty((M, N), tdt, "y")
    rstd = g.empty((M,), torch.float32, "rstd")
    mean = g.empty((M,), torch.float32, "mean") if ln else None
    dx = g.empty((M, N), tdt, "dx")
    dg = g.empty((N,), torch.float32, "dgamma")
    db = g.empty((N,), torch.float32, "dbeta") if ln else None
    ws = g.workspace(gbn.bwd_workspace_bytes(M, N, tdt, ln), misalign=ws_misalign)
    out = {}
    if ln:
        gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps, y=y, mean=mean, rstd=rstd, kernel=kernel)
        gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean, rstd, dx=dx, dgamma=dg, dbeta=db, workspace=ws,
                   kernel=kernel)
        out.update(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)
    else:
        gbn.rms_fwd(d["x"], d["gamma"], w.eps, y=y, rstd=rstd, kernel=kernel)
        gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd, dx=dx, dgamma=dg, workspace=ws, kernel=kernel)
        out.update(y=y, rstd=rstd, dx=dx, dgamma=dg)
    torch.cuda.synchronize()
    g.check()
    return {k: v.cpu() for k, v in out.items()}


def compare(w: wl.Workload, inputs: Dict[str, torch.Tensor], got: Dict[str, torch.Tensor]) -> List[tol.Report]:
    """All parity reports for one run.

    Forward and statistics: against the oracle's forward (its own float64
    statistics).  Backward: against the oracle's backward given the GPU's
    fp32 statistics widened to float64 (the backward's inputs), and dx also
    end to end against the oracle's backward from its own statistics.
    """
    x = wl.exact_double(inputs["x"])
    dy = wl.exact_double(inputs["dy"])
    g = wl.exact_double(inputs["gamma"])
    reps = []
    M = x.shape[0]
    if w.op == "ln":
        b = wl.exact_double(inputs["beta"])
        y_o, mean_o, rstd_o = oracle.ln_fwd(x, g, b, w.eps)
    else:
        b = None
        y_o, rstd_o = oracle.rms_fwd(x, g, w.eps)
        mean_o = np.zeros(M)
    ys = tol.y_scale(w.op, x, g, b, mean_o, rstd_o)
    reps.append(tol.check_elementwise("y", wl.exact_double(got["y"]), y_o, w.dtype, ys))
    reps.append(tol.check_stat("rstd", wl.exact_double(got["rstd"]), rstd_o))
    if w.op == "ln":
        reps.append(tol.check_stat("mean", wl.exact_double(got["mean"]), mean_o, np.mean(np.abs(x), axis=1)))
    del y_o
    # backward, from the GPU's saved statistics (the backward's own inputs)
    rstd_g = wl.exact_double(got["rstd"])
    mean_g = wl.exact_double(got["mean"]) if w.op == "ln" else np.zeros(M)
    if w.op == "ln":
        dx_o, dg_o, db_o = oracle.ln_bwd(dy, x, g, mean_g, rstd_g)
    else:
        dx_o, dg_o = oracle.rms_bwd(dy, x, g, rstd_g)
    dxs = tol.dx_scale(w.op, dy, x, g, mean_g, rstd_g)
    dx_g = wl.exact_double(got["dx"])
    reps.append(tol.check_elementwise("dx", dx_g, dx_o, w.dtype, dxs))
    reps.append(tol.check_param_grad("dgamma", wl.exact_double(got["dgamma"]), dg_o))
    if w.op == "ln":
        reps.append(tol.check_param_grad("dbeta", wl.exact_double(got["dbeta"]), db_o))
    del dx_o
    # dx end to end: oracle statistics instead of the GPU's
    if w.op == "ln":
        dx_e, _, _ = oracle.ln_bwd(dy, x, g, mean_o, rstd_o)
    else:
        dx_e, _ = oracle.rms_bwd(dy, x, g, rstd_o)
    reps.append(tol.check_elementwise("dx (end to end)", dx_g, dx_e, w.dtype,
                                      tol.dx_scale(w.op, dy, x, g, mean_o, rstd_o)))
    return reps


def assert_parity(w: wl.Workload, inputs: Optional[Dict[str, torch.Tensor]] = None, device="cuda",
                  kernel: str = "auto"):
    inputs = inputs if inputs is not None else wl.make_inputs(w)
    got = run_gpu(w, inputs, device, kernel)
    reps = compare(w, inputs, got)
    bad = [r for r in reps if not r.ok()]
    msg = f"{w.name} ({w.op} {w.dtype} {w.M}x{w.N}):\n  " + "\n  ".join(str(r) for r in reps)
    assert not bad, msg
    assert gbn.device_error(clear=True) == 0, "a kernel recorded a bounded-wait error"
    return reps

"""The reduction ablations (reduce_mode): fp32 atomics per CTA and the
column walk, against the float64 oracle (needs a GPU)."""
import dataclasses

import pytest
import torch

import oracle
import rmsnorm_backward_gb300 as gbn
import tolerance as tol
import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [("rms_bf16_16384x4096", "bf16", 1000, 4096), ("ln_bf16_65536x1024", "bf16", 3000, 1024),
         ("ln_f32_64x256", "f32", 64, 256), ("ln_bf16_65536x1024", "bf16", 500, 1000)]


def _run(w, d, reduce, accumulate=False, prev=None):
    N = w.N
    dg = prev.clone() if prev is not None else None
    if w.op == "ln":
        _, mean, rstd = gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps)
        db = prev.clone() if prev is not None else None
        dx, dg, db = gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean, rstd, dgamma=dg, dbeta=db, reduce=reduce,
                                accumulate=accumulate)
        return dx, [dg, db], (mean, rstd)
    _, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
    dx, dg = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd, dgamma=dg, reduce=reduce, accumulate=accumulate)
    return dx, [dg], (None, rstd)


@pytest.mark.parametrize("family,dtype,M,N", CASES)
@pytest.mark.parametrize("reduce", ["atomic", "colwalk"])
def test_reduce_mode_matches_the_oracle(family, dtype, M, N, reduce):
    w = dataclasses.replace(wl.WORKLOADS[family], dtype=dtype, M=M, N=N, name=f"{family}-{M}x{N}")
    inp = wl.make_inputs(w)
    d = {k: v.cuda() for k, v in inp.items()}
    dx, grads, (mean, rstd) = _run(w, d, reduce)
    dx_p, grads_p, _ = _run(w, d, "partials")
    torch.cuda.synchronize()
    if w.op == "ln":
        _, dg_o, db_o = oracle.ln_bwd(inp["dy"], inp["x"], inp["gamma"], mean.cpu(), rstd.cpu())
        refs = [dg_o, db_o]
    else:
        _, dg_o = oracle.rms_bwd(inp["dy"], inp["x"], inp["gamma"], rstd.cpu())
        refs = [dg_o]
    for got, ref in zip(grads, refs):
        r = tol.check_param_grad(f"{reduce}", got.cpu().double().numpy(), ref)
        assert r.ok(), str(r)
    assert torch.equal(dx, dx_p)  # the mode changes only the cross-row sums
    if reduce == "colwalk":  # deterministic: the same bits on a second run
        _, grads2, _ = _run(w, d, reduce)
        for a, b in zip(grads, grads2):
            assert torch.equal(a, b)
    # accumulate: previous contents + the sums
    prev = torch.linspace(-3, 3, N, device="cuda")
    _, grads_acc, _ = _run(w, d, reduce, accumulate=True, prev=prev)
    for got, ref in zip(grads_acc, refs):
        r = tol.check_param_grad(f"{reduce} accumulate", got.cpu().double().numpy(), ref + prev.cpu().double().numpy())
        assert r.ok(), str(r)
    assert gbn.device_error() == 0


def test_colwalk_needs_saved_statistics():
    x = torch.zeros(4, 64, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(gbn.GbnError):
        gbn.rms_bwd(x, x, g, None, eps=1e-6, reduce="colwalk")

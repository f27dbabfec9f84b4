"""Backward from host buffers (ln_bwd_host / rms_bwd_host): copies in, the
backward kernels and copies out pipelined over row chunks (needs a GPU)."""
import numpy as np
import pytest
import torch

import guards
import oracle
import rmsnorm_backward_gb300 as gbn
import tolerance as tol
import workloads as wl

pytestmark = pytest.mark.gpu

BASE = {"ln": wl.WORKLOADS["ln_bf16_65536x1024"], "rms": wl.WORKLOADS["rms_bf16_16384x4096"]}


def _w(op, dtype, M, N):
    import dataclasses
    return dataclasses.replace(BASE[op], dtype=dtype, M=M, N=N, name=f"{op}_{dtype}_{M}x{N}")


def _stats(w, inp):
    """The forward's statistics, from the GPU forward."""
    x, g = inp["x"].cuda(), inp["gamma"].cuda()
    if w.op == "ln":
        _, mean, rstd = gbn.ln_fwd(x, g, inp["beta"].cuda(), w.eps)
        return mean.cpu(), rstd.cpu()
    _, rstd = gbn.rms_fwd(x, g, w.eps)
    return None, rstd.cpu()


def _host(w, inp, mean, rstd, pinned=True, chunk_rows=0):
    """The host-buffer call on guarded host buffers (inputs, outputs) and a
    guarded device workspace; the bands and the inputs are checked after."""
    gh, gd = guards.Guarded("cpu"), guards.Guarded("cuda")
    dy, x, g = (gh.copy_in(inp[k], k, pin=pinned) for k in ("dy", "x", "gamma"))
    rs = gh.copy_in(rstd, "rstd", pin=pinned)
    M, N = w.M, w.N
    dx = gh.empty((M, N), x.dtype, "dx", pin=pinned)
    dg = gh.empty((N,), torch.float32, "dgamma", pin=pinned)
    ws = gd.workspace(gbn.bwd_host_workspace_bytes(M, N, x.dtype, w.op == "ln", chunk_rows=chunk_rows))
    if w.op == "ln":
        db = gh.empty((N,), torch.float32, "dbeta", pin=pinned)
        out = gbn.ln_bwd_host(dy, x, g, gh.copy_in(mean, "mean", pin=pinned), rs, dx=dx, dgamma=dg, dbeta=db,
                              workspace=ws, chunk_rows=chunk_rows)
    else:
        out = gbn.rms_bwd_host(dy, x, g, rs, dx=dx, dgamma=dg, workspace=ws, chunk_rows=chunk_rows)
    torch.cuda.synchronize()
    gh.check()
    gd.check()
    return [t.clone() for t in out]


def _device(w, inp, mean, rstd):
    d = {k: v.cuda() for k, v in inp.items()}
    if w.op == "ln":
        out = gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean.cuda(), rstd.cuda())
    else:
        out = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd.cuda())
    torch.cuda.synchronize()
    return [t.cpu() for t in out]


def _check_grads(w, inp, mean, rstd, got):
    x, dy, g = (wl.exact_double(inp[k]) for k in ("x", "dy", "gamma"))
    rs = wl.exact_double(rstd)
    if w.op == "ln":
        _, dg, db = oracle.ln_bwd(dy, x, g, wl.exact_double(mean), rs)
        refs = (dg, db)
    else:
        _, dg = oracle.rms_bwd(dy, x, g, rs)
        refs = (dg,)
    for name, r, t in zip(("dgamma", "dbeta"), refs, got[1:]):
        rep = tol.check_param_grad(name, wl.exact_double(t), r)
        assert rep.ok(), str(rep)


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M,N,chunk", [(1000, 512, 128), (300, 1000, 0), (37, 4096, 5), (513, 33, 64)])
def test_host_matches_device_and_oracle(op, dtype, M, N, chunk):
    w = _w(op, dtype, M, N)
    inp = wl.make_inputs(w)
    mean, rstd = _stats(w, inp)
    got = _host(w, inp, mean, rstd, chunk_rows=chunk)
    ref = _device(w, inp, mean, rstd)
    # every row goes through the same kernel arithmetic: dx is bit-identical
    assert torch.equal(got[0].view(torch.int16 if dtype != "f32" else torch.int32),
                       ref[0].view(torch.int16 if dtype != "f32" else torch.int32))
    _check_grads(w, inp, mean, rstd, got)
    # and the grouping of the partial sums is fixed: run to run identical
    again = _host(w, inp, mean, rstd, chunk_rows=chunk)
    for a, b in zip(got[1:], again[1:]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert gbn.device_error(clear=True) == 0


@pytest.mark.parametrize("op", ["ln", "rms"])
def test_host_headline_size(op):
    w = _w(op, "bf16", 16384, 4096) if op == "rms" else BASE["ln"]
    inp = wl.make_inputs(w)
    mean, rstd = _stats(w, inp)
    got = _host(w, inp, mean, rstd)
    ref = _device(w, inp, mean, rstd)
    assert torch.equal(got[0].view(torch.int16), ref[0].view(torch.int16))
    _check_grads(w, inp, mean, rstd, got)


def test_pageable_in_place_side_stream_and_empty():
    w = _w("rms", "bf16", 700, 2048)
    inp = wl.make_inputs(w)
    _, rstd = _stats(w, inp)
    ref = _device(w, inp, None, rstd)
    # pageable host memory, dx written over dy, on a side stream
    dy, x, g, rs = tuple(inp[k].clone() for k in ("dy", "x", "gamma")) + (rstd.clone(),)
    s = torch.cuda.Stream()
    dx, dg = gbn.rms_bwd_host(dy, x, g, rs, dx=dy, chunk_rows=100, stream=s)
    s.synchronize()
    assert dx.data_ptr() == dy.data_ptr()
    assert torch.equal(dx.view(torch.int16), ref[0].view(torch.int16))
    # M = 0: zeros, nothing enqueued
    e = torch.empty(0, 2048, dtype=torch.bfloat16)
    dge = torch.full((2048,), 7.0)
    gbn.rms_bwd_host(e, e, inp["gamma"], torch.empty(0), dgamma=dge)
    assert torch.count_nonzero(dge) == 0


def test_host_argument_errors():
    t = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gbn.rms_bwd_host(t.cuda(), t, t[0], torch.zeros(4))
    with pytest.raises(ValueError):
        gbn.rms_bwd_host(t, t, t[0], torch.zeros(5))
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        gbn.rms_bwd_host(t, t, t[0], torch.zeros(4), workspace=ws)

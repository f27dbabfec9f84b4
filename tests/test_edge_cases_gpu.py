"""Edge cases of the CUDA path against the oracle (needs a GPU)."""
import dataclasses

import numpy as np
import pytest
import torch

import gpu_parity
import oracle
import rmsnorm_backward_gb300 as gbn
import workloads as wl

pytestmark = pytest.mark.gpu

BASE = {"ln": wl.WORKLOADS["ln_f32_64x256"], "rms": wl.WORKLOADS["rms_bf16_16384x4096"]}


def _w(op, dtype, M, N, eps=None):
    b = BASE[op]
    return dataclasses.replace(b, dtype=dtype, M=M, N=N, eps=eps if eps is not None else b.eps,
                               name=f"{op}_{dtype}_{M}x{N}")


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M,N", [(1, 1), (7, 3), (1, 8), (300, 33), (153, 1000), (5, 4097),
                                 (200, 3072), (37, 24), (160, 520)])
def test_shapes(op, dtype, M, N):
    gpu_parity.assert_parity(_w(op, dtype, M, N))


@pytest.mark.parametrize("op", ["ln", "rms"])
def test_row_wider_than_the_staged_limit(op):
    gpu_parity.assert_parity(_w(op, "bf16", 9, 65536))


@pytest.mark.parametrize("op", ["ln", "rms"])
def test_more_rows_than_one_wave(op):
    # more than 2048 rows per CTA at one CTA per SM: G grows past the SM count
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M = sms * 2048 + 5
    w = _w(op, "bf16", M, 64)
    G, staged = gbn.bwd_plan(M, 64, torch.bfloat16, op == "ln")
    assert G > sms and staged
    gpu_parity.assert_parity(w)


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_misaligned_buffers_take_the_plain_kernel(op, dtype):
    w = _w(op, dtype, 100, 512)
    inp = wl.make_inputs(w)
    dev = {}
    for k, v in inp.items():
        # place each tensor one element past a 16-byte boundary
        buf = torch.empty(v.numel() + 8, dtype=v.dtype, device="cuda")
        t = buf[1:1 + v.numel()].view(v.shape)
        t.copy_(v)
        dev[k] = t
    assert dev["x"].data_ptr() % 16 != 0
    got = {}
    if op == "ln":
        y, mean, rstd = gbn.ln_fwd(dev["x"], dev["gamma"], dev["beta"], w.eps)
        dx, dg, db = gbn.ln_bwd(dev["dy"], dev["x"], dev["gamma"], mean, rstd)
        got.update(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)
    else:
        y, rstd = gbn.rms_fwd(dev["x"], dev["gamma"], w.eps)
        dx, dg = gbn.rms_bwd(dev["dy"], dev["x"], dev["gamma"], rstd)
        got.update(y=y, rstd=rstd, dx=dx, dgamma=dg)
    got = {k: v.cpu() for k, v in got.items()}
    reps = gpu_parity.compare(w, inp, got)
    assert all(r.ok() for r in reps), "\n".join(map(str, reps))


@pytest.mark.parametrize("op", ["ln", "rms"])
def test_constant_rows(op):
    w = _w(op, "bf16", 40, 1024, eps=1e-3)
    inp = wl.make_inputs(w)
    inp["x"][::3] = 1.5  # every third row constant: var = 0, xhat = 0 (LN)
    gpu_parity.assert_parity(w, inp)


def test_empty_batch():
    x = torch.empty(0, 256, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(256, device="cuda", dtype=torch.bfloat16)
    b = torch.zeros(256, device="cuda", dtype=torch.bfloat16)
    y, mean, rstd = gbn.ln_fwd(x, g, b, 1e-5)
    dg = torch.full((256,), 7.0, device="cuda")
    db = torch.full((256,), 7.0, device="cuda")
    gbn.ln_bwd(x, x, g, mean, rstd, dgamma=dg, dbeta=db)
    dgr = torch.full((256,), 7.0, device="cuda")
    gbn.rms_bwd(x, x, g, rstd, dgamma=dgr)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.all(dg == 0) and torch.all(db == 0) and torch.all(dgr == 0)


@pytest.mark.parametrize("name", ["rms_bf16_16384x4096", "ln_bf16_65536x1024", "ln_f16_1151x8192"])
def test_dgamma_dbeta_bit_identical_across_runs(name):
    w = wl.WORKLOADS[name]
    w = w.with_shape(min(w.M, 4096), w.N)
    d = {k: v.cuda() for k, v in wl.make_inputs(w).items()}
    outs = []
    for _ in range(5):
        if w.op == "ln":
            y, mean, rstd = gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps)
            dx, dg, db = gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean, rstd)
            outs.append((y, dx, dg, db))
        else:
            y, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
            dx, dg = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd)
            outs.append((y, dx, dg))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a.view(torch.uint8) if a.dtype != torch.float32 else a.view(torch.int32),
                               b.view(torch.uint8) if b.dtype != torch.float32 else b.view(torch.int32))


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("M", [1, 500, 5000])
def test_exact_sums_are_bit_exact(op, M):
    """dy in small multiples of 2^-8 and xhat = +-1 make every fp32 partial sum
    exact in any order, so dgamma and dbeta must equal the oracle's exactly."""
    N = 2048
    k = np.round(wl.normal(1, 40, M * N) * 8).clip(-60, 60).reshape(M, N)
    dy = torch.from_numpy(k * 2.0 ** -8).to(torch.bfloat16)
    signs = np.where(wl.uniform(1, 41, M * N).reshape(M, N) < 0.5, -1.0, 1.0)
    signs[:, 1::2] = -signs[:, 0::2]  # zero-mean rows of +-a
    a = 2.0 ** np.round(wl.uniform(1, 42, M) * 6 - 3)
    x = torch.from_numpy(signs * a[:, None]).to(torch.bfloat16)
    g = torch.from_numpy(1.0 + 0.0 * np.arange(N)).to(torch.bfloat16)
    xd, dyd, gd = x.cuda(), dy.cuda(), g.cuda()
    if op == "ln":
        b = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
        y, mean, rstd = gbn.ln_fwd(xd, gd, b, 0.0)
        dx, dgam, dbet = gbn.ln_bwd(dyd, xd, gd, mean, rstd)
        _, dg_o, db_o = oracle.ln_bwd(dy, x, g, mean.cpu(), rstd.cpu())
        assert np.array_equal(dbet.cpu().double().numpy(), db_o)
    else:
        y, rstd = gbn.rms_fwd(xd, gd, 0.0)
        dx, dgam = gbn.rms_bwd(dyd, xd, gd, rstd)
        _, dg_o = oracle.rms_bwd(dy, x, g, rstd.cpu())
    assert np.array_equal(rstd.cpu().double().numpy(), 1.0 / a)
    assert np.array_equal(dgam.cpu().double().numpy(), dg_o)


def _view(t: torch.Tensor, misalign: bool) -> torch.Tensor:
    """t on the GPU, one element past a 16-byte boundary when misalign."""
    if not misalign:
        return t.cuda()
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device="cuda")
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("N", [2048, 4096, 8192])
@pytest.mark.parametrize("misalign", [False, True])
def test_two_phases_equal_the_fused_call(op, N, misalign):
    """The phase calls (rows, then reduce) give the fused call's bits.  N =
    4096 and 8192 take the warp-specialised rows kernel, 2048 the slot
    kernel.  With x and dy one element off a 16-byte boundary the rows go
    through the plain kernel; the column reduce's order depends on the
    shape only, so the phase call, which does not know the rows kernel,
    still matches."""
    w = _w(op, "bf16", 1000, N)
    inp = wl.make_inputs(w)
    d = {k: v.cuda() for k, v in inp.items()}
    x, dy = _view(inp["x"], misalign), _view(inp["dy"], misalign)
    ws = torch.empty(gbn.bwd_workspace_bytes(w.M, w.N, torch.bfloat16, op == "ln"), dtype=torch.uint8,
                     device="cuda")
    if op == "ln":
        y, mean, rstd = gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps)
        dx, dg, db = gbn.ln_bwd(dy, x, d["gamma"], mean, rstd, workspace=ws)
        dx2 = gbn.ln_bwd_rows(dy, x, d["gamma"], mean, rstd, dx=torch.empty_like(x), workspace=ws)
        dg2, db2 = torch.empty_like(dg), torch.empty_like(db)
        gbn.bwd_reduce(ws, w.M, w.N, torch.bfloat16, True, dgamma=dg2, dbeta=db2)
        assert torch.equal(db, db2)
    else:
        y, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
        dx, dg = gbn.rms_bwd(dy, x, d["gamma"], rstd, workspace=ws)
        dx2 = gbn.rms_bwd_rows(dy, x, d["gamma"], rstd, dx=torch.empty_like(x), workspace=ws)
        dg2 = torch.empty_like(dg)
        gbn.bwd_reduce(ws, w.M, w.N, torch.bfloat16, False, dgamma=dg2)
    assert torch.equal(dx.view(torch.int16), dx2.view(torch.int16)) and torch.equal(dg, dg2)
    assert gbn.device_error() == 0


@pytest.mark.parametrize("name", ["rms_bf16_16384x4096", "ln_bf16_65536x1024", "rms_bf16_8192x16384"])
def test_full_size_backward_is_bit_identical_over_ten_runs(name):
    """The benchmarked sizes: ten backward calls on the same inputs give
    the same dx, dgamma and dbeta bits (no atomics, one summation order)."""
    w = wl.WORKLOADS[name]
    d = {k: v.cuda() for k, v in wl.make_inputs(w).items()}
    if w.op == "ln":
        _, mean, rstd = gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps)
        run = lambda: gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean, rstd)
    else:
        _, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
        run = lambda: gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd)
    first = [t.clone() for t in run()]
    for _ in range(9):
        for a, b in zip(first, run()):
            assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a.view(torch.int32),
                               b.view(torch.int16) if b.dtype != torch.float32 else b.view(torch.int32))
    assert gbn.device_error() == 0


def test_non_default_stream():
    w = _w("rms", "bf16", 777, 4096)
    inp = wl.make_inputs(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = {k: v.cuda(non_blocking=False) for k, v in inp.items()}
        y, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
        dx, dg = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd)
    s.synchronize()
    got = {"y": y.cpu(), "rstd": rstd.cpu(), "dx": dx.cpu(), "dgamma": dg.cpu()}
    reps = gpu_parity.compare(w, inp, got)
    assert all(r.ok() for r in reps), "\n".join(map(str, reps))


def test_argument_errors_are_reported():
    x = torch.randn(64, 256, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(256, device="cuda", dtype=torch.bfloat16)
    y, rstd = gbn.rms_fwd(x, g, 1e-6)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gbn.GbnError) as e:
        gbn.rms_bwd(x, x, g, rstd, workspace=small)
    assert e.value.status == 4
    with pytest.raises(gbn.GbnError) as e:
        gbn.rms_fwd(x, g, -1.0)
    assert e.value.status == 1
    with pytest.raises(ValueError):
        gbn.rms_fwd(x.cpu(), g, 1e-6)
    assert gbn.device_error() == 0


def test_reused_workspace_keeps_working():
    """Many backward calls on one workspace give the first call's bits."""
    w = wl.WORKLOADS["rms_bf16_16384x4096"].with_shape(1000, 4096)
    d = {k: v.cuda() for k, v in wl.make_inputs(w).items()}
    ws = torch.empty(gbn.bwd_workspace_bytes(w.M, w.N, torch.bfloat16, False), dtype=torch.uint8, device="cuda")
    _, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
    dx0, dg0 = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd, workspace=ws)
    for _ in range(20):
        dx, dg = gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(dg, dg0) and torch.equal(dx, dx0)
    assert gbn.device_error() == 0


@pytest.mark.parametrize("op", ["ln", "rms"])
def test_workspace_shared_by_alternating_problems(op):
    """Two different problems take turns on one workspace: every call gives
    the bits of the same problem run on a fresh workspace, never a mix with
    the other problem's partial rows."""
    base = wl.WORKLOADS["ln_bf16_65536x1024" if op == "ln" else "rms_bf16_16384x4096"]
    probs = []
    for seed in (3, 4):
        w = dataclasses.replace(base.with_shape(3000, 4096), seed=seed)
        d = {k: v.cuda() for k, v in wl.make_inputs(w).items()}
        if op == "ln":
            _, mean, rstd = gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps)
            run = (lambda d, mean, rstd: lambda ws: gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean, rstd,
                                                                workspace=ws))(d, mean, rstd)
        else:
            _, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
            run = (lambda d, rstd: lambda ws: gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd, workspace=ws))(d, rstd)
        probs.append(run)
    nbytes = gbn.bwd_workspace_bytes(3000, 4096, torch.bfloat16, op == "ln")
    fresh = [[t.clone() for t in run(torch.empty(nbytes, dtype=torch.uint8, device="cuda"))] for run in probs]
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for i in range(12):
        got = probs[i % 2](ws)
        for a, b in zip(fresh[i % 2], got):
            assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a.view(torch.int32),
                               b.view(torch.int16) if b.dtype != torch.float32 else b.view(torch.int32)), i
    assert gbn.device_error() == 0

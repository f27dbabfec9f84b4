"""Activation backward, dx = dy * f'(preact) for SiLU and GELU (erf form), on
the GPU against the float64 oracle (needs a GPU)."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_backward_gb300 as gbn
import tolerance as tol
import workloads as wl

pytestmark = pytest.mark.gpu

KINDS = ["silu", "gelu"]
FN = {"silu": gbn.silu_bwd, "gelu": gbn.gelu_bwd}
# zeros of f': SiLU' at the minimum of SiLU, GELU' at the minimum of GELU
ZEROS = {"silu": -1.2784645427610738, "gelu": -0.7517916243}


def _check(kind, dtype, dy, pre, dx, name):
    d, p = wl.exact_double(dy).reshape(-1), wl.exact_double(pre).reshape(-1)
    ref = oracle.act_bwd(kind, d, p)
    rep = tol.check_activation(name, wl.exact_double(dx).reshape(-1), ref, dtype, kind, d, p)
    assert rep.ok(), str(rep)
    return rep


def _act(kind, dtype, M, N):
    return wl.ActWorkload(f"{kind}_{dtype}_{M}x{N}", kind, dtype, M, N)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M,N", [(1, 1), (3, 7), (1, 8), (257, 1000), (96, 4097), (1024, 3 * 1024 + 5)])
def test_parity(kind, dtype, M, N):
    inp = wl.make_act_inputs(_act(kind, dtype, M, N))
    dy, pre = inp["dy"].cuda(), inp["preact"].cuda()
    dx = FN[kind](dy, pre)
    torch.cuda.synchronize()
    _check(kind, dtype, inp["dy"], inp["preact"], dx.cpu(), f"{kind} {dtype} {M}x{N}")


@pytest.mark.parametrize("kind", KINDS)
def test_full_size_sampled(kind):
    # the benchmark's 16384 x 4096 bf16 launch; the oracle recomputes a
    # strided plus a random sample of the outputs one by one
    a = wl.ACT_WORKLOADS[f"{kind}_bf16_16384x4096"]
    inp = wl.make_act_inputs(a)
    dy, pre = inp["dy"].cuda(), inp["preact"].cuda()
    dx = FN[kind](dy, pre).cpu()
    n = a.n
    rng = np.random.default_rng(7)
    idx = np.unique(np.concatenate([np.arange(0, n, 37), rng.integers(0, n, 1 << 20), np.arange(n - 4099, n)]))
    t = torch.from_numpy(idx)
    _check(kind, "bf16", inp["dy"].reshape(-1)[t], inp["preact"].reshape(-1)[t], dx.reshape(-1)[t],
           f"{a.name} sampled ({idx.size} of {n})")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_special_values(kind, dtype):
    vals = [0.0, 1e-30, -1e-30, 1e-5, -1e-5, 1.0, -1.0, ZEROS[kind], ZEROS[kind] * (1 + 2 ** -10),
            2.0, -2.0, 5.0, -5.0, 10.0, -10.0, -13.0, -13.5, 20.0, -20.0, 88.0, -88.0, -89.0, -100.0,
            -103.0, -104.0, -150.0, 1e4, -1e4, 65504.0, -65504.0, 1e30, -1e30, 3.38e38, -3.38e38]
    # and a dense sweep through both tails to where every term underflows
    p = wl.to_storage(np.concatenate([np.array(vals), np.linspace(-15.0, 15.0, 30001)]), dtype)
    p = p[torch.isfinite(p.float())]  # values beyond the dtype's range are not inputs
    for dyv in (1.0, -3.0, 1e-3):
        dy = torch.full_like(p, dyv)
        dx = FN[kind](dy.cuda(), p.cuda()).cpu()
        assert torch.isfinite(dx.float()).all()
        _check(kind, dtype, dy, p, dx, f"{kind} {dtype} special values, dy={dyv}")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("which", ["dy", "preact", "dx"])
def test_misaligned_pointer_takes_the_scalar_loop(kind, dtype, which):
    inp = wl.make_act_inputs(_act(kind, dtype, 33, 129))
    n = inp["dy"].numel()
    bufs = {}
    for k in ("dy", "preact", "dx"):
        off = 1 if k == which else 0
        b = torch.zeros(n + 16, dtype=wl.TORCH_DTYPES[dtype], device="cuda")
        bufs[k] = b[off:off + n]
    assert bufs[which].data_ptr() % 16 != 0
    bufs["dy"].copy_(inp["dy"].reshape(-1))
    bufs["preact"].copy_(inp["preact"].reshape(-1))
    FN[kind](bufs["dy"], bufs["preact"], dx=bufs["dx"])
    _check(kind, dtype, inp["dy"], inp["preact"], bufs["dx"].cpu(), f"{kind} {dtype} misaligned {which}")


@pytest.mark.parametrize("kind", KINDS)
def test_in_place_and_side_stream(kind):
    a = _act(kind, "bf16", 512, 2048 + 3)
    inp = wl.make_act_inputs(a)
    dy, pre = inp["dy"].cuda(), inp["preact"].cuda()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = FN[kind](dy, pre, dx=dy, stream=s)  # dx aliases dy
    s.synchronize()
    assert out.data_ptr() == dy.data_ptr()
    _check(kind, "bf16", inp["dy"], inp["preact"], dy.cpu(), f"{kind} in place on a side stream")


@pytest.mark.parametrize("kind", KINDS)
def test_grid_stride_tail_sizes(kind):
    # sizes around the vector width and around one full grid-stride sweep
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sweep = sms * 8 * 256 * 8  # blocks x threads x bf16 elements per 16-byte vector
    for n in (7, 8, 9, 15, 17, sweep - 1, sweep, sweep + 9, 2 * sweep + 8 * 3 + 5):
        a = _act(kind, "bf16", 1, n)
        inp = wl.make_act_inputs(a)
        dx = FN[kind](inp["dy"].cuda(), inp["preact"].cuda()).cpu()
        _check(kind, "bf16", inp["dy"], inp["preact"], dx, f"{kind} n={n}")


def test_empty_and_argument_errors():
    e = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    assert gbn.silu_bwd(e, e).numel() == 0
    a = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        gbn.gelu_bwd(a, torch.zeros(8, dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError):
        gbn.gelu_bwd(a, torch.zeros(9, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        gbn.silu_bwd(torch.zeros(4, 4, device="cuda").t(), torch.zeros(4, 4, device="cuda"))
    assert gbn.device_error(clear=True) == 0


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_host_buffers_match_the_device_call(kind, dtype):
    # small chunks, so the ramp and several chunks per buffer are exercised
    a = _act(kind, dtype, 37, 1001)
    inp = wl.make_act_inputs(a)
    ref = FN[kind](inp["dy"].cuda(), inp["preact"].cuda()).cpu()
    host = {"silu": gbn.silu_bwd_host, "gelu": gbn.gelu_bwd_host}[kind]
    dx = host(inp["dy"].pin_memory(), inp["preact"].pin_memory(), chunk=1000)
    torch.cuda.synchronize()
    iv = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(dx.view(iv), ref.view(iv))
    # in place over a pageable dy, on a side stream
    dy = inp["dy"].clone()
    s = torch.cuda.Stream()
    out = host(dy, inp["preact"].clone(), dx=dy, chunk=1000, stream=s)
    s.synchronize()
    assert out.data_ptr() == dy.data_ptr() and torch.equal(dy.view(iv), ref.view(iv))

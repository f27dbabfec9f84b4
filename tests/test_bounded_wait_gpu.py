"""The backward kernels' bounded waits, made to run out on purpose (needs a
GPU).

Every wait inside the backward kernels (a warp waiting for a bulk copy to
land, or for another warp's share of a row) gives up after a limit, records
error 1 in the device's flag and returns, after the CTA's own copies still
in flight have landed.  gbn_options.wait_limit_ns sets that limit; at one
nanosecond the first wait of a warp, whose copy was issued a moment before,
is still open and gives up.  Nothing faults and nothing hangs: the kernels
return, gbn_device_error() reads 1, and the next normal call on the same
device passes its parity checks.  ("Norm backward in Triton -- the dγ/dβ
reduction", section "3 · the historical lock + partial buffer": the
unbounded spin-wait these bounded waits replace.)
"""
import dataclasses

import pytest
import torch

import gpu_parity
import rmsnorm_backward_gb300 as gbn
import workloads as wl

pytestmark = pytest.mark.gpu

BASE = {"ln": wl.WORKLOADS["ln_bf16_65536x1024"], "rms": wl.WORKLOADS["rms_bf16_16384x4096"]}


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("N,saved", [(4096, True), (4096, False), (8192, True), (8192, False)])
def test_waits_that_run_out_report_error_1_and_the_device_stays_usable(op, N, saved):
    """The warp-specialised kernel: its consumer warps first wait for gamma's
    copy, issued just before, so at a one-nanosecond limit that wait gives
    up; the producer then gives up on the consumers and drains its copies."""
    kernel = "auto"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert gbn.bwd_plan(40 * sms, N, torch.bfloat16, op == "ln")[1] == 2
    # more rows per CTA than ring stages, so the producer waits on the
    # consumers too
    w = dataclasses.replace(BASE[op], dtype="bf16", M=40 * sms + 7, N=N, name=f"{op}_bf16_bounded_{N}")
    assert gbn.device_error(clear=True) == 0
    d = {k: v.cuda() for k, v in wl.make_inputs(w).items()}
    if op == "ln":
        _, mean, rstd = gbn.ln_fwd(d["x"], d["gamma"], d["beta"], w.eps)
        if not saved:
            mean = rstd = None
        gbn.ln_bwd(d["dy"], d["x"], d["gamma"], mean, rstd, eps=w.eps, kernel=kernel, wait_limit_ns=1)
    else:
        _, rstd = gbn.rms_fwd(d["x"], d["gamma"], w.eps)
        gbn.rms_bwd(d["dy"], d["x"], d["gamma"], rstd if saved else None, eps=w.eps, kernel=kernel,
                    wait_limit_ns=1)
    torch.cuda.synchronize()  # the kernels returned
    assert gbn.device_error(clear=True) == 1
    # the same device, the same shape family, the normal limit: parity holds
    gpu_parity.assert_parity(dataclasses.replace(w, M=3 * sms + 5), kernel=kernel)

"""CUDA path vs the float64 oracle on the seeded workloads (needs a GPU).

Each workload runs at a reduced row count that still spans every CTA several
times with a ragged last block (M = 3 * 152 + 37), and at its full size, in
the launch configuration the benchmark times (the same library calls).
"""
import pytest
import torch

import gpu_parity
import rmsnorm_backward_gb300 as gbn
import workloads as wl

NAMES = list(wl.WORKLOADS)


@pytest.mark.gpu
@pytest.mark.parametrize("name", NAMES)
def test_parity_reduced_rows(name):
    w = wl.WORKLOADS[name]
    M = min(w.M, 3 * 152 + 37)
    gpu_parity.assert_parity(w.with_shape(M, w.N))


@pytest.mark.gpu
@pytest.mark.parametrize("name", NAMES)
def test_parity_full_size(name):
    gpu_parity.assert_parity(wl.WORKLOADS[name])


@pytest.mark.gpu
@pytest.mark.parametrize("name", NAMES)
def test_aligned_workloads_take_the_staged_kernel(name):
    w = wl.WORKLOADS[name]
    G, staged = gbn.bwd_plan(w.M, w.N, wl.TORCH_DTYPES[w.dtype], w.has_beta)
    assert staged, f"{name} would take the plain-load kernel"
    assert G == min(w.M, torch.cuda.get_device_properties(0).multi_processor_count)

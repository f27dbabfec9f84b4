"""The seeded generator and the byte accounting (CPU only)."""
import json
import os

import numpy as np
import torch

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_numbers.json")


def test_worked_numbers_of_the_pages():
    g = json.load(open(GOLDEN))
    M, N, es = g["rows"], g["features"], g["elem_bytes"]
    reads = 2 * M * N * es
    writes = M * N * es
    assert round(reads / 1e9, 2) == g["dx_read_gb_x_plus_dy"]
    assert round(writes / 1e9, 2) == g["dx_write_gb"]
    total = wl.bwd_min_bytes("rms", "bf16", M, N)
    assert round(total / 1e9, 1) == g["total_gb_approx"]
    assert abs(total / (g["hbm_tb_per_s"] * 1e12) * 1e6 - g["time_us_approx"]) < 1.0
    assert round(g["workspace_groups"] * N * 4 / 1e6) == g["workspace_mb"]
    assert round(M * N * es / 1e9, 2) == g["stored_xhat_extra_read_gb"]
    assert abs(M * N * es / (g["hbm_tb_per_s"] * 1e12) * 1e6 - g["stored_xhat_extra_us_approx"]) < 1.0


def test_min_bytes_of_each_workload():
    want = {"ln_f32_64x256": 200192, "ln_f16_1151x8192": 56665080,
            "rms_bf16_16384x4096": 402743296, "ln_bf16_65536x1024": 403187712,
            "rms_bf16_8192x16384": 805437440}
    fwd = {"ln_f32_64x256": 133632, "ln_f16_1151x8192": 37757944,
           "rms_bf16_16384x4096": 268509184, "ln_bf16_65536x1024": 268963840,
           "rms_bf16_8192x16384": 536936448}
    for name, w in wl.WORKLOADS.items():
        assert wl.bwd_min_bytes(w.op, w.dtype, w.M, w.N) == want[name]
        assert wl.fwd_min_bytes(w.op, w.dtype, w.M, w.N) == fwd[name]


def test_splitmix64_known_values():
    # splitmix64 with state 0: the first outputs of the published generator
    z = wl._mix(np.array([0x9E3779B97F4A7C15, 0x3C6EF372FE94F82A], dtype=np.uint64))
    assert [hex(int(v)) for v in z] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4"]


def test_generator_is_deterministic_and_has_the_stated_moments():
    a = wl.normal(0, 1, 200000)
    b = wl.normal(0, 1, 200000)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1) < 0.01
    u = wl.uniform(0, 2, 200000)
    assert 0 < u.min() and u.max() < 1 and abs(u.mean() - 0.5) < 0.01
    # chunked generation equals one-shot generation
    big = wl.normal(3, 4, (1 << 22) + 17)
    assert np.array_equal(big[-17:], wl.normal(3, 4, (1 << 22) + 17)[-17:])


def test_workload_inputs_follow_their_recipes():
    w = wl.WORKLOADS["ln_f32_64x256"]
    d = wl.make_inputs(w)
    assert d["x"].dtype == torch.float32 and d["x"].shape == (64, 256)
    assert abs(d["gamma"].double().mean().item() - 1) < 0.05
    w5 = wl.WORKLOADS["rms_bf16_8192x16384"].with_shape(64, 16384)
    cols = wl.outlier_columns(0, 16384)
    assert len(cols) == 164 and len(set(cols.tolist())) == 164
    x = wl.make_inputs(w5)["x"].double()
    colstd = x.std(dim=0)
    mask = torch.zeros(16384, dtype=torch.bool)
    mask[torch.from_numpy(cols)] = True
    assert colstd[mask].mean() > 15 and colstd[~mask].mean() < 1.5
    w4 = wl.WORKLOADS["ln_bf16_65536x1024"].with_shape(256, 1024)
    x4 = wl.make_inputs(w4)["x"].double()
    means = x4.mean(dim=1)
    assert means.min() > -5.5 and means.max() < 5.5 and means.std() > 2
    # storage rounding is exact round-to-nearest of the float32 value
    v = np.array([1.0 + 2 ** -8 + 2 ** -20, 1.0 + 2 ** -8])
    t = wl.to_storage(v, "bf16").float().numpy()
    assert t[0] == np.float32(1.0 + 2 ** -7) and t[1] == np.float32(1.0)

"""bench.py's reference arm (the float64 oracle on host cores) prints one
JSON line with the contract's keys; it needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600, check=True).stdout
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1, out
    return json.loads(lines[0])


def test_reference_line_keys():
    d = _run("--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "ln_f32_64x256")
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "ln_f32_64x256"


def test_activation_reference_line():
    d = _run("--impl", "reference", "--activation", "gelu", "--steps", "1", "--warmup", "0")
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "gelu_bf16_16384x4096"

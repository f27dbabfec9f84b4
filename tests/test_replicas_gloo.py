"""The benchmark's multi-process path on the CPU: world size 2 over gloo.

The backward shards along rows with no data-path collective, so N GPUs run N
independent replicas; the only collectives are the barrier around the timed
region and the max over ranks of the timings.  These tests run those helpers
(and the reference arm's rank gating) in two processes on 127.0.0.1.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w, local = bench.dist_setup("gloo")
    result = {"rank": r, "world": w, "local": local}
    bench.dist_barrier(w)
    # each rank's own timing; the job's is the slowest rank's
    own = 1.5 * (r + 1)
    result["max"] = bench.dist_max(own, w, "cpu")
    # whole-job throughput as the bench forms it: units of all ranks / max time
    steps, units = 10, 1000
    result["value"] = w * steps * units / result["max"]
    # the reference arm: rank 0 alone runs and prints one line
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0",
                                              "--workload", "ln_f32_64x256"]))
    result["printed"] = buf.getvalue()
    bench.dist_barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(result, f)


def test_two_replicas_over_gloo(tmp_path):
    pytest.importorskip("torch.distributed")
    world, port = 2, _free_port()
    mp.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world and d["local"] == r
        assert d["max"] == 3.0  # the slower rank's 3.0 s, seen by both
        assert d["value"] == pytest.approx(world * 10 * 1000 / 3.0)
    line = json.loads(res[0]["printed"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert res[1]["printed"] == ""  # the other ranks do no work


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench

    assert bench.dist_setup("gloo") == (0, 1, 0)
    bench.dist_barrier(1)
    assert bench.dist_max(2.5, 1, "cpu") == 2.5

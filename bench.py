"""Benchmark of the LayerNorm / RMSNorm backward on GB300.

One step = the whole hot path over one batch of synthetic input: the forward
(y and the per-row statistics) followed by the backward (the fused per-row dx
+ partial-row kernel, then the fixed-order column reduce of dgamma / dbeta).
L2 is flushed (a 256 MiB write) before the forward and before the backward of
every step, outside the timed kernels.

Headline value: achieved HBM GB/s of the backward (minimum bytes: read x, dy,
gamma and the statistics; write dx, dgamma, dbeta) over its device time,
measured with CUDA events on the launching stream.  Printed as ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the float64 CPU oracle, timed on host cores
    python bench.py --activation silu|gelu  # the activation backward dx = dy * f'(preact)
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "LN/RMSNorm bwd achieved HBM GB/s (% of GB300 peak) and rows/s at M×N"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.HEADLINE, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--reduce", choices=["partials", "atomic", "colwalk"], default="partials",
                    help="cross-row reduction of dgamma/dbeta: the deterministic default or an ablation")
    ap.add_argument("--stats", choices=["saved", "recompute"], default="saved",
                    help="recompute: the backward gets no saved statistics and forms them from x")
    ap.add_argument("--kernel", choices=["auto", "slot", "plain"], default="auto",
                    help="the rows kernel of the public backward: the fastest that applies, or a forced one")
    ap.add_argument("--activation", choices=["silu", "gelu"], default=None,
                    help="time the activation backward on a 16384 x 4096 bf16 tensor instead of the norm")
    ap.add_argument("--steady", action="store_true",
                    help="time --steps public backward calls back to back, no L2 flush (workloads whose x and dy "
                         "exceed the L2): steady state, each call paying the previous call's dx write-back")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: every rank runs the whole workload on its GPU)
# ---------------------------------------------------------------------------
def dist_setup(backend: str):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, 0
    import torch.distributed as dist

    dist.init_process_group(backend=backend)
    return dist.get_rank(), dist.get_world_size(), int(os.environ.get("LOCAL_RANK", "0"))


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def dist_max(value: float, world: int, device) -> float:
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# measured peaks, traffic record, clocks
# ---------------------------------------------------------------------------
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources each captured kernel is built from
KERNEL_SOURCES = {
    "bwd_staged_kernel": ("gbn_device.cuh", "gbn_launch.h", "bwd_kernels.cuh"),
    "bwd_ws_kernel": ("gbn_device.cuh", "gbn_launch.h", "bwd_ws_layout.h", "bwd_ws.cuh"),
    "act_bwd_kernel": ("gbn_device.cuh", "gbn_launch.h", "act_bwd.cu"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the CUDA sources one kernel is built from (a traffic record
    taken from an ncu capture is only valid for the sources it was captured
    from)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "rmsnorm_backward_gb300", "csrc", name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of a workload's dominant kernel from an ncu
    capture, if the capture was taken of that kernel and its current sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(workload)
        if not rec or rec.get("kernel") != kernel or rec.get("source_hash") != kernel_source_hash(kernel):
            return None
    except Exception:
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu = gpu_index
        self.enabled = enabled
        self.proc = None
        self.lines = []

    def __enter__(self):
        if not self.enabled:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class Problem:
    """Device buffers and the three launches of one step for a workload."""

    def __init__(self, w: wl.Workload, device, stream, recompute: bool = False, reduce: str = "partials",
                 kernel: str = "auto"):
        import rmsnorm_backward_gb300 as gbn

        self.gbn = gbn
        self.w = w
        self.dev = device
        self.stream = stream
        inp = wl.make_inputs(w)
        self.host = inp
        self.x = inp["x"].to(device)
        self.dy = inp["dy"].to(device)
        self.gamma = inp["gamma"].to(device)
        self.beta = inp["beta"].to(device) if w.has_beta else None
        tdt = wl.TORCH_DTYPES[w.dtype]
        self.y = torch.empty_like(self.x)
        self.dx = torch.empty_like(self.x)
        self.mean = torch.empty(w.M, dtype=torch.float32, device=device) if w.has_beta else None
        self.rstd = torch.empty(w.M, dtype=torch.float32, device=device)
        self.dgamma = torch.empty(w.N, dtype=torch.float32, device=device)
        self.dbeta = torch.empty(w.N, dtype=torch.float32, device=device) if w.has_beta else None
        self.ws = torch.empty(gbn.bwd_workspace_bytes(w.M, w.N, tdt, w.has_beta, device), dtype=torch.uint8,
                              device=device)
        self.tdt = tdt

        # pre-marshalled C-ABI calls for the timed loop (no per-call Python checks)
        L = gbn.lib()
        sp = stream.cuda_stream
        code = gbn.DTYPE_CODES[tdt]
        M, N, P = w.M, w.N, (lambda t: None if t is None else t.data_ptr())
        wsb = self.ws.numel()
        self.recompute = recompute
        # the backward's statistics: the forward's, or none (formed from x)
        bmean = None if recompute else self.mean
        brstd = None if recompute else self.rstd
        beps = w.eps if recompute else 0.0
        if w.has_beta:
            self._fwd = (L.ln_fwd, (P(self.x), P(self.gamma), P(self.beta), P(self.y), P(self.mean),
                                    P(self.rstd), w.eps, M, N, code, sp))
            self._rows = (L.ln_bwd_rows, (P(self.dy), P(self.x), P(self.gamma), P(self.mean), P(self.rstd),
                                          P(self.dx), M, N, code, P(self.ws), wsb, sp))
        else:
            self._fwd = (L.rms_fwd, (P(self.x), P(self.gamma), P(self.y), P(self.rstd), w.eps, M, N, code, sp))
            self._rows = (L.rms_bwd_rows, (P(self.dy), P(self.x), P(self.gamma), P(self.rstd), P(self.dx), M, N,
                                           code, P(self.ws), wsb, sp))
        self._red = (L.gbn_bwd_reduce, (P(self.ws), wsb, M, N, code, int(w.has_beta), P(self.dgamma),
                                        P(self.dbeta), sp))
        # the public backward through the options call (contiguous rows,
        # float32 grads, overwrite, the chosen cross-row reduction)
        self.opt = gbn.GbnOptions(N, N, N, 0, 0, gbn.REDUCE_MODES[reduce], gbn.KERNELS[kernel], 0, 0)
        self.reduce = reduce
        self.kernel = kernel
        optp = ctypes.byref(self.opt)
        if w.has_beta:
            self._bwd = (L.ln_bwd_ex, (P(self.dy), P(self.x), P(self.gamma), P(bmean), P(brstd), P(self.dx),
                                       P(self.dgamma), P(self.dbeta), beps, M, N, code, P(self.ws), wsb, optp, sp))
        else:
            self._bwd = (L.rms_bwd_ex, (P(self.dy), P(self.x), P(self.gamma), P(brstd), P(self.dx),
                                        P(self.dgamma), beps, M, N, code, P(self.ws), wsb, optp, sp))

    @staticmethod
    def _call(fn_args):
        st = fn_args[0](*fn_args[1])
        if st != 0:
            raise RuntimeError(f"{fn_args[0].__name__} returned status {st}")

    def fwd(self):
        self._call(self._fwd)

    def rows_alone(self) -> bool:
        """Whether the rows kernel can be timed on its own (the phase call):
        saved statistics, the default reduce and the automatic kernel."""
        return not self.recompute and self.reduce == "partials" and self.kernel == "auto"

    def bwd_rows(self):
        # otherwise there is no separate rows phase: time the whole call
        self._call(self._rows if self.rows_alone() else self._bwd)

    def bwd_reduce(self):
        if self.rows_alone():
            self._call(self._red)

    def bwd_fused(self):
        self._call(self._bwd)

    def bwd(self):
        g = self.gbn
        if self.w.has_beta:
            g.ln_bwd(self.dy, self.x, self.gamma, self.mean, self.rstd, dx=self.dx, dgamma=self.dgamma,
                     dbeta=self.dbeta, workspace=self.ws, stream=self.stream)
        else:
            g.rms_bwd(self.dy, self.x, self.gamma, self.rstd, dx=self.dx, dgamma=self.dgamma, workspace=self.ws,
                      stream=self.stream)


class L2Flush:
    """Evicts L2 between timed kernels: writes one 256 MiB buffer, then reads
    another, so the written lines are written back before the next timed
    kernel starts and L2 holds only clean lines of neither workload tensor."""

    def __init__(self, device):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def time_steps(prob: Problem, steps: int, warmup: int, flush: L2Flush, world: int):
    """Warmup, then two timed loops of `steps` steps each.

    Loop 1 (the headline): flush, forward, flush, backward through the public
    fused call (rows kernel then column reduce, back to back).
    Loop 2 (the roofline of the dominant kernel): flush, rows kernel alone,
    then the column reduce, each bracketed by its own events.
    Returns per-step event times in ms."""
    s = prob.stream
    with torch.cuda.stream(s):
        for _ in range(warmup):
            flush()
            prob.fwd()
            flush()
            prob.bwd_fused()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        for k in range(steps):
            e = ev[k]
            flush()
            e[0].record(s)
            prob.fwd()
            e[1].record(s)
            flush()
            e[2].record(s)
            prob.bwd_fused()
            e[3].record(s)
        for k in range(steps):
            e = ev2[k]
            flush()
            e[0].record(s)
            prob.bwd_rows()
            e[1].record(s)
            prob.bwd_reduce()
            e[2].record(s)
    torch.cuda.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    fwd = np.array([e[0].elapsed_time(e[1]) for e in ev])
    bwd = np.array([e[2].elapsed_time(e[3]) for e in ev])
    rows = np.array([e[0].elapsed_time(e[1]) for e in ev2])
    red = np.array([e[1].elapsed_time(e[2]) for e in ev2])
    return fwd, bwd, rows, red, wall


def time_e2e(prob: Problem, steps: int):
    """The backward through the public host-buffer call (ln_bwd_host /
    rms_bwd_host): every step copies dy, x, gamma and the saved statistics
    from pinned host memory to the device and dx, dgamma (dbeta) back, the
    copies pipelined with the kernels over row chunks inside the call."""
    s = prob.stream
    w = prob.w
    gbn = prob.gbn
    # statistics saved by a forward, kept on the host like the other inputs
    with torch.cuda.stream(s):
        prob.fwd()
    torch.cuda.synchronize()
    h = {"dy": prob.host["dy"].pin_memory(), "x": prob.host["x"].pin_memory(),
         "gamma": prob.host["gamma"].pin_memory(), "rstd": prob.rstd.cpu().pin_memory()}
    if w.has_beta:
        h["mean"] = prob.mean.cpu().pin_memory()
    out = {"dx": torch.empty_like(prob.host["x"]).pin_memory(),
           "dgamma": torch.empty(w.N, dtype=torch.float32).pin_memory()}
    if w.has_beta:
        out["dbeta"] = torch.empty(w.N, dtype=torch.float32).pin_memory()
    ws = torch.empty(gbn.bwd_host_workspace_bytes(w.M, w.N, prob.tdt, w.has_beta, prob.dev), dtype=torch.uint8,
                     device=prob.dev)
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in out.values())

    def one():
        if w.has_beta:
            gbn.ln_bwd_host(h["dy"], h["x"], h["gamma"], h["mean"], h["rstd"], dx=out["dx"], dgamma=out["dgamma"],
                            dbeta=out["dbeta"], workspace=ws, device=prob.dev, stream=s)
        else:
            gbn.rms_bwd_host(h["dy"], h["x"], h["gamma"], h["rstd"], dx=out["dx"], dgamma=out["dgamma"],
                             workspace=ws, device=prob.dev, stream=s)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        one()
    e1.record(s)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


def cpu_baseline(w: wl.Workload, target_s: float = 10.0, threads: int = 1):
    """The float64 oracle's backward on the host, on the first rows of the
    same workload; repeated until ~target_s of CPU work.  threads > 1: the
    oracle's timed mode across host threads (row blocks, fixed-order sum of
    the per-thread partials) on a proportionally larger sample."""
    import oracle

    rows = min(w.M, max(64, (1 << 22) * threads // w.N))  # ~4M elements per call and thread
    sw = w.with_shape(rows, w.N)
    inp = wl.make_inputs(sw)
    x = wl.exact_double(inp["x"])
    dy = wl.exact_double(inp["dy"])
    g = wl.exact_double(inp["gamma"])
    if w.has_beta:
        _, mean, rstd = oracle.ln_fwd(x, g, wl.exact_double(inp["beta"]), w.eps)
    else:
        _, rstd = oracle.rms_fwd(x, g, w.eps)
    calls, t_total = 0, 0.0
    while t_total < target_s:
        t0 = time.perf_counter()
        if w.has_beta:
            oracle.ln_bwd(dy, x, g, mean, rstd, threads=threads)
        else:
            oracle.rms_bwd(dy, x, g, rstd, threads=threads)
        t_total += time.perf_counter() - t0
        calls += 1
    per_call = t_total / calls
    gbs = wl.bwd_min_bytes(w.op, w.dtype, rows, w.N) / per_call / 1e9
    how = "one thread" if threads == 1 else f"{threads} threads over row blocks"
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "rows_per_s": round(rows / per_call, 1),
            "sample": (f"float64 oracle backward (C, {how}) on the first {rows} of {w.M} rows "
                       f"of {w.name}, {calls} calls, {t_total:.1f} s; GB/s counts the {w.dtype} "
                       "workload's minimum bytes of those rows")}


def run_ours(args):
    rank, world, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = wl.WORKLOADS[args.workload]
    stream = torch.cuda.Stream(device)
    prob = Problem(w, device, stream, recompute=args.stats == "recompute", reduce=args.reduce, kernel=args.kernel)
    flush = L2Flush(device)
    import rmsnorm_backward_gb300 as gbn

    G, kind = gbn.bwd_plan(w.M, w.N, prob.tdt, w.has_beta, device)
    if args.kernel != "auto":
        kind = {"slot": 1 if kind else 0, "plain": 0}[args.kernel]
    kernel = gbn.BWD_KERNELS[kind]
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local
    with ClockSampler(gpu_index, enabled=not args.no_clocks) as clk:
        fwd, bwd, rows, red, wall = time_steps(prob, args.steps, args.warmup, flush, world)
    err = gbn.device_error(clear=True, device=device)
    if err:
        raise SystemExit(f"kernel error flag set: {err}")
    bwd_s = dist_max(float(bwd.sum()) / 1e3, world, device)
    rows_s = dist_max(float(rows.sum()) / 1e3, world, device)
    fwd_s = dist_max(float(fwd.sum()) / 1e3, world, device)
    K = args.steps
    bwd_bytes = wl.bwd_min_bytes(w.op, w.dtype, w.M, w.N)
    if args.stats == "recompute":  # no statistics are read
        bwd_bytes -= 4 * w.M * (2 if w.has_beta else 1)
    fwd_bytes = wl.fwd_min_bytes(w.op, w.dtype, w.M, w.N)
    value = world * K * bwd_bytes / bwd_s / 1e9
    peak, peak_src = measured_hbm_peak()
    # an ncu record applies to the configuration it was captured in: saved or
    # recomputed statistics with the partial-row reduce (the ablations have none)
    traffic_key = None
    if args.reduce == "partials":
        traffic_key = w.name if args.stats != "recompute" else "recompute_" + w.name
    # the fused per-row kernel: all algorithmic bytes but the dgamma/dbeta writes
    rows_bytes = bwd_bytes - 4 * w.N * (2 if w.has_beta else 1)
    rows_avg = rows_s / K
    achieved = rows_bytes / rows_avg / 1e9
    e2e_ms, h2d, d2h = time_e2e(prob, args.e2e_steps)
    e2e_ms = dist_max(e2e_ms, world, device)
    out = None
    if rank == 0:
        clocks = clk.summary()
        out = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round((fwd_s + bwd_s) / K * 1e3, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": w.dtype,
            "data": "synthetic",
            "config": {
                "workload": w.name, "op": {"ln": "layernorm", "rms": "rmsnorm"}[w.op], "M": w.M, "N": w.N,
                "eps": w.eps, "inputs": w.describe(), "seed": w.seed,
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                "l2": ("flushed before the forward and before the backward of every step: a 256 MiB write, "
                       "then a 256 MiB read of another buffer so no dirty lines carry into the timed kernel"),
                "G": G, "bwd_kernel": kernel, "stats": args.stats, "reduce": args.reduce, "kernel": args.kernel,
                "step": "forward (y, stats) then backward (dx + partial rows, then column reduce)",
                "timed": ("value = backward minimum bytes / device time of the public backward call (rows kernel "
                          "+ column reduce, CUDA events around the call); roofline = rows kernel alone, own loop"),
            },
            "rows_per_s": round(world * K * w.M / bwd_s, 1),
            "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "pct_of_measured_copy": round(100 * value / world / peak, 2),
            "bwd_us": round(bwd_s / K * 1e6, 3),
            "bwd_rows_kernel_us": round(rows_avg * 1e6, 3),
            "reduce_kernel_us": round(dist_max(float(red.sum()) / 1e3, world, device) / K * 1e6, 3)
            if world == 1 else None,
            "fwd": {"us": round(fwd_s / K * 1e6, 3), "GB/s": round(K * fwd_bytes / fwd_s / 1e9, 2),
                    "min_bytes": fwd_bytes},
            "bwd_min_bytes": bwd_bytes,
            "roofline": {
                "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(traffic_key, kernel),
                "kernel": (f"{kernel} (dx + per-CTA partial rows) alone, against the measured copy rate"
                           if prob.rows_alone() else
                           "the whole backward call (ablation, forced kernel or save-nothing variant)"),
                "algorithmic_bytes_per_launch": rows_bytes, "peak_source": peak_src,
                # the spec reading: the fused backward (rows kernel +
                # column reduce) against the nominal 8 TB/s
                "frac_nominal": round(value / world / NOMINAL_HBM_GBS, 4),
                "frac_nominal_what": "public backward call (rows kernel + column reduce) GB/s / 8000 GB/s",
            },
            "e2e": {"value": round(world * bwd_bytes / (e2e_ms / 1e3) / 1e9, 3), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 4),
                    "what": ("rms_bwd_host / ln_bwd_host: pinned host inputs and outputs, copies in, kernels "
                             "and copies out pipelined over row chunks inside the call")},
            "gpu_launches": 3 * K + 2 * K,
            "clocks": clocks,
            "wall_s_timed_region": round(wall, 3),
        }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w)
        out["cpu_baseline_threads"] = cpu_baseline(w, target_s=5.0, threads=os.cpu_count() or 1)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_reference(args):
    """The float64 CPU oracle as the reference arm (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    w = wl.WORKLOADS[args.workload]
    rows = min(w.M, max(16, (1 << 20) // w.N))  # ~1M elements per step
    sw = w.with_shape(rows, w.N)
    inp = wl.make_inputs(sw)
    x, dy, g = (wl.exact_double(inp[k]) for k in ("x", "dy", "gamma"))
    if w.has_beta:
        _, mean, rstd = oracle.ln_fwd(x, g, wl.exact_double(inp["beta"]), w.eps)
    else:
        _, rstd = oracle.rms_fwd(x, g, w.eps)

    def step():
        if w.has_beta:
            oracle.ln_bwd(dy, x, g, mean, rstd)
        else:
            oracle.rms_bwd(dy, x, g, rstd)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps * wl.bwd_min_bytes(w.op, w.dtype, rows, w.N) / dt / 1e9
    sample = (f"float64 oracle backward (C, one thread) on the first {rows} of {w.M} rows of {w.name} per step; "
              f"GB/s counts the {w.dtype} workload's minimum bytes of those rows")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "sample_rows": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# activation backward: dx = dy * f'(preact)
# ---------------------------------------------------------------------------
ACT_METRIC = "activation bwd (dx = dy * f'(preact)) achieved HBM GB/s at M×N"


def act_cpu_baseline(a, target_s: float = 10.0):
    import oracle

    n = min(a.n, 1 << 22)
    inp = wl.make_act_inputs(a.with_shape(1, n))
    d, p = wl.exact_double(inp["dy"]).reshape(-1), wl.exact_double(inp["preact"]).reshape(-1)
    calls, t_total = 0, 0.0
    while t_total < target_s:
        t0 = time.perf_counter()
        oracle.act_bwd(a.kind, d, p)
        t_total += time.perf_counter() - t0
        calls += 1
    per_call = t_total / calls
    return {"value": round(wl.act_min_bytes(a.dtype, n) / per_call / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": (f"float64 oracle {a.kind} backward (C, one thread) on the first {n} of {a.n} elements "
                       f"of {a.name}, {calls} calls, {t_total:.1f} s; GB/s counts the {a.dtype} bytes")}


def run_activation(args):
    rank, world, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import rmsnorm_backward_gb300 as gbn

    a = wl.ACT_WORKLOADS[f"{args.activation}_bf16_16384x4096"]
    inp = wl.make_act_inputs(a)
    dy, pre = inp["dy"].to(device), inp["preact"].to(device)
    dx = torch.empty_like(dy)
    stream = torch.cuda.Stream(device)
    flush = L2Flush(device)
    L = gbn.lib()
    fn = getattr(L, f"{a.kind}_bwd")
    code = gbn.DTYPE_CODES[dy.dtype]
    call_args = (dy.data_ptr(), pre.data_ptr(), dx.data_ptr(), a.n, code, stream.cuda_stream)

    def step():
        st = fn(*call_args)
        if st != 0:
            raise RuntimeError(f"{a.kind}_bwd returned status {st}")

    K = args.steps
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush()
            step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local
    torch.cuda.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index, enabled=not args.no_clocks) as clk:
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for e in ev:
                flush()
                e[0].record(stream)
                step()
                e[1].record(stream)
        torch.cuda.synchronize()
        dist_barrier(world)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    times = np.array([e[0].elapsed_time(e[1]) for e in ev])
    t_s = dist_max(float(times.sum()) / 1e3, world, device)
    nbytes = wl.act_min_bytes(a.dtype, a.n)
    value = world * K * nbytes / t_s / 1e9
    peak, peak_src = measured_hbm_peak()
    avg = t_s / K
    # end to end through the public host-buffer call: pinned host dy, preact
    # in, dx out, the copies pipelined with the kernel inside the call
    h_dy, h_pre = inp["dy"].pin_memory(), inp["preact"].pin_memory()
    h_dx = torch.empty_like(h_dy).pin_memory()
    host_fn = getattr(gbn, f"{a.kind}_bwd_host")
    hws = torch.empty(int(L.gbn_act_host_workspace_bytes(a.n, code)), dtype=torch.uint8, device=device)

    def one():
        host_fn(h_dy, h_pre, dx=h_dx, workspace=hws, device=device, stream=stream)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        one()
    e1.record(stream)
    e1.synchronize()
    e2e_ms = dist_max(e0.elapsed_time(e1) / args.e2e_steps, world, device)
    if gbn.device_error(clear=True, device=device):
        raise SystemExit("kernel error flag set")
    if rank == 0:
        out = {
            "metric": ACT_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(avg * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": a.dtype, "data": "synthetic",
            "config": {"workload": a.name, "op": f"{a.kind} backward", "M": a.M, "N": a.N,
                       "inputs": wl.ACT_RECIPE, "seed": a.seed,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "flushed before every launch (256 MiB write, then a 256 MiB read)",
                       "timed": "CUDA events around each act_bwd launch on its stream"},
            "us": round(avg * 1e6, 3),
            "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "roofline": {"bound": "hbm", "achieved": round(nbytes / avg / 1e9, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(nbytes / avg / 1e9 / peak, 4), "traffic": recorded_traffic(a.name, "act_bwd_kernel"),
                         "kernel": "act_bwd_kernel", "algorithmic_bytes_per_launch": nbytes,
                         "peak_source": peak_src},
            "e2e": {"value": round(world * nbytes / (e2e_ms / 1e3) / 1e9, 3), "unit": "GB/s",
                    "h2d_bytes_per_step": 2 * a.n * wl.ELEM_BYTES[a.dtype],
                    "d2h_bytes_per_step": a.n * wl.ELEM_BYTES[a.dtype], "ms_per_step": round(e2e_ms, 4),
                    "what": f"{a.kind}_bwd_host: pinned host dy, preact in and dx out, copies pipelined with the "
                            "kernel over chunks inside the call"},
            "gpu_launches": K,
            "clocks": clk.summary(),
            "wall_s_timed_region": round(wall, 3),
        }
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = act_cpu_baseline(a)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_act_reference(args):
    """The float64 oracle's activation backward as the reference arm (rank 0 only)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle

    a = wl.ACT_WORKLOADS[f"{args.activation}_bf16_16384x4096"]
    n = min(a.n, 1 << 20)
    inp = wl.make_act_inputs(a.with_shape(1, n))
    d, p = wl.exact_double(inp["dy"]).reshape(-1), wl.exact_double(inp["preact"]).reshape(-1)
    for _ in range(args.warmup):
        oracle.act_bwd(a.kind, d, p)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.act_bwd(a.kind, d, p)
    dt = time.perf_counter() - t0
    value = args.steps * wl.act_min_bytes(a.dtype, n) / dt / 1e9
    sample = (f"float64 oracle {a.kind} backward (C, one thread) on the first {n} of {a.n} elements of "
              f"{a.name} per step; GB/s counts the {a.dtype} bytes of those elements")
    print(json.dumps({
        "impl": "reference", "metric": ACT_METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": a.name, "M": a.M, "N": a.N, "sample_elements": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_steady(args):
    """Back-to-back public backward calls with no L2 flush between them.

    Valid where x and dy together are larger than L2: a call reads its rows
    in the order the previous call read them, so it finds none of the
    previous call's inputs there.
    What it adds to the flushed per-call timing of the default run: the dx
    lines a call leaves dirty in L2 are written back while the next call
    streams its own reads, inside the timed region."""
    rank, world, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = wl.WORKLOADS[args.workload]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    in_bytes = 2 * w.M * w.N * wl.ELEM_BYTES[w.dtype]
    if in_bytes <= l2:
        raise SystemExit(f"{w.name}: x and dy ({in_bytes} bytes) fit in the L2 ({l2} bytes)")
    stream = torch.cuda.Stream(device)
    prob = Problem(w, device, stream, recompute=args.stats == "recompute", reduce=args.reduce, kernel=args.kernel)
    flush = L2Flush(device)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local
    K = args.steps
    with torch.cuda.stream(stream):
        flush()
        prob.fwd()
        for _ in range(max(args.warmup, 3)):
            prob.bwd_fused()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index, enabled=not args.no_clocks) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(K):
                prob.bwd_fused()
            e1.record(stream)
        torch.cuda.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    err = prob.gbn.device_error(clear=True, device=device)
    if err:
        raise SystemExit(f"kernel error flag set: {err}")
    t = dist_max(e0.elapsed_time(e1) / 1e3, world, device)
    bwd_bytes = wl.bwd_min_bytes(w.op, w.dtype, w.M, w.N)
    if args.stats == "recompute":
        bwd_bytes -= 4 * w.M * (2 if w.has_beta else 1)
    value = world * K * bwd_bytes / t / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(t / K * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "stats": args.stats, "reduce": args.reduce,
                       "kernel": args.kernel,
                       "timing": ("steady state: K public backward calls back to back between two events, no L2 "
                                  "flush; x and dy exceed the L2")},
            "bwd_us": round(t / K * 1e6, 3),
            "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "pct_of_measured_copy": round(100 * value / world / measured_hbm_peak()[0], 2),
            "gpu_launches": 2 * K,
            "clocks": clk.summary(),
        }), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.steady:
        run_steady(args)
        return
    if args.activation and args.impl == "reference":
        run_act_reference(args)
    elif args.activation:
        run_activation(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

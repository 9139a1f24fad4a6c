"""Benchmark: GiB/s written per fill at 2^28 elements on GB300.

One step is one pass of the whole hot path: every fill of the C ABI at 2^28
elements (u32, u64, f32, f64; the bounded and range fills; the f32 and f64
normals) plus dropout forward and backward at p = 0.1 and 0.5 on X[2^20, 256].
The outputs (1-2 GiB each) are far larger than the 129 MB L2, so no flush is
needed between timed steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is the bytes all fills wrote per
step over the step time (GiB/s, max over ranks), the `fills` table breaks it
down per fill, `roofline` relates the slowest kernel to the measured HBM
bandwidth, `e2e` repeats the step through the same C ABI with pinned host
buffers (inputs copied in, every output copied out, inside the timed
region), `cpu_baseline` times the CPU oracle on a bounded sample.  Under
torchrun each rank fills its own counter range (weak scaling, no data
exchange).  --impl reference times the CPU oracle itself as the reference
arm.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dropout_lowbias32_hash32_gb300 import workloads as W  # noqa: E402

GIB = float(1 << 30)
N = W.N_FULL
U32 = 1 << 32
METRIC = "GiB/s written per fill at 2^28 elements; % of GB300 HBM write roofline"
WORKLOAD = ("every fill at 2^28 elements per step: u32/u64/f32/f64 (seed 0x9E3779B9, first counter "
            "cycling 0, 1, 3, 2^32-5), u32_below(1000|2^32-2), u64_below(1000|2^64-2), i32/i64 "
            "low+below32(1000) and i64 low+below64(1000) (low -500, seeds 1..4), normal_f32 and "
            "normal_f64 (seed 7), dropout fwd+bwd on X[2^20,256] at p=0.1 and 0.5 (seed 42)")


# ---------------------------------------------------------------- the step --
def fill_specs():
    """(name, dtype, bytes per element written, bytes read, call(rng, out, first, x, y))."""
    b32, b64 = (1 << 32) - 2, (1 << 64) - 2
    return [
        ("u32", "int32", 4, 0, lambda r, o, f, s: r.rng_fill_u32(W.UNIFORM_SEED, f, o, s)),
        ("u64", "int64", 8, 0, lambda r, o, f, s: r.rng_fill_u64(W.UNIFORM_SEED, f, o, s)),
        ("f32", "float32", 4, 0, lambda r, o, f, s: r.rng_fill_f32(W.UNIFORM_SEED, f, o, s)),
        ("f64", "float64", 8, 0, lambda r, o, f, s: r.rng_fill_f64(W.UNIFORM_SEED, f, o, s)),
        ("u32_below_1000", "int32", 4, 0, lambda r, o, f, s: r.rng_fill_u32_below(1, f, 1000, o, s)),
        ("u32_below_2^32-2", "int32", 4, 0, lambda r, o, f, s: r.rng_fill_u32_below(2, f, b32, o, s)),
        ("u64_below_1000", "int64", 8, 0, lambda r, o, f, s: r.rng_fill_u64_below(3, f, 1000, o, s)),
        ("u64_below_2^64-2", "int64", 8, 0, lambda r, o, f, s: r.rng_fill_u64_below(4, f, b64, o, s)),
        ("i32_range", "int32", 4, 0, lambda r, o, f, s: r.rng_fill_i32_range(1, f, W.LOW, 1000, o, s)),
        ("i64_range32", "int64", 8, 0, lambda r, o, f, s: r.rng_fill_i64_range32(2, f, W.LOW, 1000, o, s)),
        ("i64_range", "int64", 8, 0, lambda r, o, f, s: r.rng_fill_i64_range(3, f, W.LOW, 1000, o, s)),
        ("normal_f32", "float32", 4, 0, lambda r, o, f, s: r.rng_fill_normal_f32(W.NORMAL_SEED, f, o, s)),
        ("normal_f64", "float64", 8, 0, lambda r, o, f, s: r.rng_fill_normal_f64(W.NORMAL_SEED, f, o, s)),
        ("dropout_fwd_p0.1", "x", 4, 4, lambda r, o, f, s: r.rng_dropout_fwd(o[0], o[1], 0.1, W.DROPOUT_SEED, f, s)),
        ("dropout_bwd_p0.1", "dy", 4, 4, lambda r, o, f, s: r.rng_dropout_bwd(o[0], o[1], 0.1, W.DROPOUT_SEED, f, s)),
        ("dropout_fwd_p0.5", "x", 4, 4, lambda r, o, f, s: r.rng_dropout_fwd(o[0], o[1], 0.5, W.DROPOUT_SEED, f, s)),
        ("dropout_bwd_p0.5", "dy", 4, 4, lambda r, o, f, s: r.rng_dropout_bwd(o[0], o[1], 0.5, W.DROPOUT_SEED, f, s)),
    ]


# Kernels each call launches and the kernel that dominates its time.
KERNELS_PER_CALL = {"normal_f64": 2}


def bytes_written_per_step(n: int) -> int:
    return sum(n * w for _, _, w, _, _ in fill_specs())


# ------------------------------------------------------------------ peaks --
def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None)}


# ------------------------------------------------------------- CPU oracle --
def oracle_sample(orc, n_sample: int, first: int):
    """Run every fill of the step on n_sample elements with the oracle;
    returns (seconds, bytes written) per fill."""
    x = W.dropout_x(n_sample)
    dy = W.dropout_dy(n_sample)
    calls = {
        "u32": lambda: orc.fill_u32(W.UNIFORM_SEED, first, n_sample),
        "u64": lambda: orc.fill_u64(W.UNIFORM_SEED, first, n_sample),
        "f32": lambda: orc.fill_f32(W.UNIFORM_SEED, first, n_sample),
        "f64": lambda: orc.fill_f64(W.UNIFORM_SEED, first, n_sample),
        "u32_below_1000": lambda: orc.fill_u32_below(1, first, 1000, n_sample),
        "u32_below_2^32-2": lambda: orc.fill_u32_below(2, first, U32 - 2, n_sample),
        "u64_below_1000": lambda: orc.fill_u64_below(3, first, 1000, n_sample),
        "u64_below_2^64-2": lambda: orc.fill_u64_below(4, first, (1 << 64) - 2, n_sample),
        "i32_range": lambda: orc.fill_i32_range(1, first, W.LOW, 1000, n_sample),
        "i64_range32": lambda: orc.fill_i64_range32(2, first, W.LOW, 1000, n_sample),
        "i64_range": lambda: orc.fill_i64_range(3, first, W.LOW, 1000, n_sample),
        "normal_f32": lambda: orc.fill_randn(W.NORMAL_SEED, first, n_sample),
        "normal_f64": lambda: orc.fill_normal_f64(W.NORMAL_SEED, first, n_sample),
        "dropout_fwd_p0.1": lambda: orc.dropout(x, 0.1, W.DROPOUT_SEED, first),
        "dropout_bwd_p0.1": lambda: orc.dropout(dy, 0.1, W.DROPOUT_SEED, first),
        "dropout_fwd_p0.5": lambda: orc.dropout(x, 0.5, W.DROPOUT_SEED, first),
        "dropout_bwd_p0.5": lambda: orc.dropout(dy, 0.5, W.DROPOUT_SEED, first),
    }
    out = {}
    for name, _, width, _, _ in fill_specs():
        t0 = time.perf_counter()
        calls[name]()
        out[name] = (time.perf_counter() - t0, n_sample * width)
    return out


def cpu_baseline(n_sample: int = 1 << 26):
    """The oracle, single-threaded, on n_sample elements of every fill: the
    GiB/s it would write over a whole step (bytes / summed seconds)."""
    import oracle
    orc = oracle.default()
    orc.zig1024()  # builds its table outside the timing
    res = oracle_sample(orc, n_sample, 0)
    secs = sum(t for t, _ in res.values())
    written = sum(b for _, b in res.values())
    return {"value": written / secs / GIB, "unit": "GiB/s", "cores": 1, "kind": "oracle",
            "sample": f"every fill of the step on {n_sample} elements (counters 0..{n_sample - 1}), "
                      f"single-threaded C oracle, {secs:.1f} s",
            "seconds": secs}


# --------------------------------------------------------------- our arm ---
def run_ours(args):
    import torch

    import dropout_lowbias32_hash32_gb300 as rng

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    n = args.n
    dev = torch.device("cuda", local)
    specs = fill_specs()
    buf4 = torch.empty(n, dtype=torch.int32, device=dev)
    buf8 = torch.empty(n, dtype=torch.int64, device=dev)
    host_x = torch.from_numpy(W.dropout_x(n)).pin_memory()
    host_dy = torch.from_numpy(W.dropout_dy(n)).pin_memory()
    x = host_x.to(dev)
    dy = host_dy.to(dev)
    y = torch.empty_like(x)
    outs = {"int32": buf4, "float32": buf4.view(torch.float32), "int64": buf8,
            "float64": buf8.view(torch.float64), "x": (x, y), "dy": (dy, y)}
    stream = torch.cuda.current_stream(dev)
    # rank r fills elements [r n, (r + 1) n) of each global fill
    base = (rank * n) & 0xFFFFFFFF

    def first_of(step):
        return (W.FIRST_COUNTERS[step % len(W.FIRST_COUNTERS)] + base) & 0xFFFFFFFF

    def step(k, events=None):
        f = first_of(k)
        for i, (name, kind, _, _, call) in enumerate(specs):
            first = f if name in ("u32", "u64", "f32", "f64") else base
            if events is not None:
                events[i][0].record(stream)
            call(rng, outs[kind], first, stream)
            if events is not None:
                events[i][1].record(stream)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()

    # per-fill events of every timed step
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in specs]
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = rng.rng_debug_launch_count()
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for k in range(args.steps):
            step(args.warmup + k, ev[k])
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
    launches = rng.rng_debug_launch_count() - launches0
    elapsed_ms = t_start.elapsed_time(t_end)
    if dist is not None:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    per_fill_ms = {name: statistics.median(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps))
                   for i, (name, *_rest) in enumerate(specs)}

    written = bytes_written_per_step(n)
    value = written * world * args.steps / (elapsed_ms / 1e3) / GIB
    peak, peak_kind = measured_peak_hbm()
    fills = {}
    for name, _, width, read, _ in specs:
        ms = per_fill_ms[name]
        gbs = (width + read) * n / (ms / 1e3) / 1e9
        fills[name] = {"ms": round(ms, 4), "gib_s_written": round(width * n / (ms / 1e3) / GIB, 1),
                       "gb_s_traffic": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 3)}
    dominant = max(specs, key=lambda s: per_fill_ms[s[0]])
    dname, _, dwidth, dread, _ = dominant
    dms = per_fill_ms[dname]
    achieved = (dwidth + dread) * n / (dms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 3), "traffic": None, "kernel": dname,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s"}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(rng, torch, specs, outs, (host_x, host_dy), x, dy, n, stream, barrier, dist, dev,
                      min(args.steps, 2), world)

    result = None
    if rank == 0:
        result = {
            "metric": METRIC, "value": round(value, 1), "unit": "GiB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic (counter-based fills need no input; dropout X ~ U(-1,1), dY ~ N(0,1) f32 "
                    "from numpy PCG64 seeds 11, 12)",
            "config": {"workload": WORKLOAD, "elements_per_fill": n, "fills_per_step": len(specs),
                       "bytes_written_per_step": written, "l2": "outputs of 1-2 GiB per fill exceed "
                       "the 129 MB L2; no flush between steps", "parallelism": f"counter-range shards x{world}"},
            "fills": fills, "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks.summary(), "cpu_baseline": None if args.no_cpu else cpu_baseline(),
        }
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return result


def run_e2e(rng, torch, specs, outs, host_inputs, x, dy, n, stream, barrier, dist, dev, steps, world):
    """The step through the C ABI with host buffers: each dropout input is
    copied from pinned host memory, each fill's output is copied back to
    pinned host memory, inside the timed region."""
    host_out = torch.empty(n * 8, dtype=torch.uint8, pin_memory=True)
    host_x, host_dy = host_inputs
    h2d = d2h = 0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for k in range(steps):
        for name, kind, width, _, call in specs:
            if kind in ("x", "dy"):
                src, dst = (host_x, x) if kind == "x" else (host_dy, dy)
                dst.copy_(src, non_blocking=True)
                h2d += n * 4
                target = outs[kind]
                call(rng, target, 0, stream)
                res = target[1]
            else:
                res = outs[kind]
                call(rng, res, 0, stream)
            host_out[:n * width].copy_(res.view(torch.uint8).view(-1)[:n * width], non_blocking=True)
            d2h += n * width
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = t0.elapsed_time(t1)
    if dist is not None:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = bytes_written_per_step(n) * world * steps / (ms / 1e3) / GIB
    return {"value": round(value, 1), "unit": "GiB/s", "h2d_bytes_per_step": h2d // steps,
            "d2h_bytes_per_step": d2h // steps, "steps": steps}


# --------------------------------------------------------- reference arm ---
def run_reference(args):
    """The CPU oracle as the reference arm: each step runs every fill of the
    step on a bounded sample and the metric scales to GiB/s written."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    orc = oracle.default()
    orc.zig1024()
    n_sample = args.ref_sample
    for k in range(args.warmup):
        oracle_sample(orc, max(n_sample // 16, 1024), k)
    t0 = time.perf_counter()
    written = 0
    for k in range(args.steps):
        res = oracle_sample(orc, n_sample, W.FIRST_COUNTERS[k % 4])
        written += sum(b for _, b in res.values())
    secs = time.perf_counter() - t0
    value = written / secs / GIB
    result = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GiB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "elements_per_fill": N,
                                        "reference_sample_per_fill": n_sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GiB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: every fill of the step on {n_sample} elements, "
                                   "single-threaded C oracle"},
        "e2e": {"value": round(value, 4), "unit": "GiB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)
    return result


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--n", type=int, default=N, help="elements per fill (default 2^28)")
    ap.add_argument("--ref-sample", type=int, default=1 << 20, help="oracle elements per fill and step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

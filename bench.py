"""Benchmark: GiB/s written per fill at 2^28 elements on GB300.

One step is one pass of the whole hot path: every fill of the C ABI at 2^28
elements (u32, u64, f32, f64; the bounded and range fills; the f32 and f64
normals) plus dropout forward and backward at p = 0.1 and 0.5 on X[2^20, 256].
The outputs (1-2 GiB each) are far larger than the 129 MB L2, so no flush is
needed between timed steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--only FILL[,FILL...]] [--n ELEMENTS] [--no-e2e] [--no-cpu] [--no-next]

Prints one JSON line (rank 0).  `value` is the bytes all fills wrote per
step over the step time (GiB/s, max over ranks); `fills` breaks it down per
fill (CUDA events around each call on its stream); `roofline` relates the
kernel with the largest share of the step to the measured HBM bandwidth and
`slowest_fill` gives the slowest call with the pipe that bounds it;
`next_rows` times the fills beyond the step (paired normals, narrow fills)
one by one, outside `value`; `configs` times the normals at 2^24 and 2^28
from first counters 0, 1 and 3; `context_curand` times cuRAND's Philox
fills of the same size on the same GPU (context only); `e2e`
repeats the step through the same C ABI with pinned host buffers (inputs
copied in, every output copied out, inside the timed region);
`cpu_baseline` times the CPU oracle on a bounded sample.  Under torchrun
each rank fills its own counter range (weak scaling, no data exchange).
--impl reference times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)



def _load_workloads():
    # by file path, so that the reference (oracle) arm does not run the
    # package's __init__, which maps the CUDA library
    import importlib.util
    path = os.path.join(ROOT, "dropout_lowbias32_hash32_gb300", "workloads.py")
    spec = importlib.util.spec_from_file_location("_lowbias32_workloads", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


W = _load_workloads()

GIB = float(1 << 30)
N = W.N_FULL
U32 = 1 << 32
METRIC = "GiB/s written per fill at 2^28 elements; % of GB300 HBM write roofline"
WORKLOAD = ("every fill at 2^28 elements per step: u32/u64/f32/f64 (seed 0x9E3779B9, first counter "
            "cycling 0, 1, 3, 2^32-5), u32_below(1000|2^32-2), u64_below(1000|2^64-2), i32/i64 "
            "low+below32(1000) and i64 low+below64(1000) (low -500, seeds 1..4), normal_f32 and "
            "normal_f64 (seed 7), dropout fwd+bwd on X[2^20,256] at p=0.1 and 0.5 (seed 42)")
CSRC = os.path.join(ROOT, "dropout_lowbias32_hash32_gb300", "csrc")
# the arithmetic types the step's fills compute in and store
DTYPE = "mixed: u32/u64/i32/i64 integer hashing, f32 and f64 arithmetic and outputs"


# ---------------------------------------------------------------- the step --
class Fill:
    """One call of the step: output buffer kind, bytes written and read per
    element, the kernel it launches and its source file, and the call."""

    def __init__(self, name, kind, written, read, kernel, source, call):
        self.name, self.kind, self.written, self.read = name, kind, written, read
        self.kernel, self.source, self.call = kernel, source, call


def fill_specs():
    b32, b64 = (1 << 32) - 2, (1 << 64) - 2
    F = Fill
    return [
        F("u32", "int32", 4, 0, "fill_kernel<GenU32>", "fill_uniform.cu",
          lambda r, o, f, s: r.rng_fill_u32(W.UNIFORM_SEED, f, o, s)),
        F("u64", "int64", 8, 0, "fill_kernel<GenU64>", "fill_uniform.cu",
          lambda r, o, f, s: r.rng_fill_u64(W.UNIFORM_SEED, f, o, s)),
        F("f32", "float32", 4, 0, "fill_kernel<GenF32>", "fill_uniform.cu",
          lambda r, o, f, s: r.rng_fill_f32(W.UNIFORM_SEED, f, o, s)),
        F("f64", "float64", 8, 0, "fill_kernel<GenF64>", "fill_uniform.cu",
          lambda r, o, f, s: r.rng_fill_f64(W.UNIFORM_SEED, f, o, s)),
        F("u32_below_1000", "int32", 4, 0, "fill_kernel<GenBelow32>", "fill_bounded.cu",
          lambda r, o, f, s: r.rng_fill_u32_below(1, f, 1000, o, s)),
        F("u32_below_2^32-2", "int32", 4, 0, "fill_kernel<GenBelow32>", "fill_bounded.cu",
          lambda r, o, f, s: r.rng_fill_u32_below(2, f, b32, o, s)),
        F("u64_below_1000", "int64", 8, 0, "fill_kernel<GenBelow64<1,0>>", "fill_bounded.cu",
          lambda r, o, f, s: r.rng_fill_u64_below(3, f, 1000, o, s)),
        F("u64_below_2^64-2", "int64", 8, 0, "fill_kernel<GenBelow64<1,1>>", "fill_bounded.cu",
          lambda r, o, f, s: r.rng_fill_u64_below(4, f, b64, o, s)),
        F("i32_range", "int32", 4, 0, "fill_kernel<GenI32Range>", "fill_bounded.cu",
          lambda r, o, f, s: r.rng_fill_i32_range(1, f, W.LOW, 1000, o, s)),
        F("i64_range32", "int64", 8, 0, "fill_kernel<GenI64Range32>", "fill_bounded.cu",
          lambda r, o, f, s: r.rng_fill_i64_range32(2, f, W.LOW, 1000, o, s)),
        F("i64_range", "int64", 8, 0, "fill_kernel<GenI64Range<1,0>>", "fill_bounded.cu",
          lambda r, o, f, s: r.rng_fill_i64_range(3, f, W.LOW, 1000, o, s)),
        F("normal_f32", "float32", 4, 0, "fill_kernel<GenNormalF32<1>>", "normal_f32.cu",
          lambda r, o, f, s: r.rng_fill_normal_f32(W.NORMAL_SEED, f, o, s)),
        F("normal_f64", "float64", 8, 0, "zig_table_pass<1>+zig_miss_pass", "normal_f64.cu",
          lambda r, o, f, s: r.rng_fill_normal_f64(W.NORMAL_SEED, f, o, s)),
        F("dropout_fwd_p0.1", "x", 4, 4, "dropout_v8_kernel", "dropout.cu",
          lambda r, o, f, s: r.rng_dropout_fwd(o[0], o[1], 0.1, W.DROPOUT_SEED, f, s)),
        F("dropout_bwd_p0.1", "dy", 4, 4, "dropout_v8_kernel", "dropout.cu",
          lambda r, o, f, s: r.rng_dropout_bwd(o[0], o[1], 0.1, W.DROPOUT_SEED, f, s)),
        F("dropout_fwd_p0.5", "x", 4, 4, "dropout_v8_kernel", "dropout.cu",
          lambda r, o, f, s: r.rng_dropout_fwd(o[0], o[1], 0.5, W.DROPOUT_SEED, f, s)),
        F("dropout_bwd_p0.5", "dy", 4, 4, "dropout_v8_kernel", "dropout.cu",
          lambda r, o, f, s: r.rng_dropout_bwd(o[0], o[1], 0.5, W.DROPOUT_SEED, f, s)),
    ]


def next_specs():
    """Fills beyond the measured step (timed separately, not part of `value`)."""
    F = Fill
    return [
        F("normal_f32_pairs", "float32", 4, 0, "fill_kernel<GenNormalF32Pairs>", "normal_f32.cu",
          lambda r, o, f, s: r.rng_fill_normal_f32_pairs(W.NORMAL_SEED, f, o, s)),
        F("normal_f32_precise", "float32", 4, 0, "fill_kernel<GenNormalF32Precise>", "normal_f32.cu",
          lambda r, o, f, s: r.rng_fill_normal_f32_precise(W.NORMAL_SEED, f, o, s)),
        F("exponential_f32", "float32", 4, 0, "neglog_table_kernel<GenExpF32>", "exponential.cu",
          lambda r, o, f, s: r.rng_fill_exponential_f32(W.NORMAL_SEED, f, o, s)),
        F("exponential_f64", "float64", 8, 0, "fill_kernel<GenExpF64>", "exponential.cu",
          lambda r, o, f, s: r.rng_fill_exponential_f64(W.NORMAL_SEED, f, o, s)),
        F("u8", "uint8", 1, 0, "fill_kernel<GenU8>", "fill_narrow.cu",
          lambda r, o, f, s: r.rng_fill_u8(W.UNIFORM_SEED, f, o, s)),
        F("u16", "int16", 2, 0, "fill_kernel<GenU16>", "fill_narrow.cu",
          lambda r, o, f, s: r.rng_fill_u16(W.UNIFORM_SEED, f, o, s)),
        F("f16", "float16", 2, 0, "fill_kernel<GenF16>", "fill_narrow.cu",
          lambda r, o, f, s: r.rng_fill_f16(W.UNIFORM_SEED, f, o, s)),
        F("bool", "bool", 1, 0, "fill_kernel<GenBool>", "fill_narrow.cu",
          lambda r, o, f, s: r.rng_fill_bool(W.UNIFORM_SEED, f, o, s)),
    ]


def selected_specs(only: str | None):
    """The step's fills, or with --only the named fills of the step or beyond it."""
    specs = fill_specs()
    if not only:
        return specs
    every = specs + next_specs()
    want = only.split(",")
    unknown = set(want) - {s.name for s in every}
    if unknown:
        raise SystemExit(f"unknown fills: {sorted(unknown)}")
    return [s for s in every if s.name in want]


# ------------------------------------------------------------------ peaks --
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return json.load(fh), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0}, "fallback"


def source_digest(source: str) -> str:
    """sha256 over a kernel's own source file and every header a kernel can
    include (csrc/*.cuh, *.h, *.inc and include/*): a change to any of them
    voids the kernel's recorded DRAM traffic."""
    import glob
    h = hashlib.sha256()
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                     glob.glob(os.path.join(CSRC, "*.inc")) + glob.glob(os.path.join(ROOT, "include", "*")))
    for path in [os.path.join(CSRC, source)] + headers:
        with open(path, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, source: str):
    """DRAM bytes per element of `kernel` from profiles/dram_traffic.txt (an
    ncu capture of dram__bytes_read.sum + dram__bytes_write.sum), or None if
    there is none or the kernel's sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    digest = source_digest(source)
    for line in lines:
        f = line.split()
        if len(f) >= 5 and f[0] == kernel and not line.startswith("#"):
            elements, read, write, dig = int(f[1]), int(f[2]), int(f[3]), f[4]
            if dig == digest:
                return (read + write) / elements
    return None


class ClockSampler:
    """SM clock, power and clock-event reasons sampled every 5 ms through NVML
    while the timed region runs (read-only queries)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str | None, period: float = 0.005):
        self.period, self.samples, self.max_mhz = period, [], None
        self.stop = threading.Event()
        self.thread = None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            handle = ctypes.c_void_p()
            if uuid is None or nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) != 0:
                raise OSError("no NVML handle for this device")
            self.nvml, self.handle = nvml, handle
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.error = None
        except OSError as exc:
            self.nvml, self.error = None, str(exc)

    def _run(self):
        clk, mw, reasons = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop.is_set():
            ok = self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0
            self.nvml.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(mw))
            get_reasons(self.handle, ctypes.byref(reasons))
            if ok:
                self.samples.append((clk.value, mw.value / 1000.0, reasons.value))
            self.stop.wait(self.period)

    def __enter__(self):
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [self.error or "no samples"]}
        reasons = sorted({name for _, _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples),
                "power_w_max": round(max(s[1] for s in self.samples), 1)}


# ------------------------------------------------------------- CPU oracle --
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_calls(orc, n_sample: int):
    """The step's fills on the oracle: fill -> call(first, off, n) returning
    elements [off, off + n) of the sample whose element 0 has counter first."""
    x = W.dropout_x(n_sample)
    dy = W.dropout_dy(n_sample)

    def drop(a, p):
        return lambda first, off, n: orc.dropout(a[off:off + n], p, W.DROPOUT_SEED, first + off)

    return {
        "u32": lambda first, off, n: orc.fill_u32(W.UNIFORM_SEED, first + off, n),
        "u64": lambda first, off, n: orc.fill_u64(W.UNIFORM_SEED, first + off, n),
        "f32": lambda first, off, n: orc.fill_f32(W.UNIFORM_SEED, first + off, n),
        "f64": lambda first, off, n: orc.fill_f64(W.UNIFORM_SEED, first + off, n),
        "u32_below_1000": lambda first, off, n: orc.fill_u32_below(1, first + off, 1000, n),
        "u32_below_2^32-2": lambda first, off, n: orc.fill_u32_below(2, first + off, U32 - 2, n),
        "u64_below_1000": lambda first, off, n: orc.fill_u64_below(3, first + off, 1000, n),
        "u64_below_2^64-2": lambda first, off, n: orc.fill_u64_below(4, first + off, (1 << 64) - 2, n),
        "i32_range": lambda first, off, n: orc.fill_i32_range(1, first + off, W.LOW, 1000, n),
        "i64_range32": lambda first, off, n: orc.fill_i64_range32(2, first + off, W.LOW, 1000, n),
        "i64_range": lambda first, off, n: orc.fill_i64_range(3, first + off, W.LOW, 1000, n),
        "normal_f32": lambda first, off, n: orc.fill_randn(W.NORMAL_SEED, first + off, n),
        "normal_f64": lambda first, off, n: orc.fill_normal_f64(W.NORMAL_SEED, first + off, n),
        "dropout_fwd_p0.1": drop(x, 0.1),
        "dropout_bwd_p0.1": drop(dy, 0.1),
        "dropout_fwd_p0.5": drop(x, 0.5),
        "dropout_bwd_p0.5": drop(dy, 0.5),
        "normal_f32_pairs": lambda first, off, n: orc.fill_randn_paired(W.NORMAL_SEED, first + off, n),
        "normal_f32_precise": lambda first, off, n: orc.fill_randn_precise(W.NORMAL_SEED, first + off, n),
        "exponential_f32": lambda first, off, n: orc.fill_exponential_f32_own(W.NORMAL_SEED, first + off, n),
        "exponential_f64": lambda first, off, n: orc.fill_exponential_f64(W.NORMAL_SEED, first + off, n),
        "u8": lambda first, off, n: orc.fill_u8(W.UNIFORM_SEED, first + off, n),
        "u16": lambda first, off, n: orc.fill_u16(W.UNIFORM_SEED, first + off, n),
        "f16": lambda first, off, n: orc.fill_f16_bits(W.UNIFORM_SEED, first + off, n),
        "bool": lambda first, off, n: orc.fill_bool(W.UNIFORM_SEED, first + off, n),
    }


def run_split(call, first: int, n: int, pool, parts: int):
    """One fill of n elements cut into `parts` counter ranges run on the
    pool's threads (the oracle's C calls release the GIL), concatenated."""
    bounds = [n * k // parts for k in range(parts + 1)]
    futs = [pool.submit(call, first, a, b - a) for a, b in zip(bounds, bounds[1:]) if b > a]
    return np.concatenate([f.result() for f in futs])


def oracle_sample(orc, specs, n_sample: int, first: int, pool=None, parts: int = 1, keep=False):
    """Run the step's fills on n_sample elements with the oracle, on one thread
    or split over the pool; returns {fill: (seconds, bytes written[, output])}."""
    calls = oracle_calls(orc, n_sample)
    out = {}
    for spec in specs:
        t0 = time.perf_counter()
        if pool is None:
            res = calls[spec.name](first, 0, n_sample)
        else:
            res = run_split(calls[spec.name], first, n_sample, pool, parts)
        out[spec.name] = (time.perf_counter() - t0, n_sample * spec.written) + ((res,) if keep else ())
    return out


def cpu_baseline(specs, n_sample: int = 1 << 26):
    """The oracle on n_sample elements of every fill of the step: on one
    thread, then cut into counter ranges over all host cores, whose
    concatenation must equal the one-thread output (the slice invariant).
    The value is the all-core rate, in GiB/s written over the whole step."""
    import concurrent.futures as cf

    import oracle
    orc = oracle.default()
    orc.zig1024()  # builds its table outside the timing
    cores = host_cores()
    single = multi = 0.0
    written = 0
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        for spec in specs:
            one = oracle_sample(orc, [spec], n_sample, 0, keep=True)[spec.name]
            split = oracle_sample(orc, [spec], n_sample, 0, pool=pool, parts=cores, keep=True)[spec.name]
            if one[2].tobytes() != split[2].tobytes():
                raise RuntimeError(f"oracle slice invariant broken on {spec.name}")
            single += one[0]
            multi += split[0]
            written += one[1]
    return {"value": round(written / multi / GIB, 4), "unit": "GiB/s", "cores": cores, "kind": "oracle",
            "single_core_value": round(written / single / GIB, 4),
            "sample": f"every fill of the step on {n_sample} elements (counters 0..{n_sample - 1}), the C "
                      f"oracle cut into {cores} counter ranges on {cores} threads ({multi:.1f} s; one thread: "
                      f"{single:.1f} s, same output)"}


# --------------------------------------------------------------- our arm ---
def device_uuid(torch, dev):
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    if uuid is None:
        return None
    uuid = str(uuid)
    return uuid if uuid.startswith("GPU-") else "GPU-" + uuid


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
    specs = selected_specs(args.only)
    buf4 = torch.empty(n, dtype=torch.int32, device=dev)
    buf8 = torch.empty(n, dtype=torch.int64, device=dev)
    needs_inputs = any(s.kind in ("x", "dy") for s in specs)
    host_x = torch.from_numpy(W.dropout_x(n)).pin_memory() if needs_inputs else None
    host_dy = torch.from_numpy(W.dropout_dy(n)).pin_memory() if needs_inputs else None
    x = host_x.to(dev) if needs_inputs else None
    dy = host_dy.to(dev) if needs_inputs else None
    y = torch.empty(n, dtype=torch.float32, device=dev) if needs_inputs else None
    outs = {"int32": buf4, "float32": buf4.view(torch.float32), "int64": buf8,
            "float64": buf8.view(torch.float64), "x": (x, y), "dy": (dy, y),
            "uint8": buf4.view(torch.uint8)[:n], "int16": buf4.view(torch.int16)[:n],
            "float16": buf4.view(torch.float16)[:n], "bool": buf4.view(torch.bool)[:n]}
    stream = torch.cuda.current_stream(dev)
    # rank r fills elements [r n, (r + 1) n) of each global fill
    base = (rank * n) & 0xFFFFFFFF

    def step(k, events=None):
        cycled = (W.FIRST_COUNTERS[k % len(W.FIRST_COUNTERS)] + base) & 0xFFFFFFFF
        for i, spec in enumerate(specs):
            first = cycled if spec.name in ("u32", "u64", "f32", "f64") else base
            if events is not None:
                events[i][0].record(stream)
            spec.call(rng, outs[spec.kind], first, stream)
            if events is not None:
                events[i][1].record(stream)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in specs]
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = rng.rng_debug_launch_count()
    with ClockSampler(device_uuid(torch, dev)) as clocks:
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
    fill_ms = {spec.name: statistics.median(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps))
               for i, spec in enumerate(specs)}
    fill_min = {spec.name: min(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps))
                for i, spec in enumerate(specs)}

    written = sum(n * s.written for s in specs)
    value = written * world * args.steps / (elapsed_ms / 1e3) / GIB
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    ceiling = write_ceiling(rng, torch, buf4, stream, max(args.steps, 5))
    wpeak = max(ceiling["memset_gb_s"], ceiling["store_v4_gb_s"])
    fills = {}
    for s in specs:
        ms = fill_ms[s.name]
        gbs = (s.written + s.read) * n / (ms / 1e3) / 1e9
        fills[s.name] = {"ms": round(ms, 4), "min_ms": round(fill_min[s.name], 4), "gib_s_written": round(s.written * n / (ms / 1e3) / GIB, 1),
                         "gb_s_traffic": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 3),
                         "kernel": s.kernel}
        if s.read == 0:
            fills[s.name]["frac_of_write_ceiling"] = round(gbs / wpeak, 3)

    # the kernel with the largest share of the step, over all of its calls
    by_kernel = {}
    for s in specs:
        ms, nbytes, src = by_kernel.get(s.kernel, (0.0, 0, s.source))
        by_kernel[s.kernel] = (ms + fill_ms[s.name], nbytes + (s.written + s.read) * n, src)
    kname, (kms, kbytes, ksrc) = max(by_kernel.items(), key=lambda kv: kv[1][0])
    calls = sum(1 for s in specs if s.kernel == kname)
    achieved = kbytes / (kms / 1e3) / 1e9
    per_elem = ncu_traffic(kname, ksrc)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 3),
                "traffic": None if per_elem is None else int(per_elem * n),
                "kernel": kname, "calls_per_step": calls,
                "share_of_step": round(kms / sum(fill_ms.values()), 3),
                "algorithmic_bytes_per_launch": kbytes // calls,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"
                if peak_kind == "measured" else "fallback 6.8 TB/s"}

    slowest = max(specs, key=lambda s: fill_ms[s.name])
    slow = {"fill": slowest.name, "kernel": slowest.kernel, "ms": fills[slowest.name]["ms"],
            "frac_of_hbm": fills[slowest.name]["frac_of_hbm"]}
    if slowest.name == "normal_f64":
        # the fast path spends one DFMA on three elements in four (the fourth takes the exact
        # integer product); GB300 retires 2 DFMA per SM and cycle
        props = torch.cuda.get_device_properties(dev)
        mhz = clocks.summary().get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
        fp64_peak = 2.0 * props.multi_processor_count * mhz * 1e6
        dfma = 3 / 4 * n / (fill_ms["normal_f64"] / 1e3)
        slow.update({"bound": "fp64", "achieved": round(dfma / 1e9, 1), "peak": round(fp64_peak / 1e9, 1),
                     "unit": "G DFMA/s (3 per 4 elements on the fast path)", "frac": round(dfma / fp64_peak, 3)})

    next_rows = None
    if not args.no_next and not args.only:
        next_rows = {}
        views = {"uint8": buf4.view(torch.uint8), "int16": buf4.view(torch.int16),
                 "float16": buf4.view(torch.float16), "bool": buf4.view(torch.bool), "float32": outs["float32"],
                 "float64": outs["float64"]}
        for spec in next_specs():
            out = views[spec.kind][:n]
            for _ in range(3):
                spec.call(rng, out, base, stream)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(max(args.steps, 5))]
            for a, b in evs:
                a.record(stream)
                spec.call(rng, out, base, stream)
                b.record(stream)
            torch.cuda.synchronize()
            ms = statistics.median(a.elapsed_time(b) for a, b in evs)
            gbs = spec.written * n / (ms / 1e3) / 1e9
            next_rows[spec.name] = {"ms": round(ms, 4), "gib_s_written": round(spec.written * n / (ms / 1e3) / GIB, 1),
                                    "frac_of_hbm": round(gbs / peak, 3),
                                    "frac_of_write_ceiling": round(gbs / wpeak, 3), "kernel": spec.kernel}

    context = None
    if not args.no_context and not args.only:
        context = curand_context(torch, buf8, stream, max(args.steps, 5), n)

    configs = None
    if not args.no_configs and not args.only:
        configs = normals_configs(rng, torch, buf8, stream, dev, max(args.steps, 5), base)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(rng, torch, specs, outs, (host_x, host_dy), x, dy, n, stream, barrier, dist, dev,
                      min(args.steps, 2), world)

    result = None
    if rank == 0:
        result = {
            "metric": METRIC, "value": round(value, 1), "unit": "GiB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
            "data": "synthetic (counter-based fills need no input; dropout X ~ U(-1,1), dY ~ N(0,1) f32 "
                    "from numpy PCG64 seeds 11, 12)",
            "config": {"workload": WORKLOAD if not args.only else f"{args.only} at {n} elements",
                       "elements_per_fill": n, "fills_per_step": len(specs), "bytes_written_per_step": written,
                       "l2": "outputs of 1-2 GiB per fill exceed the 129 MB L2; no flush between steps",
                       "parallelism": f"counter-range shards x{world}"},
            "fills": fills, "write_ceiling": ceiling, "roofline": roofline, "slowest_fill": slow, "next_rows": next_rows,
            "configs": configs, "context_curand": context, "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
            "cpu_baseline": None if args.no_cpu else cpu_baseline(specs),
        }
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return result


def normals_configs(rng, torch, buf8, stream, dev, reps, base):
    """The normals configuration rows: normal_f32 and normal_f64 (seed 7) at
    2^24 and 2^28 elements from first counters 0, 1 and 3, each the median of
    `reps` event-timed calls after 3 untimed ones.  Outputs of 2^24 elements
    (64 and 128 MiB) fit in the 129 MB L2, so a 512 MiB buffer is written
    between those timed calls (outside the events) to flush it; the 2^28
    outputs are larger than L2."""
    flush = torch.empty(1 << 29, dtype=torch.uint8, device=dev)
    rows = []
    for name, kind, written, fill in (
            ("normal_f32", torch.float32, 4, rng.rng_fill_normal_f32),
            ("normal_f64", torch.float64, 8, rng.rng_fill_normal_f64)):
        for n in W.NORMAL_SIZES:
            out = buf8.view(kind)[:n]
            for first in (0, 1, 3):
                c = (base + first) & 0xFFFFFFFF
                for _ in range(3):
                    fill(W.NORMAL_SEED, c, out, stream)
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(reps)]
                for a, b in evs:
                    if n * written <= (256 << 20):
                        flush.zero_()
                    a.record(stream)
                    fill(W.NORMAL_SEED, c, out, stream)
                    b.record(stream)
                torch.cuda.synchronize()
                ms = statistics.median(a.elapsed_time(b) for a, b in evs)
                rows.append({"fill": name, "elements": n, "first_counter": first, "ms": round(ms, 4),
                             "gib_s_written": round(written * n / (ms / 1e3) / GIB, 1),
                             "l2": "flushed between calls" if n * written <= (256 << 20) else "output > L2"})
    del flush
    return rows


def curand_context(torch, buf8, stream, reps, n):
    """cuRAND's Philox4x32-10 (host API), timed on the same GPU the same way
    as the fills (median of `reps` event-timed calls after 3 untimed ones) at
    the same size: context only, as the pages set their A100 fills beside it
    (tandem-cuda "Performance"); not a target and not part of the step."""
    lib = None
    for name in ("libcurand.so", "libcurand.so.10", "/usr/local/cuda/lib64/libcurand.so"):
        try:
            lib = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if lib is None:
        return {"unavailable": "libcurand not found"}
    gen = ctypes.c_void_p()
    philox = 161  # CURAND_RNG_PSEUDO_PHILOX4_32_10
    if lib.curandCreateGenerator(ctypes.byref(gen), philox) != 0:
        return {"unavailable": "curandCreateGenerator failed"}
    sz, vp = ctypes.c_size_t, ctypes.c_void_p
    lib.curandSetStream.argtypes = [vp, vp]
    lib.curandSetPseudoRandomGeneratorSeed.argtypes = [vp, ctypes.c_ulonglong]
    for f in ("curandGenerate", "curandGenerateUniform", "curandGenerateUniformDouble"):
        getattr(lib, f).argtypes = [vp, vp, sz]
    lib.curandGenerateNormal.argtypes = [vp, vp, sz, ctypes.c_float, ctypes.c_float]
    lib.curandGenerateNormalDouble.argtypes = [vp, vp, sz, ctypes.c_double, ctypes.c_double]
    lib.curandSetStream(gen, vp(stream.cuda_stream or None))
    lib.curandSetPseudoRandomGeneratorSeed(gen, 7)
    ptr = vp(buf8.data_ptr())
    calls = [("u32 (curandGenerate)", 4, lambda: lib.curandGenerate(gen, ptr, n)),
             ("f32 uniform (curandGenerateUniform)", 4, lambda: lib.curandGenerateUniform(gen, ptr, n)),
             ("f64 uniform (curandGenerateUniformDouble)", 8, lambda: lib.curandGenerateUniformDouble(gen, ptr, n)),
             ("normal f32 (curandGenerateNormal)", 4, lambda: lib.curandGenerateNormal(gen, ptr, n, 0.0, 1.0)),
             ("normal f64 (curandGenerateNormalDouble)", 8,
              lambda: lib.curandGenerateNormalDouble(gen, ptr, n, 0.0, 1.0))]
    rows = {}
    try:
        for name, size, call in calls:
            for _ in range(3):
                if call() != 0:
                    raise RuntimeError(name)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for a, b in evs:
                a.record(stream)
                call()
                b.record(stream)
            torch.cuda.synchronize()
            ms = statistics.median(a.elapsed_time(b) for a, b in evs)
            rows[name] = {"ms": round(ms, 4), "gib_s_written": round(size * n / (ms / 1e3) / GIB, 1)}
    except RuntimeError as exc:
        rows["unavailable"] = f"{exc} failed"
    finally:
        lib.curandDestroyGenerator(gen)
    return {"generator": "cuRAND Philox4x32-10, host API", "elements": n, "rows": rows}


def write_ceiling(rng, torch, buf, stream, reps):
    """The write ceiling measured live on this GPU, outside the timed region:
    cudaMemsetAsync and the plainest 16-byte store kernel over the 4-byte
    output buffer (median of reps event-timed calls after 3 untimed)."""
    nbytes = buf.numel() * buf.element_size()
    out = {"bytes": nbytes}
    for which, key in ((0, "memset_gb_s"), (1, "store_v4_gb_s")):
        for _ in range(3):
            rng.rng_debug_write_ceiling(which, buf, stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in evs:
            a.record(stream)
            rng.rng_debug_write_ceiling(which, buf, stream)
            b.record(stream)
        torch.cuda.synchronize()
        out[key] = round(nbytes / (statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3) / 1e9, 1)
    return out


def run_e2e(rng, torch, specs, outs, host_inputs, x, dy, n, stream, barrier, dist, dev, steps, world):
    """The step through the C ABI with host buffers, inside the timed region:
    each dropout input is copied from pinned host memory and every fill's
    output is copied back to pinned host memory.  Three streams overlap the
    two copy directions with the fills: the fills run on `stream`,
    host-to-device copies on one side stream and device-to-host copies on
    another; outputs and dropout inputs are double-buffered on the device,
    and events keep a fill from overwriting a buffer before its copy out has
    read it (and a copy in from overwriting an input a dropout still reads)."""
    del outs, x, dy  # the pipelined step has its own double buffers
    host_x, host_dy = host_inputs
    dtypes = {"int32": torch.int32, "float32": torch.float32, "int64": torch.int64, "float64": torch.float64,
              "x": torch.float32, "dy": torch.float32}
    dev_out = [torch.empty(n * 8, dtype=torch.uint8, device=dev) for _ in range(2)]
    host_out = [torch.empty(n * 8, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    dev_in = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def event(s):
        e = torch.cuda.Event()
        e.record(s)
        return e

    def one_step(state):
        h2d = d2h = 0
        for spec in specs:
            b = state["k"] % 2
            if state["out_free"][b] is not None:
                stream.wait_event(state["out_free"][b])
            out = dev_out[b].view(dtypes[spec.kind])[:n]
            if spec.kind in ("x", "dy"):
                ib = state["ki"] % 2
                if state["in_free"][ib] is not None:
                    s_in.wait_event(state["in_free"][ib])
                with torch.cuda.stream(s_in):
                    dev_in[ib].copy_(host_x if spec.kind == "x" else host_dy, non_blocking=True)
                stream.wait_event(event(s_in))
                spec.call(rng, (dev_in[ib], out), 0, stream)
                state["in_free"][ib] = event(stream)
                state["ki"] += 1
                h2d += n * 4
            else:
                spec.call(rng, out, 0, stream)
            nbytes = n * spec.written
            s_out.wait_event(event(stream))
            with torch.cuda.stream(s_out):
                host_out[b][:nbytes].copy_(dev_out[b][:nbytes], non_blocking=True)
            state["out_free"][b] = event(s_out)
            state["k"] += 1
            d2h += nbytes
        return h2d, d2h

    state = {"k": 0, "ki": 0, "out_free": [None, None], "in_free": [None, None]}
    one_step(state)  # untimed warm-up
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    start = event(stream)
    s_in.wait_event(start)
    s_out.wait_event(start)
    h2d = d2h = 0
    for _ in range(steps):
        a, b = one_step(state)
        h2d, d2h = h2d + a, d2h + b
    stream.wait_event(event(s_out))
    stream.wait_event(event(s_in))
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = t0.elapsed_time(t1)
    if dist is not None:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = sum(n * s.written for s in specs) * world * steps / (ms / 1e3) / GIB
    return {"value": round(value, 1), "unit": "GiB/s", "h2d_bytes_per_step": h2d // steps,
            "d2h_bytes_per_step": d2h // steps, "steps": steps,
            "pipelining": "fills, host-to-device and device-to-host copies on three streams"}


# --------------------------------------------------------- reference arm ---
def run_reference(args):
    """The CPU oracle as the reference arm: each step runs every fill of the
    step on a bounded sample and the metric scales to GiB/s written."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import concurrent.futures as cf

    import oracle
    orc = oracle.default()
    orc.zig1024()
    specs = selected_specs(args.only)
    n_sample = args.ref_sample
    cores = host_cores()
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        for k in range(args.warmup):
            oracle_sample(orc, specs, max(n_sample // 16, 1024), k, pool=pool, parts=cores)
        t0 = time.perf_counter()
        written = 0
        for k in range(args.steps):
            res = oracle_sample(orc, specs, n_sample, W.FIRST_COUNTERS[k % 4], pool=pool, parts=cores)
            written += sum(r[1] for r in res.values())
        secs = time.perf_counter() - t0
    value = written / secs / GIB
    result = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GiB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic", "config": {"workload": WORKLOAD, "elements_per_fill": N,
                                        "reference_sample_per_fill": n_sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GiB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: every fill of the step on {n_sample} elements, the C oracle "
                                   f"cut into {cores} counter ranges on {cores} threads"},
        "e2e": {"value": round(value, 4), "unit": "GiB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)
    return result


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--n", type=int, default=N, help="elements per fill (default 2^28)")
    ap.add_argument("--only", help="comma-separated fills of the step to run (default: all)")
    ap.add_argument("--ref-sample", type=int, default=1 << 20, help="oracle elements per fill and step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the fills beyond the step")
    ap.add_argument("--no-configs", action="store_true", help="skip the normals configuration rows")
    ap.add_argument("--no-context", action="store_true", help="skip the cuRAND context rows")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

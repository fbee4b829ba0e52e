#!/usr/bin/env python3
"""Benchmark of the row-major GEMM library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-extras] [--no-cpu-baseline]

One step is one C-ABI call computing C = alpha*A*B + beta*C on the named
workload (default: bf16 8192^3, the tensor-core path). Inputs are resident in
HBM before the timed region; A + B alone exceed the 129 MB L2, so no L2 flush
is needed between steps. The device-timed value uses CUDA events on the
launching stream around exactly K back-to-back steps, after W warm-up steps,
bracketed by a barrier and a device synchronise; the max over ranks is taken.

The printed JSON line also carries:
  e2e           the same metric through the C ABI with pinned HOST buffers:
                every step copies A and B host->device and C device->host;
                three steps are in flight on three streams (serial_ms_per_step
                gives the one-stream figure).
  roofline      achieved TFLOP/s of the dominant kernel against the measured
                peak of its pipe, and ncu DRAM traffic per launch when a
                capture of the current kernel source is recorded.
  cpu_baseline  the CPU oracle timed on this host's cores on a bounded row
                sample of the same workload (rank 0, N = 1 only).
  clocks        SM clock (median) and throttle reasons sampled by nvidia-smi
                during the timed region.
  extras        the other workloads (fp32 4096^3, fp16 8192^3, int8 8192^3),
                each with its own roofline fraction.

--impl reference times the CPU oracle itself (the only reference that exists
for this path) on the same workload, a bounded row sample per step.
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(weak scaling, no data exchange); value = all ranks' flops / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (TOPS int8) and % of FP32/tensor-pipe peak at M=N=K=4096/8192"

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}

# workload name -> description, entry point, pipe that bounds it
WORKLOADS = {
    "bf16_8192": ("bf16 GEMM, row-major, M=N=K=8192, N(0,1) rounded to bf16, fp32 accumulate "
                  "and fp32 C, alpha=1, beta=0", "bf16", "tensor", 1),
    "f16_8192": ("fp16 GEMM, row-major, M=N=K=8192, N(0,1) rounded to fp16, fp32 accumulate "
                 "and fp32 C, alpha=1, beta=0", "f16", "tensor", 1),
    "f32_4096": ("fp32 SGEMM (SIMT, exact fp32), row-major, M=N=K=4096, N(0,1), alpha=1, beta=0",
                 "f32", "alu", 2),
    "s8_8192": ("int8 GEMM, row-major, M=N=K=8192, uniform -128..127, exact int32 accumulate "
                "and int32 C, alpha=1, beta=0", "s8", "tensor", 3),
    "f32_8192": ("fp32 SGEMM (SIMT, exact fp32), row-major, M=N=K=8192, N(0,1), alpha=1, beta=0",
                 "f32", "alu", 2),
    "bf16_4096": ("bf16 GEMM, row-major, M=N=K=4096, N(0,1) rounded to bf16, fp32 accumulate "
                  "and fp32 C, alpha=1, beta=0", "bf16", "tensor", 1),
    "s8_4096": ("int8 GEMM, row-major, M=N=K=4096, uniform -128..127, exact int32 accumulate "
                "and int32 C, alpha=1, beta=0", "s8", "tensor", 3),
}

# Sources whose change invalidates recorded ncu traffic for a workload.
KERNEL_SOURCES = {
    "bf16_8192": ["gemm_tc_kernel.cuh", "gemm_tc_f16.cu", "work_split.cuh", "ptx.cuh"],
    "f16_8192": ["gemm_tc_kernel.cuh", "gemm_tc_f16.cu", "work_split.cuh", "ptx.cuh"],
    "s8_8192": ["gemm_tc_kernel.cuh", "gemm_tc_int.cu", "work_split.cuh", "ptx.cuh"],
    "f32_4096": ["sgemm_simt.cu", "work_split.cuh", "ptx.cuh"],
    "f32_8192": ["sgemm_simt.cu", "work_split.cuh", "ptx.cuh"],
    "bf16_4096": ["gemm_tc_kernel.cuh", "gemm_tc_f16.cu", "work_split.cuh", "ptx.cuh"],
    "s8_4096": ["gemm_tc_kernel.cuh", "gemm_tc_int.cu", "work_split.cuh", "ptx.cuh"],
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(name: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[name]:
        with open(os.path.join(ROOT, "dense_gemm_row_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str):
    """DRAM bytes per launch from profiles/ncu_traffic.txt, only if recorded
    for the current kernel source (digest match)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    digest = source_digest(name)
    for line in lines:
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == name and parts[1] == digest:
            return float(parts[2])
    return None


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi in the background; samples are kept with their wall time."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        time.sleep(0.5)  # let the first samples arrive

    def _reader(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        def parse(line):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                return None
            try:
                return {"sm": float(f[1]), "max": float(f[2]),
                        "reasons": {"hw_slowdown": f[5], "hw_thermal_slowdown": f[6],
                                    "sw_thermal_slowdown": f[7], "sw_power_cap": f[8]}}
            except ValueError:
                return None
        rows = [(t, parse(l)) for t, l in self.samples]
        rows = [(t, r) for t, r in rows if r]
        inside = [r for t, r in rows if t0 - 0.15 <= t <= t1 + 0.15]
        window = "timed"
        if not inside:
            inside = [r for _, r in rows]
            window = "warmup+timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "none"}
        reasons = sorted({k for r in inside for k, v in r["reasons"].items() if v == "Active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["max"] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ----------------------------------------------------------------- GPU timing

def flops_of(M, N, K):
    return 2.0 * M * N * K


def entry(binding, kind):
    return {"bf16": binding.gemm_bf16, "f16": binding.gemm_f16, "f32": binding.gemm_f32,
            "s8": binding.gemm_s8}[kind]


def time_device(binding, torch, kind, p_dev, steps, warmup, stream, dist=None):
    A, B, C, alpha, beta = p_dev
    M, K = A.shape
    N = B.shape[1]
    fn = entry(binding, kind)
    args = (M, N, K, alpha, A, A.stride(0), B, B.stride(0), beta, C, C.stride(0), stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn(*args)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record(stream)
    for _ in range(steps):
        fn(*args)
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    return ms, t0, t1


L2_BYTES = 129e6


def time_device_flushed(binding, torch, kind, p_dev, steps, warmup, stream):
    """For inputs that fit in L2: each timed call is preceded, outside its
    event pair and on the same stream, by a 256 MB write that evicts L2.
    Returns the summed device time of the calls and the wall window."""
    A, B, C, alpha, beta = p_dev
    M, K = A.shape
    N = B.shape[1]
    fn = entry(binding, kind)
    args = (M, N, K, alpha, A, A.stride(0), B, B.stride(0), beta, C, C.stride(0), stream)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn(*args)
    torch.cuda.synchronize()
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)]
    t0 = time.time()
    with torch.cuda.stream(stream):
        for e0, e1 in pairs:
            flush.zero_()
            e0.record(stream)
            fn(*args)
            e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in pairs)
    del flush
    return ms, t0, t1


def time_e2e(binding, torch, kind, p_host, p_dev, steps, stream):
    """Host -> device copy of A and B, the C-ABI call, device -> host copy of C."""
    (Ah, Bh, Ch), (A, B, C, alpha, beta) = p_host, p_dev
    M, K = A.shape
    N = B.shape[1]
    fn = entry(binding, kind)
    args = (M, N, K, alpha, A, A.stride(0), B, B.stride(0), beta, C, C.stride(0), stream)

    def step():
        with torch.cuda.stream(stream):
            A.copy_(Ah, non_blocking=True)
            B.copy_(Bh, non_blocking=True)
            fn(*args)
            Ch.copy_(C, non_blocking=True)
    step()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    h2d = Ah.numel() * Ah.element_size() + Bh.numel() * Bh.element_size()
    d2h = Ch.numel() * Ch.element_size()
    return ev0.elapsed_time(ev1), h2d, d2h


def time_e2e_pipelined(binding, torch, kind, p_host, p_dev, steps, stream, depth=3):
    """The same end-to-end step, `depth` steps in flight: step i runs on stream
    i % depth with its own device buffers (H2D of A and B from the pinned host
    copies, the C-ABI call, D2H of C into its own pinned buffer), so one step's
    copies overlap another step's GEMM, as a caller streaming problems through
    the library would arrange it. Every step still moves all of its bytes."""
    (Ah, Bh, Ch), (A, B, C, alpha, beta) = p_host, p_dev
    M, K = A.shape
    N = B.shape[1]
    fn = entry(binding, kind)
    sets = [(A, B, C, Ch)]
    for _ in range(depth - 1):
        sets.append((torch.empty_like(A), torch.empty_like(B), torch.empty_like(C),
                     torch.empty_like(Ch).pin_memory()))
    streams = [torch.cuda.Stream() for _ in range(depth)]

    def step(i):
        a, b, c, ch = sets[i % depth]
        s = streams[i % depth]
        with torch.cuda.stream(s):
            a.copy_(Ah, non_blocking=True)
            b.copy_(Bh, non_blocking=True)
            fn(M, N, K, alpha, a, a.stride(0), b, b.stride(0), beta, c, c.stride(0), s)
            ch.copy_(c, non_blocking=True)
    for i in range(depth):
        step(i)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for s in streams:
        s.wait_event(ev0)
    for i in range(steps):
        step(i)
    for s in streams:
        done = torch.cuda.Event()
        done.record(s)
        stream.wait_event(done)
    ev1.record(stream)
    torch.cuda.synchronize()
    del sets
    return ev0.elapsed_time(ev1)


def device_problem(torch, p):
    A = p.A.cuda()
    B = p.B.cuda()
    C = p.C0.cuda()
    return A, B, C, p.alpha, p.beta


def peak_for(kind, peaks, sm_count, sustained=False):
    if kind == "f32":
        # FP32 SIMT: SMs x 128 FMA lanes x 2 flops x maximum SM clock.
        mhz = float(peaks.get("sm_max_mhz", 2070.0))
        return sm_count * 128 * 2 * mhz * 1e6 / 1e12
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    # fp16 and the int8 path (run as integer-valued fp16 on kind::f16) share the
    # bf16 dense rate of the tensor pipe.
    return float(peaks.get(key, FALLBACK_PEAKS[key]))


# ------------------------------------------------------------- CPU baseline

def cpu_oracle_sample(p, seconds: float):
    """Times the oracle on a row sample of p sized for about `seconds`."""
    import torch  # noqa: F401
    from oracle import oracle as o
    M, K = p.A.shape
    N = p.B.shape[1]

    def run(rows):
        idx = list(range(rows))
        t = time.perf_counter()
        o.gemm_rows(p.A, p.B, idx, p.alpha, p.beta, p.C0)
        return time.perf_counter() - t

    probe = min(M, 8)
    t_probe = run(probe)
    rows = probe
    if t_probe < seconds:
        rows = int(min(M, max(probe, probe * seconds / max(t_probe, 1e-6))))
    t = run(rows) if rows != probe else t_probe
    return {"rows": rows, "seconds": t, "flops": flops_of(rows, N, K), "cores": o.num_threads(),
            "sample": f"rows 0..{rows - 1} of A ({rows} of {M}) against all of B; "
                      f"{flops_of(rows, N, K) / 1e9:.1f} GFLOP per sample"}


def cpu_oracle_configs(w):
    """The oracle on the small configs in full (fp32 128^3 integers, the
    1023x777x513 ragged case, 4096^3) on all host threads, and 1024^3 on one
    thread (a child process with OMP_NUM_THREADS=1: OpenMP fixes its thread
    count at start-up)."""
    from oracle import oracle as o
    out = {}
    for name in ("f32_int128", "f32_ragged", "f32_4096"):
        q = w.config(name)
        M, K = q.A.shape
        N = q.B.shape[1]
        t = time.perf_counter()
        o.gemm(q.A, q.B, q.alpha, q.beta, q.C0 if q.beta != 0 else None)
        dt = time.perf_counter() - t
        out[name] = {"seconds": dt, "gflops": flops_of(M, N, K) / dt / 1e9,
                     "cores": o.num_threads()}
    code = ("import json, time, torch\n"
            "from oracle import oracle as o\n"
            "g = torch.Generator().manual_seed(9)\n"
            "A = torch.randn(1024, 1024, generator=g); B = torch.randn(1024, 1024, generator=g)\n"
            "t = time.perf_counter(); o.gemm(A, B, 1.0, 0.0); dt = time.perf_counter() - t\n"
            "print(json.dumps({'seconds': dt, 'cores': o.num_threads()}))\n")
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                           timeout=600, env=dict(os.environ, OMP_NUM_THREADS="1"))
        one = json.loads(r.stdout.strip().splitlines()[-1])
        one["gflops"] = flops_of(1024, 1024, 1024) / one["seconds"] / 1e9
        out["f32_1024_one_core"] = one
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        out["f32_1024_one_core"] = {"error": str(e)[:200]}
    return out


def measure_peaks(binding, torch, peaks, sm_count, stream, gpu_id):
    """The build's own peak microbenchmarks: packed fp32 FMA and tcgen05
    kind::f16 issue loops (best of 5 launches of about 10 ms each)."""
    sink = torch.zeros(1, device="cuda")
    runs = (("ffma", lambda it: binding.peak_ffma(it, sink, stream), 65536),
            ("tc_f16", lambda it: binding.peak_tc_f16(it, stream), 40000))
    out = {}
    for name, fn, iters in runs:
        fn(256)
        torch.cuda.synchronize()
        sampler = ClockSampler(gpu_id)
        sampler.start()
        times, flops = [], 0.0
        t0 = time.time()
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            flops = fn(iters)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        t1 = time.time()
        sampler.stop()
        clocks = sampler.summary(t0, t1)
        ms = min(times)
        out[name] = {"tflops": flops / (ms / 1e3) / 1e12, "ms": ms, "iters": iters,
                     "sm_mhz": clocks["sm_mhz"], "reasons": clocks["reasons"]}
    max_mhz = peaks.get("sm_max_mhz", 2070.0)
    nominal = sm_count * 128 * 2 * max_mhz * 1e6 / 1e12
    out["ffma"]["nominal_at_max_clock"] = nominal
    out["ffma"]["frac_of_nominal"] = out["ffma"]["tflops"] / nominal
    out["tc_f16"]["cublas_burst"] = peaks.get("bf16_tflops")
    out["tc_f16"]["dense_at_max_clock"] = sm_count * 8192 * max_mhz * 1e6 / 1e12
    binding.check_device_error()
    return out


# ------------------------------------------------------------------ reference

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from dense_gemm_row_gb300 import workloads as w
    name = args.workload
    desc, kind, bound, _ = WORKLOADS[name]
    p = w.config(name)
    M, K = p.A.shape
    N = p.B.shape[1]
    # Size one step so the whole run ends within about two minutes.
    total_steps = max(1, args.steps + args.warmup)
    per_step = min(20.0, max(0.5, 120.0 / total_steps))
    cal = cpu_oracle_sample(p, per_step)
    rows = cal["rows"]
    from oracle import oracle as o
    idx = list(range(rows))
    for _ in range(args.warmup):
        o.gemm_rows(p.A, p.B, idx, p.alpha, p.beta, p.C0)
    t = time.perf_counter()
    for _ in range(args.steps):
        o.gemm_rows(p.A, p.B, idx, p.alpha, p.beta, p.C0)
    elapsed = time.perf_counter() - t
    value = flops_of(rows, N, K) * args.steps / elapsed / 1e12
    unit = "TOPS" if kind == "s8" else "TFLOP/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64" if kind == "s8" else "f64", "data": "synthetic",
        "config": {"workload": desc, "M": M, "N": N, "K": K, "parallelism": "cpu-host"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cal["cores"], "kind": "oracle",
                         "sample": cal["sample"] + " per step"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def aggregate_ranks(torch, dist, ms, flops_per_step, steps, device):
    """Whole-job throughput over the ranks: every rank ran `steps` steps of
    `flops_per_step` in `ms` milliseconds of its own; the job's time is the
    slowest rank's. Returns (max ms over ranks, TFLOP/s of all ranks together).
    Without a process group this is the single-GPU figure."""
    world = 1
    ms_max = float(ms)
    if dist is not None:
        world = dist.get_world_size()
        t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
    value = world * flops_per_step * steps / (ms_max / 1e3) / 1e12
    return ms_max, value


# ------------------------------------------------------------ other workloads

def measure_extra(binding, torch, w, name, peaks, sm_count, stream, gpu_id):
    """Device-timed throughput of another named workload, with its own clock
    samples and roofline fraction."""
    desc, kind, bound, _ = WORKLOADS[name]
    q = w.config(name)
    q_dev = device_problem(torch, q)
    M, K = q.A.shape
    N = q.B.shape[1]
    steps = 100 if kind != "f32" else 60
    in_l2 = sum(t.numel() * t.element_size() for t in q_dev[:3]) < 1.5 * L2_BYTES
    sampler = ClockSampler(gpu_id)
    sampler.start()
    if in_l2:
        ms, t0, t1 = time_device_flushed(binding, torch, kind, q_dev, steps, 5, stream)
    else:
        ms, t0, t1 = time_device(binding, torch, kind, q_dev, steps, 5, stream)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    f = flops_of(M, N, K)
    ach = f / (ms / steps / 1e3) / 1e12
    pk = peak_for(kind, peaks, sm_count)
    out = {"workload": desc, "value": ach, "unit": "TOPS" if kind == "s8" else "TFLOP/s",
           "ms_per_step": ms / steps, "bound": bound, "peak": pk, "frac": ach / pk,
           "traffic": recorded_traffic(name),
           "l2": ("flushed by a 256 MB write before each timed call" if in_l2
                  else "no flush: A+B+C exceed 1.5 x the 129 MB L2"),
           "clocks": {"sm_mhz": clocks["sm_mhz"], "reasons": clocks["reasons"],
                      "samples": clocks["samples"]}}
    if kind == "f32" and clocks["sm_mhz"]:
        out["frac_at_sampled_clock"] = ach / (sm_count * 128 * 2 * clocks["sm_mhz"] * 1e6 / 1e12)
    if kind == "s8":
        out["note"] = "step includes the two int8->fp16 widening launches"
    elif kind == "f32":
        out["note"] = "step includes the transposition of A ahead of the SIMT kernel"
    del q_dev
    torch.cuda.empty_cache()
    return out


def time_skinny(binding, torch, kind, p_dev, stream, steps=20):
    """Seconds per call of a memory-bound shape, calls back to back. Operands
    that fit in L2 (int8 8192 x 8192 is 67 MB) would be read from it by the
    next call, so the calls then cycle through enough copies of A and B that
    each copy has been evicted by the time it is read again (at least twice
    the L2 between reuses); larger operands are used as they are."""
    A, B, C, alpha, beta = p_dev
    nbytes = A.numel() * A.element_size() + B.numel() * B.element_size()
    copies = 1
    if nbytes < 1.5 * L2_BYTES:
        copies = int(math.ceil(2 * L2_BYTES / nbytes)) + 1
    def copy_of(t):  # same strides (a 16-bit B keeps its padded row stride)
        return torch.empty_strided(t.size(), t.stride(), dtype=t.dtype,
                                   device=t.device).copy_(t)
    sets = [(A, B)] + [(copy_of(A), copy_of(B)) for _ in range(copies - 1)]
    M, K = A.shape
    N = B.shape[1]
    fn = entry(binding, kind)
    calls = [(M, N, K, alpha, a, a.stride(0), b, b.stride(0), beta, C, C.stride(0), stream)
             for a, b in sets]
    with torch.cuda.stream(stream):
        for i in range(max(3, copies)):
            fn(*calls[i % copies])
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        fn(*calls[i % copies])
    ev1.record(stream)
    torch.cuda.synchronize()
    del sets, calls
    return copies, ev0.elapsed_time(ev1) / steps / 1e3


def measure_skinny(binding, torch, peaks, stream):
    """Memory-bound shapes M in {1, 16, 64}, N = K = 8192, and tall, narrow
    ones (M = K = 8192, N = 1; N = 16 for fp32 and int8): HBM GB/s of the
    algorithmic bytes (A and B read once, C written once) against the
    measured copy bandwidth; operands smaller than 1.5 x L2 are read from
    rotating copies, so that no call finds them in L2 (time_skinny)."""
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    N = K = 8192
    out = {}
    for kind, dt, cdt in (("bf16", torch.bfloat16, torch.float32),
                          ("f16", torch.float16, torch.float32),
                          ("f32", torch.float32, torch.float32),
                          ("s8", torch.int8, torch.int32)):
        if kind == "s8":
            B = torch.randint(-128, 128, (K, N), device="cuda", dtype=torch.int8, generator=g)
        else:
            B = torch.randn(K, N, device="cuda", generator=g).to(dt)
        for M in (1, 16, 64):
            if kind == "s8":
                A = torch.randint(-128, 128, (M, K), device="cuda", dtype=torch.int8,
                                  generator=g)
                alpha, beta = 1, 0
            else:
                A = torch.randn(M, K, device="cuda", generator=g).to(dt)
                alpha, beta = 1.0, 0.0
            C = torch.zeros(M, N, device="cuda", dtype=cdt)
            copies, t = time_skinny(binding, torch, kind, (A, B, C, alpha, beta), stream)
            nbytes = (A.numel() * A.element_size() + B.numel() * B.element_size()
                      + C.numel() * C.element_size())
            out[f"{kind}_M{M}"] = {"M": M, "N": N, "K": K, "ms": t * 1e3,
                                   "operand_copies": copies, "gbs": nbytes / t / 1e9,
                                   "frac_hbm": nbytes / t / 1e9 / hbm,
                                   "tflops": flops_of(M, N, K) / t / 1e12}
        del B
        torch.cuda.empty_cache()
    # Tall and narrow: matrix times vector (N = 1), and 16 columns for fp32 and
    # int8; A (M x K) streamed once. A 16-bit B keeps its row stride at 8 (the
    # tensor-map layout rule of the 16-bit entry points), one column used.
    M = 8192
    for kind, dt, cdt, widths in (("bf16", torch.bfloat16, torch.float32, (1,)),
                                  ("f32", torch.float32, torch.float32, (1, 16)),
                                  ("s8", torch.int8, torch.int32, (1, 16))):
        if kind == "s8":
            A = torch.randint(-128, 128, (M, K), device="cuda", dtype=torch.int8, generator=g)
            Bw = torch.randint(-128, 128, (K, 16), device="cuda", dtype=torch.int8, generator=g)
            alpha, beta = 1, 0
        else:
            A = torch.randn(M, K, device="cuda", generator=g).to(dt)
            Bw = torch.randn(K, 16 if kind == "f32" else 8, device="cuda", generator=g).to(dt)
            alpha, beta = 1.0, 0.0
        for n in widths:
            B = Bw[:, :n] if kind == "bf16" else Bw[:, :n].contiguous()
            C = torch.zeros(M, n, device="cuda", dtype=cdt)
            copies, t = time_skinny(binding, torch, kind, (A, B, C, alpha, beta), stream)
            nbytes = (A.numel() * A.element_size() + K * n * B.element_size()
                      + C.numel() * C.element_size())
            out[f"{kind}_N{n}"] = {"M": M, "N": n, "K": K, "ms": t * 1e3,
                                   "operand_copies": copies, "gbs": nbytes / t / 1e9,
                                   "frac_hbm": nbytes / t / 1e9 / hbm,
                                   "tflops": flops_of(M, n, K) / t / 1e12}
            del B, C
        del A, Bw
    torch.cuda.empty_cache()
    return out


def measure_types(binding, torch, peaks, stream):
    """The further entry points (uint8, 16-bit C, tf32, fp64) and the extended
    forms (transposed operands, strided batches), device-timed at one size
    each: TFLOP/s (TOPS for uint8) and the fraction of the pipe's peak. tf32's
    peak is the measured bf16 rate times the nominal tf32/bf16 ratio (1.1 /
    2.25 PFLOP/s dense); fp64's is the nominal 1.25 TFLOP/s (no measured fp64
    peak exists)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(4321)
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    out = {}

    def run(name, fn, args, steps, flops, peak, unit, note=None):
        with torch.cuda.stream(stream):
            for _ in range(2):
                fn(*args)
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            fn(*args)
        ev1.record(stream)
        torch.cuda.synchronize()
        t = ev0.elapsed_time(ev1) / steps / 1e3
        ach = flops / t / 1e12
        out[name] = {"ms": t * 1e3, "value": ach, "unit": unit, "peak": peak,
                     "frac": ach / peak}
        if note:
            out[name]["note"] = note

    S = 8192
    f = flops_of(S, S, S)
    A8 = torch.randint(0, 256, (S, S), device="cuda", dtype=torch.int32, generator=g).to(
        torch.uint8)
    B8 = torch.randint(0, 256, (S, S), device="cuda", dtype=torch.int32, generator=g).to(
        torch.uint8)
    C32 = torch.empty(S, S, device="cuda", dtype=torch.int32)
    run("u8_8192", binding.gemm_u8, (S, S, S, 1, A8, S, B8, S, 0, C32, S, stream), 20, f, bf16,
        "TOPS", "includes widening and the row/column offset sums")
    del A8, B8, C32
    for kind, dt, fn in (("f16_f16", torch.float16, binding.gemm_f16_f16),
                         ("bf16_bf16", torch.bfloat16, binding.gemm_bf16_bf16)):
        A = torch.randn(S, S, device="cuda", generator=g).to(dt)
        B = torch.randn(S, S, device="cuda", generator=g).to(dt)
        C = torch.empty(S, S, device="cuda", dtype=dt)
        run(f"{kind}_8192", fn, (S, S, S, 1.0, A, S, B, S, 0.0, C, S, stream), 20, f, bf16,
            "TFLOP/s")
        del A, B, C
    A = torch.randn(S, S, device="cuda", generator=g)
    B = torch.randn(S, S, device="cuda", generator=g)
    C = torch.empty(S, S, device="cuda")
    run("tf32_8192", binding.gemm_tf32, (S, S, S, 1.0, A, S, B, S, 0.0, C, S, stream), 20, f,
        bf16 * 1.1 / 2.25, "TFLOP/s", "includes the K-major copy of B")
    del A, B, C
    D = 2048
    A = torch.randn(D, D, device="cuda", generator=g, dtype=torch.float64)
    B = torch.randn(D, D, device="cuda", generator=g, dtype=torch.float64)
    C = torch.empty(D, D, device="cuda", dtype=torch.float64)
    run("f64_2048", binding.gemm_f64, (D, D, D, 1.0, A, D, B, D, 0.0, C, D, stream), 3,
        flops_of(D, D, D), 1.25, "TFLOP/s", "peak is the nominal fp64 rate")
    del A, B, C
    A = torch.randn(S, S, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(S, S, device="cuda", generator=g).to(torch.bfloat16)
    C = torch.empty(S, S, device="cuda")
    for ops in ("NT", "TN", "TT"):
        oa = binding.OP_T if ops[0] == "T" else binding.OP_N
        ob = binding.OP_T if ops[1] == "T" else binding.OP_N
        run(f"bf16_8192_{ops}", binding.gemm_bf16_ex,
            (oa, ob, S, S, S, 1.0, A, S, 0, B, S, 0, 0.0, C, S, 0, 1, stream), 20, f, bf16,
            "TFLOP/s")
    del A, B, C
    nb, E = 64, 1024
    A = torch.randn(nb, E, E, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(nb, E, E, device="cuda", generator=g).to(torch.bfloat16)
    C = torch.empty(nb, E, E, device="cuda")
    run("bf16_batched_64x1024", binding.gemm_bf16_ex,
        (binding.OP_N, binding.OP_N, E, E, E, 1.0, A, E, E * E, B, E, E * E, 0.0, C, E, E * E,
         nb, stream), 20, nb * flops_of(E, E, E), bf16, "TFLOP/s")
    # 137 GFLOP against 537 MB (A and B read once, fp32 C written once): the
    # problem sits at the roofline's ridge, and at the measured peaks the bytes
    # take longer than the flops. Its bound is the slower of the two.
    d = out["bf16_batched_64x1024"]
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    nbytes = nb * (2 * E * E * 2 + E * E * 4)
    t = d["ms"] / 1e3
    t_bound = max(nb * flops_of(E, E, E) / (bf16 * 1e12), nbytes / (hbm * 1e9))
    d["gbs"] = nbytes / t / 1e9
    d["frac_hbm"] = d["gbs"] / hbm
    d["roofline_bound"] = "hbm" if nbytes / (hbm * 1e9) >= t_bound else "tensor"
    d["frac_of_roofline"] = t_bound / t
    del A, B, C
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ compact summary

def compact_configs(name, head, extras, skinny, types):
    """One short entry per measured workload -- [value (TFLOP/s or TOPS),
    fraction of its pipe's peak, ms per call, median SM MHz, throttle reasons]
    -- plus the fraction of HBM bandwidth of each short, wide shape and the
    batched many-small fraction (of the tensor peak, and of its roofline bound:
    the slower of its flops at the tensor peak and its bytes at HBM speed)."""
    def entry(d):
        c = d.get("clocks") or {}
        mhz = c.get("sm_mhz")
        return [round(d["value"], 1), round(d["frac"], 3), round(d["ms_per_step"], 4),
                None if mhz is None else round(mhz), c.get("reasons", [])]
    out = {"key": "[value, frac_of_peak, ms, sm_mhz, reasons]", name: entry(head)}
    for k, d in extras.items():
        out[k] = entry(d)
    if skinny:
        out["skinny_frac_hbm"] = {k: round(d["frac_hbm"], 3) for k, d in skinny.items()}
    if "bf16_batched_64x1024" in types:
        d = types["bf16_batched_64x1024"]
        out["bf16_batched_64x1024_frac"] = round(d["frac"], 3)
        if "frac_of_roofline" in d:
            out["bf16_batched_64x1024_frac_of_roofline"] = [round(d["frac_of_roofline"], 3),
                                                           d["roofline_bound"]]
    return out


# ----------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="bf16_8192", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-skinny", action="store_true")
    ap.add_argument("--no-types", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    from dense_gemm_row_gb300 import binding
    from dense_gemm_row_gb300 import workloads as w

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist = tdist

    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(local_rank)
    sm_count = props.multi_processor_count
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        pass

    name = args.workload
    desc, kind, bound, launches_per_step = WORKLOADS[name]
    p = w.config(name)
    M, K = p.A.shape
    N = p.B.shape[1]
    p_dev = device_problem(torch, p)
    stream = torch.cuda.Stream()

    sampler = ClockSampler(gpu_id)
    sampler.start()
    ms, t0, t1 = time_device(binding, torch, kind, p_dev, args.steps, args.warmup, stream, dist)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    binding.check_device_error()

    flops = flops_of(M, N, K)
    ms_max, value = aggregate_ranks(torch, dist, ms, flops, args.steps, "cuda")
    step_ms = ms_max / args.steps

    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    unit = "TOPS" if kind == "s8" else "TFLOP/s"
    peak = peak_for(kind, peaks, sm_count)
    kernel_ms = ms / args.steps
    achieved = flops / (kernel_ms / 1e3) / 1e12
    traffic = recorded_traffic(name)
    roofline = {"bound": bound, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": (f"{peak_src}: " + ("SMs x 128 FP32 lanes x 2 x max SM clock "
                                                   f"({sm_count} SMs, {peaks.get('sm_max_mhz')} MHz)"
                                                   if kind == "f32" else "bf16_tflops (burst)")),
                "kernel": "gemm_tc_kernel" if kind != "f32" else "sgemm_simt_kernel",
                "kernel_ms": kernel_ms}
    if kind == "s8":
        roofline["note"] = "step time includes the two int8->fp16 widening launches"
    elif kind == "f32":
        roofline["note"] = ("step time includes the transposition of A (M x K -> K x M) that "
                            "lets the SIMT kernel copy A tiles in 16-byte chunks")
    if kind != "f32":
        # Context for a long timed loop: the measured sustained (power-capped)
        # peak, and the fraction of the dense rate at the clock sampled during
        # the timed region (152 x 8192 flop/clk for kind::f16 at that clock).
        sus = peak_for(kind, peaks, sm_count, sustained=True)
        roofline["frac_of_sustained_peak"] = achieved / sus
        roofline["sustained_peak"] = sus
        if clocks.get("sm_mhz"):
            roofline["frac_at_sampled_clock"] = achieved / (
                sm_count * 8192 * clocks["sm_mhz"] * 1e6 / 1e12)

    # End to end through the C ABI with pinned host buffers.
    Ah = p.A.pin_memory()
    Bh = p.B.pin_memory()
    Ch = torch.empty(p.C0.shape, dtype=p.C0.dtype).pin_memory()
    serial_ms, h2d, d2h = time_e2e(binding, torch, kind, (Ah, Bh, Ch), p_dev, args.e2e_steps,
                                   stream)
    e2e_ms = time_e2e_pipelined(binding, torch, kind, (Ah, Bh, Ch), p_dev, args.e2e_steps,
                                stream)
    e2e = {"value": flops * args.e2e_steps / (e2e_ms / 1e3) / 1e12, "unit": unit,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": e2e_ms / args.e2e_steps,
           "form": "3 steps in flight on 3 streams (copies of one step overlap another's GEMM)",
           "serial_ms_per_step": serial_ms / args.e2e_steps}

    extras = {}
    if not args.no_extras:
        for other in ("f32_4096", "f16_8192", "s8_8192", "bf16_8192", "f32_8192", "bf16_4096",
                      "s8_4096"):
            if other == name:
                continue
            extras[other] = measure_extra(binding, torch, w, other, peaks, sm_count, stream,
                                          gpu_id)
        binding.check_device_error()

    skinny = {}
    if not args.no_skinny:
        skinny = measure_skinny(binding, torch, peaks, stream)
    types = {}
    if not args.no_types:
        types = measure_types(binding, torch, peaks, stream)
        binding.check_device_error()

    micro = {}
    if not args.no_extras:
        micro = measure_peaks(binding, torch, peaks, sm_count, stream, gpu_id)
        roofline["microbench_peak"] = micro["ffma" if kind == "f32" else "tc_f16"]["tflops"]
        roofline["frac_of_microbench_peak"] = achieved / roofline["microbench_peak"]

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cal = cpu_oracle_sample(p, args.cpu_seconds)
        cpu = {"value": cal["flops"] / cal["seconds"] / 1e12, "unit": unit,
               "cores": cal["cores"], "kind": "oracle", "sample": cal["sample"],
               "seconds": cal["seconds"]}
        if not args.no_extras:
            cpu["configs"] = cpu_oracle_configs(w)

    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "f16": "f16", "f32": "f32", "s8": "s8"}[kind],
        "data": "synthetic (seeded; no dataset)",
        "config": {"workload": desc, "M": M, "N": N, "K": K,
                   "l2": "no flush: A+B exceed the 129 MB L2" if kind != "f32"
                   else "no flush: A+B+C = 192 MiB exceed the 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"],
                   "window": clocks["window"]},
        "extras": extras,
        "peaks_microbench": micro,
        "skinny": skinny,
        "types": types,
    }
    # Last, so that a reader keeping only the end of the line still has every
    # config's throughput, roofline fraction and clock record.
    line["configs"] = compact_configs(name, {"value": value, "ms_per_step": step_ms,
                                             "frac": achieved / peak,
                                             "clocks": clocks}, extras, skinny, types)
    print(json.dumps(line, separators=(",", ":")), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

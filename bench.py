"""Benchmark of the GEMM library on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-suite] [--no-cpu-baseline] [--no-cublas] [--no-e2e]

A step is one call of the library on the headline workload, by default the largest of the
configurations: fp16 inputs, fp32 accumulation and output, M = N = K = 8192, alpha = 1,
beta = 0 (uniform[-1,1] inputs rounded to fp16, seed 3; 1.1 TFLOP per call).  Inputs are
resident in HBM when the timed region starts; L2 is flushed (a 512 MB write) before every
timed step, so only the GEMM itself sits between each step's CUDA events.

Printed: ONE JSON line (rank 0) with the throughput (2*M*N*K / device time, TFLOP/s), the
roofline of the kernel, the CPU oracle timed on the host cores, the end-to-end number
through the public API with host buffers, the SM clocks seen during the timed region and,
under "suite", every configuration of the method (SGEMM 256^3 and its integer twin, the
ragged 1001 x 777 x 513 problem, the M = N sweep 128 ... 16384 with K = 1024, 4096^3; HGEMM
2048^3, 4096^3, 8192^3 and the integer 2048 x 2048 x 1024 twin; the linear-layer problem
16384 x 4096 x 4096 with op(B) = T and beta = 1), each timed the same way: min, median and
max device time, TFLOP/s, fraction of the roofline, achieved HBM bandwidth (compulsory
bytes / median time), launches per call, the clocks sampled while it ran, cuBLAS through
torch as a side column and, for the two small SGEMM configurations, the oracle's time on
one core and on all cores.

--impl reference times the CPU oracle (the only reference implementation of this path)
on the same workload, on rank 0 only, as bounded row-slab samples.

Multi-GPU: the path has no exchange step, so N GPUs run N independent replicas of the
same step (weak scaling); value = all replicas' flops / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS (2MNK/device time) FP32 & fp16→fp32, % of GB300 roofline"
UNIT = "TFLOPS"
# The pages' own best hand-written kernel on this exact workload (yekq.top "LeetGPU 第二题",
# results table, v4 2-D register coarsening on an RTX 4090): 13848.77 GFLOPS.  Context only.
PAGES_RAGGED_GFLOPS = 13848.77
# FP32 FFMA roofline: 152 SMs x 128 FP32 lanes x 2 flop (fused multiply-add) x 2.07 GHz.
SMS, FP32_LANES, SM_MAX_GHZ = 152, 128, 2.070
FFMA_PEAK_TFLOPS = SMS * FP32_LANES * 2 * SM_MAX_GHZ / 1e3
L2_FLUSH_BYTES = 512 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------------ clocks during the run
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []  # (monotonic time of arrival, csv line)
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let the first sample arrive before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def summary(self, t0=None, t1=None):
        """Median SM clock, maximum clock, throttle reasons seen and peak power of the samples
        that arrived in [t0, t1] (all samples when no window is given)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, power = [], [], set(), []
        for t, ln in list(self.samples):
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(self.REASONS, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}

    def stop(self):
        if self.proc is None:
            return self.summary()
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        return self.summary()


# ------------------------------------------------------------------ helpers
def whole_job_value(local_total_ms, steps, flops_per_step, world, device=None):
    """Whole-job TFLOP/s of `world` replicas: every rank did `steps` steps of
    `flops_per_step`; the job took as long as its slowest rank (max over ranks)."""
    total_ms = float(local_total_ms)
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return world * steps * flops_per_step / (total_ms * 1e-3) / 1e12, total_ms


# The CUDA sources each profiled kernel is built from (its launch planning included).
KERNEL_SOURCES = {
    "sgemm_ffma": ("sgemm_*", "gemm_internal.h"),
    "hgemm_tcgen05": ("hgemm_tcgen05.cu", "gemm_internal.h"),
}


def csrc_digest(kernel: str) -> str:
    """First 16 hex digits of a sha256 over the CUDA sources of one kernel (file names and
    contents, in name order)."""
    import glob

    paths = set()
    for pattern in KERNEL_SOURCES[kernel]:
        paths.update(glob.glob(os.path.join(ROOT, "dense_gemm_sgemm_gb300", "csrc", pattern)))
    h = hashlib.sha256()
    for path in sorted(paths):
        h.update(os.path.basename(path).encode())
        h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def _profile_fields(kernel: str, profile: str):
    """Fields of a committed ncu summary, if the kernel's sources are unchanged since the
    capture (else None)."""
    path = os.path.join(ROOT, "profiles", profile)
    try:
        digest = csrc_digest(kernel)
        fields = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        return fields if fields.get("source_sha256_16") == digest else None
    except Exception:
        return None


def _traffic_from_profile(kernel: str, profile: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's sources are
    unchanged since the capture."""
    fields = _profile_fields(kernel, profile)
    try:
        return float(fields["dram_bytes_per_launch"]) if fields else None
    except (KeyError, ValueError):
        return None


def _ncu_duration_us(kernel: str, profile: str):
    """The kernel's duration under ncu (one launch, cold L2, serialised) from the same summary."""
    fields = _profile_fields(kernel, profile)
    try:
        return float(fields["duration_us"]) if fields else None
    except (KeyError, ValueError):
        return None


def _gemm_fn(w):
    from dense_gemm_sgemm_gb300 import gemm_hgemm_f16f32, gemm_sgemm_f32

    return gemm_sgemm_f32 if w.dtype == "f32" else gemm_hgemm_f16f32


def _device_inputs(w):
    from dense_gemm_sgemm_gb300 import workloads

    host = workloads.make_inputs(w)
    return host, {k: v.cuda() for k, v in host.items()}


def time_device(w, dev, steps, warmup, flush, barrier=None):
    """Per-step CUDA-event times (ms) of the library call, L2 flushed before each step; also
    the wall time and the number of library kernels launched in the timed region."""
    import torch

    from dense_gemm_sgemm_gb300 import gemm_kernel_launches

    fn = _gemm_fn(w)
    stream = torch.cuda.current_stream()

    def call():
        fn(w.opA, w.opB, w.M, w.N, w.K, w.alpha, dev["A"], w.lda, dev["B"], w.ldb, w.beta,
           dev["C"], w.ldc, stream)

    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    launches0 = gemm_kernel_launches()
    wall0 = time.perf_counter()
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        call()
        e.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches = gemm_kernel_launches() - launches0
    if barrier:
        barrier()
    return [s.elapsed_time(e) for s, e in ev], wall, launches


def time_e2e(w, host, steps, sets=3):
    """End to end through the public host-memory entry point (gemm_*_host): each step is one
    call on page-locked host buffers that copies the step's A, B and C_in to the device,
    runs the GEMM and copies C back, in order on the call's stream.  Steps rotate over
    three streams, each with its own host buffers (and, inside the library, its own device
    staging area), the way a caller streaming independent GEMMs would run them: the copies
    of one step overlap the GEMMs of its neighbours."""
    import torch

    from dense_gemm_sgemm_gb300 import (gemm_bgemm_bf16f32_host, gemm_hgemm_f16f32_host,
                                        gemm_sgemm_f32_host)

    fn = {"f32": gemm_sgemm_f32_host, "f16": gemm_hgemm_f16f32_host,
          "bf16": gemm_bgemm_bf16f32_host}[w.dtype]
    pinned = [{k: v.pin_memory() for k, v in host.items()} for _ in range(sets)]
    streams = [torch.cuda.Stream() for _ in range(sets)]
    names = ["A", "B"] + (["C"] if w.beta != 0.0 else [])
    h2d = sum(pinned[0][k].numel() * pinned[0][k].element_size() for k in names)
    d2h = w.M * w.N * 4

    def step(i):
        b = pinned[i % sets]
        fn(w.opA, w.opB, w.M, w.N, w.K, w.alpha, b["A"], w.lda, b["B"], w.ldb, w.beta, b["C"],
           w.ldc, streams[i % sets])

    for i in range(2 * sets):  # allocates each stream's staging area
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(streams[0])
    for s in streams[1:]:
        s.wait_event(t0)
    for i in range(steps):
        step(i)
    for s in streams[1:]:
        streams[0].wait_stream(s)
    t1.record(streams[0])
    t1.synchronize()
    ms = t0.elapsed_time(t1) / steps
    return {"value": round(w.flops / (ms * 1e-3) / 1e12, 4), "unit": UNIT,
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "api": f"{fn.__name__} on page-locked host buffers",
            "pipelined": f"{sets} streams round-robin, each with its own host buffers"}


def oracle_sample(w, host, budget_s):
    """Time the CPU oracle on a row slab of w sized to about budget_s seconds."""
    import numpy as np

    import oracle

    A = host["A"].numpy()
    B = host["B"].numpy()
    if w.dtype == "f16":
        A, B = A.view(np.uint16), B.view(np.uint16)
    C = host["C"].numpy()
    threads = oracle.default_threads()

    def run(rows):
        # rows of op(A) = N are contiguous rows of A; op(A) = T keeps every column block
        if w.opA == "N":
            a = A[:rows]
        else:
            a = A  # the oracle reads only the first `rows` columns through lda
        t0 = time.perf_counter()
        oracle.gemm(w.opA, w.opB, rows, w.N, w.K, w.alpha, a, w.lda, B, w.ldb, w.beta,
                    C[:rows] if w.beta != 0.0 else None, w.ldc, dtype=w.dtype, threads=threads)
        return time.perf_counter() - t0

    probe = max(1, min(w.M, threads))
    t = run(probe)
    per_row = max(t / probe, 1e-7)
    rows = int(max(probe, min(w.M, budget_s / per_row)))
    return rows, threads, run


# ------------------------------------------------------------------ the two arms
def run_reference(args, rank, world):
    from dense_gemm_sgemm_gb300 import workloads

    if rank != 0:
        return 0
    w = workloads.by_name(args.workload)
    host = workloads.make_inputs(w)
    per_step_budget = max(0.01, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    rows, threads, run = oracle_sample(w, host, per_step_budget)
    for _ in range(args.warmup):
        run(rows)
    times = [run(rows) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    flops = 2 * rows * w.N * w.K
    val = flops / (ms * 1e-3) / 1e12
    sample = f"rows 0..{rows - 1} of op(A) (of {w.M}) x full B, per step; fp64 oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                   "beta": w.beta, "opA": w.opA, "opB": w.opB, "seed": w.seed},
        "cpu_baseline": {"value": round(val, 6), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _roofline_peak(w, peaks):
    """Compute peak of the path (TFLOP/s), its kind and source, and the roofline of this
    problem: the lesser of the compute peak and intensity x measured HBM bandwidth."""
    if w.dtype == "f32":
        peak, bound, src = FFMA_PEAK_TFLOPS, "alu", "152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz"
    else:
        peak, bound = peaks["bf16_tflops"], "tensor"
        src = f"bf16 dense burst ({peaks['source']}); fp16 has the same nominal rate"
    hbm_roof = w.flops / w.algorithmic_bytes * peaks["hbm_gbs"] / 1e3
    return peak, bound, src, min(peak, hbm_roof)


def run_ours(args, rank, world, local):
    import torch

    import dense_gemm_sgemm_gb300 as lib
    from dense_gemm_sgemm_gb300 import workloads

    lib.load()  # fails loudly when the CUDA library is missing
    torch.cuda.set_device(local)
    barrier = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = dist.barrier
    peaks = _peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    w = workloads.by_name(args.workload)
    host, dev = _device_inputs(w)
    clocks = ClockSampler(local)
    clocks.start()
    t0 = time.monotonic()
    step_ms, wall, launches = time_device(w, dev, args.steps, args.warmup, flush, barrier)
    clk = clocks.summary(t0, time.monotonic())
    status = lib.gemm_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {lib.gemm_status_string(status)}")
    value, total_ms = whole_job_value(sum(step_ms), args.steps, w.flops, world,
                                      torch.device("cuda", local))
    mean_ms = statistics.fmean(step_ms)
    achieved = w.flops / (mean_ms * 1e-3) / 1e12
    kernel = "sgemm_ffma" if w.dtype == "f32" else "hgemm_tcgen05"
    peak, bound, peak_src, roof = _roofline_peak(w, peaks)
    traffic = _traffic_from_profile(kernel, f"{kernel}_{w.name}.txt")
    ncu_us = _ncu_duration_us(kernel, f"{kernel}_{w.name}.txt")
    # The library's own FFMA-chain probe, run after the timed region: a measured FP32
    # multiply-add ceiling beside the one derived from unit counts and the maximum clock.
    probe = round(lib.gemm_measure_fp32_fma_peak(), 2) if w.dtype == "f32" else None
    vs = (round(value / (PAGES_RAGGED_GFLOPS / 1e3), 4)
          if w.name == workloads.sgemm_ragged().name else None)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": vs,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                   "beta": w.beta, "opA": w.opA, "opB": w.opB, "seed": w.seed,
                   "dist": f"A {w.dist_a}, B {w.dist_b}" + (f", C {w.dist_c}" if w.beta else ""),
                   "l2": "flushed before every timed step (512 MB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": bound, "achieved": round(achieved, 4),
                     "peak": round(peak, 2), "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": w.algorithmic_bytes, "peak_source": peak_src,
                     "roof": round(roof, 2), "frac_of_roof": round(achieved / roof, 4),
                     "frac_of_sustained": (round(achieved / peaks["bf16_tflops_sustained"], 4)
                                           if w.dtype != "f32" else None),
                     "peak_fma_probe": probe,
                     # kernel-only time from the ncu summary (cold L2, no event overhead)
                     "ncu_kernel_us": ncu_us,
                     "frac_kernel_only": (round(w.flops / (ncu_us * 1e-6) / 1e12 / peak, 4)
                                          if ncu_us else None),
                     "median_ms": round(statistics.median(step_ms), 5),
                     "min_ms": round(min(step_ms), 5), "max_ms": round(max(step_ms), 5)},
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
    }
    if not args.no_e2e:
        line["e2e"] = time_e2e(w, host, max(3, min(args.steps, 200)))
    del host, dev
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_suite:
        line["suite"] = run_suite(peaks, flush, clocks, cublas=not args.no_cublas,
                                  oracle_times=not args.no_cpu_baseline)
    clocks.stop()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = workloads.make_inputs(w)
        rows, threads, run = oracle_sample(w, host, 1.0)
        reps = max(1, int(10.0 / max(run(rows), 1e-3)))
        times = [run(rows) for _ in range(reps)]
        cpu = 2 * rows * w.N * w.K / statistics.median(times) / 1e12
        line["cpu_baseline"] = {"value": round(cpu, 6), "unit": UNIT, "cores": threads,
                                "kind": "oracle",
                                "sample": f"rows 0..{rows - 1} of {w.M} (x full B), "
                                          f"{reps} repetitions, median"}
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# Every configuration of the method; the pages' own figure where one exists for that exact
# problem (their hardware, context only).
def suite_workloads():
    from dense_gemm_sgemm_gb300 import workloads

    out = [workloads.sgemm_256(), workloads.sgemm_256(integer=True), workloads.sgemm_ragged()]
    out += [workloads.sgemm_sweep(mn) for mn in workloads.SWEEP_MN]
    out += [workloads.sgemm_cube(4096)]
    out += [workloads.hgemm_square(n) for n in workloads.HGEMM_SQUARE]
    out += [workloads.hgemm_square(2048, integer=True, K=1024), workloads.linear_fp16()]
    return out


PAGES_CONTEXT = {
    "sgemm_ragged_1001x777x513": "13.85 TFLOP/s, v4 2-D register coarsening, RTX 4090 (yekq.top)",
    "sgemm_sweep_16384x16384x1024": "12.66 TFLOP/s, V3 double buffer, V100 (ssxxe.cn)",
    "hgemm_4096x4096x4096": "103.10 TFLOP/s, WMMA v7, RTX 5080 (dandandamowang.xyz)",
}


def _cublas_call(w, dev):
    """torch.matmul on the same operands (cuBLAS; TF32 off for fp32).  Its fp16 GEMM writes
    fp16 and ignores alpha, beta and C_in: a side reference, not the same output."""
    import torch

    A = dev["A"][:, : w.a_shape[1]]
    B = dev["B"][:, : w.b_shape[1]]
    a = A if w.opA == "N" else A.t()
    b = B if w.opB == "N" else B.t()
    return lambda: torch.matmul(a, b)


def _time_fn(fn, reps, warmup, flush):
    import torch

    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in ev]


def run_suite(peaks, flush, clocks, cublas=True, oracle_times=True):
    """Every configuration, timed like the headline step (L2 flushed before each timed call):
    at least 30 calls and about 0.2 s of calls per configuration."""
    import torch

    torch.backends.cuda.matmul.allow_tf32 = False
    out = []
    for w in suite_workloads():
        host, dev = _device_inputs(w)
        probe_ms, _, _ = time_device(w, dev, 3, 3, flush)
        reps = int(min(400, max(30, 0.2 / (statistics.median(probe_ms) * 1e-3 + 1e-4))))
        t0 = time.monotonic()
        ms, _, launches = time_device(w, dev, reps, 5, flush)
        clk = clocks.summary(t0, time.monotonic())
        med = statistics.median(ms)
        tf = w.flops / (med * 1e-3) / 1e12
        peak, bound, src, roof = _roofline_peak(w, peaks)
        entry = {"workload": w.name, "dtype": w.dtype, "M": w.M, "N": w.N, "K": w.K,
                 "opA": w.opA, "opB": w.opB, "alpha": w.alpha, "beta": w.beta, "reps": reps,
                 "min_us": round(min(ms) * 1e3, 2), "median_us": round(med * 1e3, 2),
                 "max_us": round(max(ms) * 1e3, 2), "tflops": round(tf, 3),
                 "bound": bound, "peak": round(peak, 1), "frac": round(tf / peak, 4),
                 "roof": round(roof, 1), "frac_of_roof": round(tf / roof, 4),
                 "hbm_gbs": round(w.algorithmic_bytes / (med * 1e-3) / 1e9, 1),
                 "hbm_frac": round(w.algorithmic_bytes / (med * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                 "algorithmic_bytes": w.algorithmic_bytes,
                 "launches_per_call": launches / reps, "clocks": clk, "peak_source": src}
        if w.name in PAGES_CONTEXT:
            entry["pages"] = PAGES_CONTEXT[w.name]
        if cublas:
            cms = _time_fn(_cublas_call(w, dev), min(reps, 100), 5, flush)
            entry["cublas_tflops"] = round(w.flops / (statistics.median(cms) * 1e-3) / 1e12, 3)
            entry["cublas_note"] = ("torch.matmul, TF32 off" if w.dtype == "f32"
                                    else "torch.matmul, fp16 output, no alpha/beta")
        if oracle_times and w.name.startswith(("sgemm_256cube", "sgemm_ragged")):
            import oracle

            for key, threads in (("oracle_1core_s", 1), ("oracle_all_cores_s", oracle.default_threads())):
                t = time.perf_counter()
                oracle.gemm(w.opA, w.opB, w.M, w.N, w.K, w.alpha, host["A"].numpy(), w.lda,
                            host["B"].numpy(), w.ldb, w.beta,
                            host["C"].numpy() if w.beta != 0.0 else None, w.ldc, threads=threads)
                entry[key] = round(time.perf_counter() - t, 4)
            entry["oracle_cores"] = oracle.default_threads()
        out.append(entry)
        del host, dev
        torch.cuda.empty_cache()
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="hgemm_8192x8192x8192",
                    help="workload of the timed step (names in dense_gemm_sgemm_gb300.workloads)")
    ap.add_argument("--no-suite", action="store_true", help="skip the per-configuration suite")
    ap.add_argument("--no-cublas", action="store_true", help="skip the cuBLAS side column")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the oracle")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg through the host-memory entry point")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = _dist()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())

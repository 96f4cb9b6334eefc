"""Benchmark of the fused GEMM + scale + ReLU library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gsr|reference]

One step = one call of gemm_scale_relu on the whole workload (A, B resident in HBM).
Metric: TFLOP/s = 2*M*N*K / time, device-timed with CUDA events on the launching stream,
as the tutorial's benchmark_op does ("Tutorial14: 使用TileLang语言编写attention算子",
section 2: warm-up calls, CUDA events around back-to-back calls, 2*M*N*K / latency).

Prints ONE JSON line (rank 0).  Besides the timing it carries:
  roofline      the kernel's achieved TFLOP/s (or GB/s for the HBM-bound small-M shape)
                against the measured peak in MEASURED_PEAKS.json, with the DRAM traffic
                per launch from the committed ncu summary when it matches the current
                kernel sources;
  e2e           the same metric through gemm_scale_relu_host: pinned host A, B copied in
                and C copied out inside the timed region, every step;
  cpu_baseline  the fp64 CPU oracle timed on this host on a bounded sample of rows;
  clocks        SM clocks and throttle reasons sampled by nvidia-smi during the timed region
                (and, under median5_window, during the longer repeats that follow it);
  median5       the median over 5 repeats of >= 100 back-to-back calls after the timed region;
  per_config    the other four GEMM configurations, each timed the same way in the same run,
                with its own roofline and CPU-oracle time.
With --impl reference the line times the oracle itself (the CPU reference arm).
N > 1 (torchrun): every rank runs its own full copy of the workload (replicas, weak
scaling); the time is the max over ranks and the value the sum of all ranks' work.
"""
from __future__ import annotations

import argparse
import re
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

from tensor_core_gemm_multistage_gb300.workloads import (ATTN_WORKLOADS, WORKLOADS,  # noqa: E402
                                                          workload_inputs)

METRIC = "fused GEMM+scale+ReLU TFLOP/s and % of GB300 dense FP16 peak, 1 GPU"
DEFAULT_WORKLOAD = "llm_mlp_up"
L2_BYTES = 126 * 1024 * 1024
# The sources each kernel is built from: a DRAM-traffic figure stays valid while they do.
_SHARED_SOURCES = ["csrc/ptx.cuh", "csrc/device_common.cuh", "csrc/kernels.h"]
KERNEL_SOURCES = {
    "gsr_tiled_kernel": ["csrc/gemm_tiled.cu"] + _SHARED_SOURCES,
    "gsr_pair_kernel": ["csrc/gemm_pair.cu"] + _SHARED_SOURCES,
    "gsr_skinny_kernel": ["csrc/gemm_skinny.cu"] + _SHARED_SOURCES,
    "gsr_attention_kernel": ["csrc/attention_fwd.cu", "csrc/attention.h"] + _SHARED_SOURCES,
}
KERNEL_NAMES = {0: "gsr_tiled_kernel", 1: "gsr_skinny_kernel", 2: "gsr_pair_kernel", 3: "gsr_pair_kernel"}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


# ---------------------------------------------------------------------------- helpers

def _code_only(text: str) -> str:
    """C/CUDA source without comments and blank space, so that a comment edit keeps a hash."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "tensor_core_gemm_multistage_gb300")
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(pkg, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def read_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel sources; lines: `workload kernel sources_hash bytes_per_launch note...`."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    cur = kernel_source_hash(kernel)
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload \
                    and parts[1] == kernel and parts[2] == cur:
                return float(parts[3])
    return None


def tensor_peak_key(region_ms: float) -> str:
    """Which measured tensor peak a timed region compares with: a back-to-back loop of half a
    second or more runs under the power cap like the sustained cuBLAS loop (seconds long);
    a shorter one like the burst figure."""
    return "bf16_tflops_sustained" if region_ms >= 500.0 else "bf16_tflops"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int) -> float:
    """Max of a float over all ranks (identity at world size 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank: float, max_ms: float) -> float:
    """Replica mode: every rank runs the whole workload, so the job does world x the work in
    the slowest rank's time."""
    return world * flops_per_rank / (max_ms * 1e-3) / 1e12


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, timestamped on arrival."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid: str | None, interval_ms: int = 100):
        self.uuid = uuid
        self.samples = []
        self.proc = None
        self.interval_ms = interval_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        threading.Thread(target=self._read, daemon=True).start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append((time.time(), float(parts[1]), float(parts[2]), parts[4:9],
                                     parts[0]))
            except ValueError:
                pass

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        mine = [s for s in self.samples if s[4] == self.uuid]
        if not mine and self.samples:    # uuid not reported: the first GPU listed
            first = self.samples[0][4]
            mine = [s for s in self.samples if s[4] == first]
        self.samples = mine
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside:   # region shorter than the sampling interval: nearest samples under load
            inside = [s for s in self.samples if t0 - 1.0 <= s[0] <= t1 + 0.5]
            window = "around the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no samples"}
        reasons = set()
        for s in inside:
            flags = s[3]
            for name, flag in zip(self.REASONS, flags[1:5]):
                if flag.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


def gpu_uuid():
    try:
        import torch
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


# ---------------------------------------------------------------------------- CPU oracle

def time_oracle(A, B, alpha, seconds: float):
    """Run the oracle on chunks of whole rows of C (one row per host thread per chunk)
    until about `seconds` have passed; returns (rows done, elapsed s, threads used)."""
    import oracle
    oracle.build()
    M = A.shape[0]
    threads = oracle.max_threads()
    chunk = min(M, threads)
    done, t_total, row = 0, 0.0, 0
    while done == 0 or t_total < seconds:          # at least one chunk
        rows = [(row + i) % M for i in range(chunk)]
        t = time.perf_counter()
        oracle.gemm_scale_relu(A, B, alpha, rows=rows)
        t_total += time.perf_counter() - t
        done += chunk
        row = (row + chunk) % M
    return done, t_total, chunk


# ---------------------------------------------------------------------------- arms

def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401
    import oracle
    oracle.build()
    A, B = workload_inputs(w)
    # calibrate with one chunk (one row per host thread), then size each step as a whole
    # number of chunks so that the --warmup + --steps run stays within about two minutes
    threads = oracle.max_threads()
    chunk = min(w.M, threads)
    t = time.perf_counter()
    oracle.gemm_scale_relu(A, B, w.alpha, rows=list(range(chunk)))
    per_chunk = max(time.perf_counter() - t, 1e-6)
    budget = 120.0
    chunks = max(1, int(budget / ((args.steps + args.warmup) * per_chunk)))
    rows_per_step = min(w.M, chunks * chunk)
    row = 0
    for _ in range(args.warmup):
        oracle.gemm_scale_relu(A, B, w.alpha, rows=[(row + i) % w.M for i in range(rows_per_step)])
        row += rows_per_step
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_scale_relu(A, B, w.alpha, rows=[(row + i) % w.M for i in range(rows_per_step)])
        row += rows_per_step
    elapsed = time.perf_counter() - t0
    flops = 2.0 * rows_per_step * w.N * w.K * args.steps
    value = flops / elapsed / 1e12
    sample = "%d of %d output rows (whole rows of C) per step" % (rows_per_step, w.M)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded randn, fp16)",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": min(threads, rows_per_step),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, epilogue="scale_relu"):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
            "epilogue": epilogue,
            "inputs": "A,B fp16 from seeded randn" + (", B*K^-1/2" if w.b_std_inv_sqrt_k else ""),
            "accumulate": "f32", "output": "f16",
            "l2": ("inputs larger than L2 (A+B %d MiB > 126 MiB), no flush"
                   % ((w.M * w.K + w.K * w.N) * 2 >> 20))
            if (w.M * w.K + w.K * w.N) * 2 > L2_BYTES else "flush L2 between steps"}


def host_cpu_model() -> str:
    """Model name of the host CPU (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def run_block(step, calls: int, stream, flush) -> float:
    """Mean time of one call over `calls` back-to-back calls, CUDA events on the launching
    stream: around the whole run, or around each call when L2 is flushed between calls."""
    import torch
    if flush is None:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(calls):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / calls
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(calls)]
    for i in range(calls):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(x.elapsed_time(y) for x, y in ev) / calls


def gemm_roofline(w, path, kernel, kernel_ms, region_ms, peaks, peaks_src):
    """Roofline object of one GEMM workload: HBM bytes for the small-M kernel, tensor flops
    otherwise, against the measured peak; DRAM traffic from the committed ncu summary."""
    if path == 1:
        achieved = w.bytes / (kernel_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        r = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
             "frac": achieved / peak, "kernel": kernel,
             "per_launch": "%d algorithmic bytes (A+B read once, C written once)" % w.bytes}
        key = "hbm_gbs"
    else:
        achieved = w.flops / (kernel_ms * 1e-3) / 1e12
        key = tensor_peak_key(region_ms)
        peak = float(peaks[key])
        r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
             "frac": achieved / peak, "kernel": kernel,
             "per_launch": "%d algorithmic flops (2*M*N*K)" % w.flops,
             "frac_of_burst": achieved / float(peaks["bf16_tflops"])}
    r["traffic"] = read_traffic(w.name, kernel)
    r["peak_source"] = "%s: %s%s" % (peaks_src, key, "" if path == 1 else
                                     "; fp16 dense rate taken equal to the bf16 rate (nominal ratio 1)")
    return r


def time_gemm(gsr, w, args, dev, stream, world, epilogue="scale_relu"):
    """Warm-up, then exactly args.steps calls timed with CUDA events on the launching stream
    (per call and around the whole region), between barriers and synchronisations.  Inputs
    that fit in L2 are evicted before every call by a 256 MiB write outside the call's events.
    Returns the timing record and the device inputs (for the e2e leg)."""
    import torch

    A, B = workload_inputs(w)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.empty(w.M, w.N, dtype=torch.float16, device=dev)
    inputs_bytes = (w.M * w.K + w.K * w.N) * 2
    flush = None
    if inputs_bytes <= L2_BYTES:
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    if epilogue == "bias_gelu":
        from tensor_core_gemm_multistage_gb300.workloads import make_bias
        dbias = make_bias(w.N, seed=1).to(dev)

        def step():
            gsr.gemm_bias_gelu(dA, dB, dbias, dC, stream=stream)
    elif epilogue == "scale":
        def step():
            gsr.gemm_scale(dA, dB, dC, w.alpha, stream=stream)
    else:
        def step():
            gsr.gemm_scale_relu(dA, dB, dC, w.alpha, stream=stream)

    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    torch.cuda.synchronize()
    status, code = gsr.device_status(stream)
    if status != gsr.Status.OK:
        raise RuntimeError("%s: device status %s code %#x" % (w.name, status.name, code))
    kernel_ms = [a.elapsed_time(b) for a, b in ev]
    region_ms = start.elapsed_time(stop)
    step_ms = region_ms / args.steps if flush is None else sum(kernel_ms) / args.steps
    med, wall_repeats = None, None
    if args.repeats > 0:
        # After the timed region: `repeats` more runs of max(100, steps) back-to-back calls
        # each, timed the same way; the median of their mean call times.
        tr0 = time.time()
        reps = [run_block(step, max(100, args.steps), stream, flush) for _ in range(args.repeats)]
        wall_repeats = (tr0, time.time())
        med = statistics.median(reps)
    warm = None
    if flush is not None and args.repeats > 0:
        # Context for the flushed workloads: the page's own way of timing them, back-to-back
        # calls with the operands left in L2 (median of the same repeats, no flush)
        warm = statistics.median(run_block(step, max(100, args.steps), stream, None)
                                 for _ in range(args.repeats))
    rec = {
        "step_ms": max_over_ranks(step_ms, world),
        "kernel_ms": max_over_ranks(sum(kernel_ms) / len(kernel_ms), world),
        "median5_ms": max_over_ranks(med, world) if med is not None else None,
        "region_ms": region_ms, "wall": (t_wall0, t_wall1), "wall_repeats": wall_repeats,
        "warm_ms": max_over_ranks(warm, world) if warm is not None else None,
        "l2": ("inputs larger than L2 (A+B %d MiB > 126 MiB), no flush" % (inputs_bytes >> 20))
        if flush is None else "flush L2 between steps (256 MiB write outside each call's events)",
    }
    return rec, (A, B, dA, dB, dC, flush, step)


def oracle_baseline(A, B, w, seconds: float):
    """The CPU oracle on one configuration: all of C when that fits in about `seconds` (the
    per-row time measured on one chunk of rows first), else whole rows until `seconds` have
    passed, with the full time extrapolated from the per-row time (and labelled so)."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    chunk = min(w.M, threads)
    t = time.perf_counter()
    oracle.gemm_scale_relu(A, B, w.alpha, rows=list(range(chunk)))
    per_row = max(time.perf_counter() - t, 1e-9) / chunk
    if per_row * w.M <= seconds:
        t = time.perf_counter()
        oracle.gemm_scale_relu(A, B, w.alpha)
        secs = time.perf_counter() - t
        return {"value": w.flops / secs / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": "all %d rows of C, %.2f s" % (w.M, secs), "per_row_ms": secs / w.M * 1e3,
                "full_s": secs}
    rows, secs, cores = time_oracle(A, B, w.alpha, seconds)
    return {"value": 2.0 * rows * w.N * w.K / secs / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "sample": "%d whole rows of C (of %d), %.1f s" % (rows, w.M, secs),
            "per_row_ms": secs / rows * 1e3, "extrapolated_full_s": secs / rows * w.M,
            "extrapolated_note": "extrapolated: measured per-row time x M rows, not a full run"}


def per_config_entry(w, rec, path, kernel, peaks, peaks_src, world):
    value = whole_job_tflops(world, w.flops, rec["step_ms"])
    e = {"M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha, "kernel": kernel,
         "ms_per_step": rec["step_ms"], "kernel_ms": rec["kernel_ms"], "TFLOP/s": value,
         "median5_ms": rec["median5_ms"],
         "median5_TFLOP/s": (whole_job_tflops(world, w.flops, rec["median5_ms"])
                             if rec["median5_ms"] else None),
         "l2": rec["l2"],
         "roofline": gemm_roofline(w, path, kernel, rec["kernel_ms"], rec["region_ms"], peaks,
                                   peaks_src)}
    if path == 1:
        e["GB/s"] = w.bytes / (rec["kernel_ms"] * 1e-3) / 1e9
    if rec.get("warm_ms"):
        e["l2_warm"] = {"ms_per_step": rec["warm_ms"],
                        "TFLOP/s": whole_job_tflops(world, w.flops, rec["warm_ms"]),
                        "how": "context: back-to-back calls with A and B left in L2 (no flush), median "
                               "of the repeats of >= 100 calls"}
    return e


def run_gsr(args, w):
    import torch

    import tensor_core_gemm_multistage_gb300 as gsr

    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gsr.build()
    stream = torch.cuda.current_stream(dev)
    path = gsr.select_path(w.M, w.N, w.K)
    kernel = KERNEL_NAMES[path]
    peaks, peaks_src = measured_peaks()

    sampler = ClockSampler(gpu_uuid(), interval_ms=5).start() if rank == 0 else None
    rec, (A, B, dA, dB, dC, flush, step) = time_gemm(gsr, w, args, dev, stream, world, args.epilogue)
    t_wall0, t_wall1 = rec["wall"]
    inputs_bytes = (w.M * w.K + w.K * w.N) * 2

    # end-to-end through the host entry point: pinned host in, pinned host out
    e2e = None
    if args.e2e_steps > 0 and args.epilogue == "scale_relu":
        hA, hB = A.pin_memory(), B.pin_memory()
        hC = torch.empty(w.M, w.N, dtype=torch.float16).pin_memory()
        gsr.gemm_scale_relu_host(hA, hB, hC, dA, dB, dC, w.alpha, stream=stream)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            gsr.gemm_scale_relu_host(hA, hB, hC, dA, dB, dC, w.alpha, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world)
        e2e = {"value": whole_job_tflops(world, w.flops, e2e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": inputs_bytes, "d2h_bytes_per_step": w.M * w.N * 2,
               "ms_per_step": e2e_ms, "steps": args.e2e_steps}
        del hA, hB, hC

    # Context only (the tutorial compares its fused kernel with unfused PyTorch): the same
    # workload as torch.relu((A @ B) * alpha) and as a plain cuBLAS fp16 matmul.
    context = None
    if args.torch_context:
        context = {}
        for label, fn in (("torch_unfused_relu_matmul_scale", lambda: torch.relu((dA @ dB) * w.alpha)),
                          ("cublas_matmul_only", lambda: torch.matmul(dA, dB, out=dC))):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for i in range(args.steps):
                if flush is not None:
                    flush.zero_()
                evs[i][0].record(stream)
                fn()
                evs[i][1].record(stream)
            c1.record(stream)
            torch.cuda.synchronize()
            ms = (c0.elapsed_time(c1) / args.steps if flush is None
                  else sum(a.elapsed_time(b) for a, b in evs) / args.steps)
            context[label] = {"ms_per_step": ms, "TFLOP/s": w.flops / (ms * 1e-3) / 1e12}
    del dA, dB, dC, flush, step

    # The other configurations, measured the same way in the same process (same steps and
    # warm-up): each is its own JSON object under "per_config".
    per_config = {}
    if args.per_config and args.epilogue == "scale_relu":
        for name, ow in WORKLOADS.items():
            if name == w.name:
                continue
            opath = gsr.select_path(ow.M, ow.N, ow.K)
            orec, bufs = time_gemm(gsr, ow, args, dev, stream, world)
            oA, oB = bufs[0], bufs[1]
            del bufs
            per_config[name] = per_config_entry(ow, orec, opath, KERNEL_NAMES[opath], peaks,
                                                peaks_src, world)
            torch.cuda.empty_cache()
            if world == 1 and args.cpu_seconds > 0:
                # the oracle in full where it takes a few seconds, else a sample of whole rows
                per_config[name]["cpu_baseline"] = oracle_baseline(oA, oB, ow, min(5.0, args.cpu_seconds))
            del oA, oB
    if sampler is not None:
        sampler.stop()

    if rank != 0:
        return 0

    value = whole_job_tflops(world, w.flops, rec["step_ms"])
    roofline = gemm_roofline(w, path, kernel, rec["kernel_ms"], rec["region_ms"], peaks, peaks_src)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded randn, fp16)", "config": config_of(w, args.epilogue),
        "roofline": roofline,
        "kernel_ms": rec["kernel_ms"],
        "median5": {"ms_per_step": rec["median5_ms"],
                    "TFLOP/s": (whole_job_tflops(world, w.flops, rec["median5_ms"])
                                if rec["median5_ms"] else None),
                    "how": "after the timed region: median over %d repeats of the mean call "
                           "time of %d back-to-back calls" % (args.repeats, max(100, args.steps))},
        "gpu_launches": args.steps,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if context is not None:
        line["context"] = context
    if per_config:
        line["per_config"] = per_config
    if sampler is not None:
        line["clocks"] = sampler.summary(t_wall0, t_wall1)
        if rec["wall_repeats"] is not None:
            # the timed region is a few tens of ms, so a handful of samples at most; the
            # median5 repeats run the same kernel for longer and give the clock under load
            line["clocks"]["median5_window"] = sampler.summary(*rec["wall_repeats"])
    if world == 1 and args.cpu_seconds > 0:
        rows, secs, cores = time_oracle(A, B, w.alpha, args.cpu_seconds)
        per_row_s = secs / rows
        line["cpu_baseline"] = {
            "value": 2.0 * rows * w.N * w.K / secs / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": "%d whole rows of C (of %d), %.1f s" % (rows, w.M, secs),
            "per_row_ms": per_row_s * 1e3,
            "extrapolated_full_s": per_row_s * w.M,
            "extrapolated_note": "extrapolated: measured per-row time x M rows, not a full run",
            "cpu_model": host_cpu_model()}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_attention(args, w):
    """Attention forward on one GPU: same timing rules as the GEMM arm."""
    import torch

    import tensor_core_gemm_multistage_gb300 as gsr
    from tensor_core_gemm_multistage_gb300.workloads import attention_inputs

    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gsr.build()
    q, k, v = attention_inputs(w, seed=0, device=dev)
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def step():
        gsr.flash_attention_fwd(q, k, v, o, causal=w.causal, stream=stream)

    # Q, K, V and O that fit in L2 are evicted between steps (a 256 MiB write outside each
    # step's event pair), so every step reads its inputs from HBM.
    io_bytes = 4 * w.B * w.H * w.S * w.D * 2
    flush = (torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
             if io_bytes <= 2 * L2_BYTES else None)

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / args.steps

    sampler = ClockSampler(gpu_uuid(), interval_ms=5).start() if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    t_wall0 = time.time()
    kernel_ms = timed(step)
    t_wall1 = time.time()
    barrier(world)
    status, code = gsr.device_status(stream)
    if status != gsr.Status.OK:
        raise RuntimeError("device status %s code %#x" % (status.name, code))
    kernel_ms = max_over_ranks(kernel_ms, world)
    context = None
    if args.torch_context:
        sdpa = lambda: torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=w.causal)
        for _ in range(args.warmup):
            sdpa()
        torch.cuda.synchronize()
        ms = timed(sdpa)
        context = {"torch_sdpa": {"ms_per_step": ms, "TFLOP/s": w.flops / (ms * 1e-3) / 1e12}}
    if sampler is not None:
        sampler.stop()
    if rank != 0:
        return 0
    peaks, peaks_src = measured_peaks()
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    peak_key = tensor_peak_key(kernel_ms * args.steps)
    peak = float(peaks[peak_key])
    line = {
        "metric": "attention forward TFLOP/s (FlashAttention-style, fp16 in, fp32 softmax), 1 GPU",
        "value": whole_job_tflops(world, w.flops, kernel_ms), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": kernel_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded randn, fp16)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "causal": w.causal,
                   "flops": "4*B*H*D*(unmasked query-key pairs)",
                   "l2": ("Q, K, V, O %d MiB; " % (io_bytes >> 20)) +
                         ("flush L2 between steps" if flush is not None else "larger than L2, no flush")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "kernel": "gsr_attention_kernel",
                     "traffic": read_traffic(w.name, "gsr_attention_kernel"),
                     "frac_of_burst": achieved / float(peaks["bf16_tflops"]),
                     "peak_source": "%s: %s; fp16 rate taken equal" % (peaks_src, peak_key)},
        "gpu_launches": args.steps,
    }
    if sampler is not None:
        line["clocks"] = sampler.summary(t_wall0, t_wall1)
    if context is not None:
        line["context"] = context
    if world == 1 and args.cpu_seconds > 0:
        from oracle.attention import attention
        qs, ks, vs = (x[:1, :1].cpu() for x in (q, k, v))      # one head
        t = time.perf_counter()
        attention(qs, ks, vs, causal=w.causal)
        secs = time.perf_counter() - t
        line["cpu_baseline"] = {"value": 4 * w.D * w.pairs / secs / 1e12, "unit": "TFLOP/s",
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": "one (batch, head) of the workload, %.1f s" % secs}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gsr", "reference"], default="gsr")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(ATTN_WORKLOADS),
                    default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--epilogue", choices=["scale_relu", "scale", "bias_gelu"], default="scale_relu",
                    help="scale_relu: the fused operator (default); scale: alpha*A@B; "
                         "bias_gelu: GELU(A@B + bias)")
    ap.add_argument("--repeats", type=int, default=5,
                    help="repeats of max(100, steps) calls after the timed region (median reported)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="time only the selected workload, not the other four GEMM configurations")
    ap.add_argument("--torch-context", action="store_true",
                    help="also time torch.relu((A@B)*alpha) and a plain cuBLAS matmul (context)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload in ATTN_WORKLOADS:
        if args.impl == "reference":
            ap.error("the reference arm times the GEMM oracle; attention workloads are gsr-only")
        return run_attention(args, ATTN_WORKLOADS[args.workload])
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gsr(args, w)


if __name__ == "__main__":
    sys.exit(main())

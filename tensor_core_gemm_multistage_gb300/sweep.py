"""Knob sweep: time every runtime configuration of the library on one shape.

The aikraft.ru TileLang tutorial survey ("Knobs" section, 3) tunes a tiled matmul by
trying block sizes, pipeline depth and an L2-swizzle flag, keeping the fastest
configuration that fits in shared memory.  Here tile shapes and pipeline depths are fixed
per kernel at compile time (each kernel's shared-memory budget is checked by a
static_assert), so the runtime knobs are:

  kernel   tiled 128x256, 128x128 or 128x64, CTA pair 256x256 or 256x128, small-M (M <= 256)
  raster   the grouping of tile rows for L2 reuse (gsr_set_raster_group)
  b_copy   3-D copies for B, or separate 64-column 2-D boxes (CTA-pair kernels, N % 64 == 0)
  l2       the CTA-pair kernels' L2 handling: "default" (serpentine K order across waves,
           evict-last A and B, evict-first C stores), "k_forward" (every wave walks K forward),
           "b_evict_first" (B copies marked evict-first)
  split    the small-M kernel's split-K: slabs per 128-column tile (gsr_set_split_k; 0: its
           own choice, as many slabs as fill the SMs once)

    python -m tensor_core_gemm_multistage_gb300.sweep --M 8192 --N 8192 --K 8192

prints one JSON line per configuration and a last line naming the fastest one and the
kernel the library picks on its own.

    python -m tensor_core_gemm_multistage_gb300.sweep --check-choice

times the library's own choice against each of the five main kernels (default knobs) on
shapes around the boundaries of that choice (pair against one-CTA tiles, 256- against
128-wide pair tiles, 256- against 128- against 64-wide one-CTA tiles), one JSON line per shape with the
ratio of the choice's time to the fastest kernel's.  Timing: CUDA events around back-to-back calls after
warm-up, as the tutorial's benchmark_op does; every configuration is timed in several
rounds of shuffled order and the median is kept.  A development tool; nothing here changes the
library's defaults.
"""
from __future__ import annotations

import argparse
import json
import sys

from . import binding as gsr

KERNELS = {"tiled_128x256": gsr.PATH_TILED_256, "tiled_128x128": gsr.PATH_TILED_128,
           "tiled_128x64": gsr.PATH_TILED_64,
           "pair_256x256": gsr.PATH_PAIR, "pair_256x128": gsr.PATH_PAIR_128, "small_m": gsr.PATH_SKINNY}
RASTERS = (0, 4, 16)     # 0: the kernel's default grouping
SPLITS = (0, 1, 2, 4, 8, 16, 32)   # small-M slabs per tile; 0: the kernel's default
NO_3D_B = 2              # test flag bit 1
L2_MODES = {"default": 0, "k_forward": 4, "b_evict_first": 32}   # test flag bits 2 and 5


def candidates(M: int, N: int, K: int):
    """Every (kernel, raster, b_copy, l2, split) combination that is valid for this shape."""
    out = []
    for name, path in KERNELS.items():
        if name == "small_m" and M > 256:       # forced, the small-M kernel takes up to 256 rows
            continue
        rasters = (0,) if name == "small_m" else RASTERS
        copies = ("3d", "2d") if (name.startswith("pair_") and N % 64 == 0) else ("default",)
        l2s = tuple(L2_MODES) if name.startswith("pair_") else ("default",)
        splits = tuple(x for x in SPLITS if x <= (K + 63) // 64) if name == "small_m" else (0,)
        for r in rasters:
            for c in copies:
                for l2 in l2s:
                    for sp in splits:
                        out.append({"kernel": name, "path": path, "raster": r, "b_copy": c, "l2": l2,
                                    "split": sp})
    return out


def time_config(cfg, A, B, C, alpha, warmup=5, iters=30):
    import torch
    gsr.set_path_override(cfg["path"])
    gsr.set_raster_group(cfg["raster"])
    gsr.set_test_flags((NO_3D_B if cfg["b_copy"] == "2d" else 0) | L2_MODES[cfg.get("l2", "default")])
    gsr.set_split_k(cfg.get("split", 0))
    try:
        for _ in range(warmup):
            gsr.gemm_scale_relu(A, B, C, alpha)
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(iters):
            gsr.gemm_scale_relu(A, B, C, alpha)
        e.record()
        torch.cuda.synchronize()
        status, code = gsr.device_status()
        if status != gsr.Status.OK:
            raise RuntimeError("device status %s (%#x)" % (status.name, code))
        return s.elapsed_time(e) / iters
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)
        gsr.set_raster_group(0)
        gsr.set_test_flags(0)
        gsr.set_split_k(0)


def sweep(M: int, N: int, K: int, alpha: float = 0.5, warmup: int = 5, iters: int = 30, seed=0,
          rounds: int = 3):
    """Time every candidate `rounds` times, each round in a fresh random order, and keep the
    median: under the GPU's power cap a configuration timed right after a cool-down runs at a
    higher clock, so a fixed order would favour whichever comes first."""
    import random
    import statistics

    import torch
    from .workloads import make_inputs
    A, B = make_inputs(M, N, K, seed=seed)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.empty(M, N, dtype=torch.float16, device="cuda")
    cands = candidates(M, N, K)
    times = [[] for _ in cands]
    order = list(range(len(cands)))
    rng = random.Random(seed)
    for _ in range(rounds):
        rng.shuffle(order)
        for i in order:
            times[i].append(time_config(cands[i], dA, dB, dC, alpha, warmup, iters))
    results = []
    for cfg, ts in zip(cands, times):
        ms = statistics.median(ts)
        r = {k: v for k, v in cfg.items() if k != "path"}
        r.update({"M": M, "N": N, "K": K, "ms": ms, "ms_all": ts,
                  "TFLOP/s": 2.0 * M * N * K / (ms * 1e-3) / 1e12})
        results.append(r)
    best = min(results, key=lambda r: r["ms"])
    auto = {0: "tiled", 1: "small_m", 2: "pair_256x256", 3: "pair_256x128"}[gsr.select_path(M, N, K)]
    return results, best, auto


# Shapes around the path choice's boundaries: 64 / 70 / 80 / 81 pair tiles of 256 x 256 (the
# choice moves to CTA pairs at 76, half the SMs), narrow N where 256-wide pair tiles leave a
# badly filled last wave, and one-CTA tile widths on either side of half a wave of 128 x 256
# and with N short of a multiple of 256.
CHOICE_SHAPES = [(2048, 2048, 2048), (2304, 2304, 2048), (1792, 2560, 2048), (2048, 2560, 2048),
                 (4096, 1024, 4096), (4096, 1280, 4096), (16384, 128, 4096), (16384, 384, 4096),
                 (16384, 640, 4096), (16384, 1152, 4096), (3072, 3072, 1024), (6144, 6144, 2048),
                 (1536, 2048, 2048), (1024, 2048, 1024), (1280, 2048, 2048), (2000, 3000, 1000),
                 (1024, 1024, 1024), (8192, 384, 4096), (12288, 192, 4096), (1024, 1024, 4096),
                 (1000, 1000, 200), (768, 1536, 2048), (1024, 1536, 1024), (512, 2048, 4096),
                 (1152, 2048, 1024), (256, 16384, 4096), (256, 16384, 8192), (2048, 2048, 8192),
                 (100, 28672, 8192), (80, 32768, 4096), (4096, 16384, 256), (4096, 16384, 512)]
CHOICE_KERNELS = {"auto": gsr.PATH_AUTO, "tiled_128x256": gsr.PATH_TILED_256,
                  "tiled_128x128": gsr.PATH_TILED_128, "tiled_128x64": gsr.PATH_TILED_64,
                  "pair_256x256": gsr.PATH_PAIR,
                  "pair_256x128": gsr.PATH_PAIR_128}
FLUSH_BELOW = 100 << 20   # operands smaller than this would stay in L2 between calls


def _time_calls(path, A, B, C, alpha, calls, flush):
    """Mean time of one call (ms): CUDA events around `calls` back-to-back calls, or around each
    call with a write of `flush` (larger than L2) before it."""
    import torch
    gsr.set_path_override(path)
    try:
        if flush is None:
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(calls):
                gsr.gemm_scale_relu(A, B, C, alpha)
            e.record()
            torch.cuda.synchronize()
            return s.elapsed_time(e) / calls
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(calls)]
        for a, b in ev:
            flush.zero_()
            a.record()
            gsr.gemm_scale_relu(A, B, C, alpha)
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / calls
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)


def check_choice(shapes=None, alpha: float = 0.5, rounds: int = 7, seed: int = 3):
    """The library's choice against each main kernel: per shape, the median over `rounds`
    shuffled rounds of each one's mean call time (L2 flushed between calls when A and B are
    smaller than FLUSH_BELOW, else back to back), the fastest kernel and auto / fastest."""
    import random
    import statistics

    import torch
    from .workloads import make_inputs
    names = {0: "tiled", 1: "small_m", 2: "pair_256x256", 3: "pair_256x128"}
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rows = []
    for M, N, K in (shapes or CHOICE_SHAPES):
        A, B = make_inputs(M, N, K, seed=seed)
        dA, dB = A.cuda(), B.cuda()
        dC = torch.empty(M, N, dtype=torch.float16, device="cuda")
        flush = flush_buf if (M * K + K * N) * 2 < FLUSH_BELOW else None
        calls = 100 if flush is not None else 30
        times = {k: [] for k in CHOICE_KERNELS}
        for k, path in CHOICE_KERNELS.items():          # warm-up, and every kernel must run
            _time_calls(path, dA, dB, dC, alpha, 3, flush)
            status, code = gsr.device_status()
            if status != gsr.Status.OK:
                raise RuntimeError("%s on %dx%dx%d: %s (%#x)" % (k, M, N, K, status.name, code))
        rng = random.Random(seed)
        for _ in range(rounds):
            order = list(CHOICE_KERNELS)
            rng.shuffle(order)
            for k in order:
                times[k].append(_time_calls(CHOICE_KERNELS[k], dA, dB, dC, alpha, calls, flush))
        med = {k: statistics.median(v) * 1e3 for k, v in times.items()}
        fastest = min((k for k in med if k != "auto"), key=med.get)
        rows.append({"M": M, "N": N, "K": K, "l2_flushed": flush is not None, "us": med,
                     "choice": names[gsr.select_path(M, N, K)], "fastest": fastest,
                     "choice_over_fastest": med["auto"] / med[fastest]})
        del dA, dB, dC
        torch.cuda.empty_cache()
    return rows


def main(argv=None):
    ap = argparse.ArgumentParser(description="time every runtime configuration on one shape")
    ap.add_argument("--check-choice", action="store_true",
                    help="time the library's choice against the main kernels on boundary shapes")
    ap.add_argument("--M", type=int)
    ap.add_argument("--N", type=int)
    ap.add_argument("--K", type=int)
    ap.add_argument("--alpha", type=float, default=0.5)
    ap.add_argument("--iters", type=int, default=30)
    ap.add_argument("--rounds", type=int, default=3)
    args = ap.parse_args(argv)
    gsr.lib()
    if args.check_choice:
        for row in check_choice(alpha=args.alpha, rounds=max(args.rounds, 1)):
            print(json.dumps(row))
        return 0
    if args.M is None or args.N is None or args.K is None:
        ap.error("--M, --N and --K are required without --check-choice")
    results, best, auto = sweep(args.M, args.N, args.K, args.alpha, iters=args.iters,
                                rounds=args.rounds)
    for r in results:
        print(json.dumps(r))
    print(json.dumps({"best": best, "library_choice": auto}))
    return 0


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python3
"""Throughput of the persistent warp-specialised bf16 GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one D = A * B^T over the workload's synthetic operands (default
cube8192: M = N = K = 8192, bf16, U[-1,1], seed 3, SM-pair tiles, persistent
grid).  Prints ONE JSON line on rank 0.  Under torchrun each rank drives its own
GPU on its own copy of the workload (weak scaling, no collective on the data
path); the value is the FLOPs of all ranks over the slowest rank's time.

--impl reference times the CPU oracle instead (the plain fp64 triple loop on the
host cores) on a bounded sample of rows of the same workload each step.
"""
from __future__ import annotations

import argparse
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

METRIC = "bf16 GEMM TFLOP/s (device-timed, 1×GB300) and % of dense-bf16 tensor peak"
UNIT = "TFLOP/s"
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_BYTES = 129e6


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="cube8192")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-comparator", dest="comparator", action="store_false",
                    help="skip timing torch.matmul (cuBLAS) as a library comparator")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target duration of the CPU-oracle baseline sample")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing
class Dist:
    def __init__(self, backend: str):
        import torch.distributed as dist
        self.dist = dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.active = self.world > 1
        self.backend = backend
        if self.active and not dist.is_initialized():
            dist.init_process_group(backend=backend)

    def barrier(self):
        if self.active:
            self.dist.barrier()

    def max(self, value: float, device=None) -> float:
        if not self.active:
            return value
        import torch
        t = torch.tensor([value], dtype=torch.float64, device=device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.active and self.dist.is_initialized():
            self.dist.destroy_process_group()


def aggregate(per_rank_flops: float, steps: int, max_ms: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank's work over the slowest rank's time."""
    return world * per_rank_flops * steps / (max_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ peaks, clocks, profiles
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples; keeps those inside [t0, t1]."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()

    def _reader(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        t0, t1 = self.window or (0.0, float("inf"))
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ts, line in self.samples:
            if not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def profiled_traffic(kernel_tag: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel (its device code and planner, build.kernel_digest), else None."""
    from warp_specialized_tma_gb300 import build as libbuild
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.traffic.txt")
    try:
        kv = {}
        with open(path) as fh:
            for line in fh:
                if "=" in line and not line.startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_digest") != libbuild.kernel_digest():
            return None
        return int(float(kv["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------------ CPU oracle sample
def oracle_rate(A, B, K: int, seconds: float, max_rows: int | None = None):
    """(TFLOP/s, rows, seconds, threads) of the oracle on rows of D = A * B^T,
    sized to take about `seconds` on all host cores."""
    import numpy as np
    import oracle
    from warp_specialized_tma_gb300 import inputs
    Ab, Bb = inputs.bits(A), inputs.bits(B)
    threads = oracle.max_threads()
    M, N = Ab.shape[0], Bb.shape[0]
    t0 = time.perf_counter()
    oracle.gemm_rows(Ab, Bb, K=K, rows=np.arange(threads) % M)
    per_wave = max(time.perf_counter() - t0, 1e-6)
    waves = max(1, int(seconds / per_wave))
    rows = threads * waves if max_rows is None else min(threads * waves, max_rows)
    sel = np.random.default_rng(0).integers(0, M, size=rows)
    t0 = time.perf_counter()
    oracle.gemm_rows(Ab, Bb, K=K, rows=sel)
    dt = time.perf_counter() - t0
    return 2.0 * rows * N * K / dt / 1e12, rows, dt, threads


# ------------------------------------------------------------------ arms
def workload_config(name: str, info: dict | None):
    from warp_specialized_tma_gb300 import inputs
    w = inputs.WORKLOADS[name]
    M, N, K = w["M"], w["N"], w["K"]
    cfg = {
        "workload": f"{name}: D = A*B^T, M={M} N={N} K={K}, A[M,K] and B[N,K] K-major bf16, "
                    f"{w['dist']} seed {w['seed']}, fp32 accumulation, bf16 D",
        "M": M, "N": N, "K": K,
        "l2": f"inputs larger than L2 (A+B = {2 * (M * K + N * K) / 2**20:.0f} MiB > 129 MB); no flush"
        if 2 * (M * K + N * K) > L2_BYTES else "L2 flushed between steps",
    }
    if info:
        cfg.update({"cta_group": info["cta_group"], "tile": f"{info['tile_m']}x{info['tile_n']}x{info['tile_k']}",
                    "stages": info["stages"], "grid_ctas": info["grid_ctas"], "persistent": info["persistent"],
                    "acc_buffers": info["acc_buffers"], "setmaxnreg": info["setmaxnreg"]})
    return cfg


def run_reference(args):
    """The CPU oracle as the reference arm: rank 0 only, bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from warp_specialized_tma_gb300 import inputs
    import oracle
    w = inputs.WORKLOADS[args.workload]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.make_workload(args.workload)
    import numpy as np
    Ab, Bb = inputs.bits(A), inputs.bits(B)
    threads = oracle.max_threads()
    total = args.steps + args.warmup
    # the whole run takes about 150 s whatever the step count: a step is a
    # sample of D -- random rows, and a contiguous block of columns (a view of
    # B's rows, no copy) once one row per thread is more than a step's share
    per_step_budget = min(2.0, 150.0 / max(total, 1))
    t0 = time.perf_counter()
    oracle.gemm_rows(Ab, Bb, K=K, rows=np.arange(threads) % M)
    per_wave = max(time.perf_counter() - t0, 1e-6)
    rows = threads * max(1, int(per_step_budget / per_wave))
    cols = N if per_wave <= per_step_budget else max(8, min(N, int(N * per_step_budget / per_wave)))
    rng = np.random.default_rng(1)

    def step():
        c0 = int(rng.integers(0, N - cols + 1))
        oracle.gemm_rows(Ab, Bb[c0:c0 + cols], K=K, rows=rng.integers(0, M, size=rows))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = 2.0 * rows * cols * K * args.steps / dt / 1e12
    sample = (f"{rows} random rows x {cols} contiguous columns of D per step (of {M} x {N}), K={K}; "
              f"{args.steps} steps in {dt:.1f} s")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    from warp_specialized_tma_gb300 import binding, inputs
    from warp_specialized_tma_gb300 import build as libbuild

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the GEMM has no CPU path)")
    dist = Dist("nccl")
    world = dist.world
    local = dist.local_rank
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    libbuild.build()

    w = inputs.WORKLOADS[args.workload]
    M, N, K = w["M"], w["N"], w["K"]
    flops = 2.0 * M * N * K
    A, B = inputs.make_workload(args.workload)
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    g = binding.Gemm(local)
    info = g.plan(M, N, K)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 3)):
        g.run(dA, dB, dD, stream)
    st, detail = g.device_status()
    if st != binding.OK:
        raise RuntimeError(f"device watchdog tripped during warm-up: {detail:#x}")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)  # let nvidia-smi start sampling
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_begin.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        g.run(dA, dB, dD, stream)
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    dist.barrier()
    clocks.mark(wall0, wall1)
    clock_info = clocks.stop()

    st, detail = g.device_status()
    if st != binding.OK:
        raise RuntimeError(f"device watchdog tripped in the timed region: {detail:#x}")
    ms_total = t_begin.elapsed_time(t_end)
    max_ms = dist.max(ms_total, dev)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_ms = statistics.fmean(launch_ms)
    value = aggregate(flops, args.steps, max_ms, world)

    # End to end through the C ABI with host operands (pinned): every step copies
    # its A and B host -> device, multiplies and copies D device -> host.  Steps
    # alternate between two streams, each with its own device buffers and its
    # own handle (a handle's workspace serves one launch at a time), so the
    # copies of one step overlap the multiply of the other.
    hA, hB = A.pin_memory(), B.pin_memory()
    streams = [stream, torch.cuda.Stream(dev)]
    bufs = [(dA, dB, dD), (torch.empty_like(dA), torch.empty_like(dB), torch.empty_like(dD))]
    hDs = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    gs = [g, binding.Gemm(local)]
    gs[1].plan(M, N, K)
    for i in range(4):
        j = i % 2
        gs[j].run_host(hA, hB, hDs[j], *bufs[j], streams[j])
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(dev)
    e0.record(streams[0])
    streams[1].wait_event(e0)
    for i in range(args.e2e_steps):
        j = i % 2
        gs[j].run_host(hA, hB, hDs[j], *bufs[j], streams[j])
    streams[0].wait_stream(streams[1])
    e1.record(streams[0])
    torch.cuda.synchronize(dev)
    e2e_ms = dist.max(e0.elapsed_time(e1), dev)
    e2e_value = aggregate(flops, args.e2e_steps, e2e_ms, world)

    # Library comparator (not an oracle): cuBLAS through torch.matmul on the
    # same device operands, outside the timed region above.  The GPU's clock
    # under its power cap depends on what ran just before, so the comparator and
    # this kernel run in alternating back-to-back loops (ours, cuBLAS, cuBLAS,
    # ours, ...) of the same total length, and both rates are reported.
    lib_tflops = ours_alt = None
    if args.comparator:
        dD2 = torch.empty_like(dD)
        for _ in range(max(args.warmup, 3)):
            torch.matmul(dA, dB.t(), out=dD2)
        torch.cuda.synchronize(dev)
        chunk = max(1, args.steps // 4)
        t_lib = t_ours = 0.0

        def loop(fn):
            l0 = torch.cuda.Event(enable_timing=True)
            l1 = torch.cuda.Event(enable_timing=True)
            l0.record(stream)
            for _ in range(chunk):
                fn()
            l1.record(stream)
            torch.cuda.synchronize(dev)
            return l0.elapsed_time(l1)

        ours_fn = lambda: g.run(dA, dB, dD, stream)  # noqa: E731
        lib_fn = lambda: torch.matmul(dA, dB.t(), out=dD2)  # noqa: E731
        for c in range(4):
            for fn in ((ours_fn, lib_fn) if c % 2 == 0 else (lib_fn, ours_fn)):
                ms = loop(fn)
                if fn is lib_fn:
                    t_lib += ms
                else:
                    t_ours += ms
        lib_tflops = flops * 4 * chunk / (t_lib * 1e-3) / 1e12
        ours_alt = flops * 4 * chunk / (t_ours * 1e-3) / 1e12
        st2, detail2 = g.device_status()
        if st2 != binding.OK:
            raise RuntimeError(f"device watchdog tripped in the comparator loops: {detail2:#x}")
        del dD2

    # The host link's bound on the end-to-end rate (a link measurement, no
    # kernel): a step's bytes moved on the link's best schedule -- A and B
    # host -> device on one stream while a D goes device -> host on the other.
    def copies(i):
        with torch.cuda.stream(streams[0]):
            bufs[0][0].copy_(hA, non_blocking=True)
            bufs[0][1].copy_(hB, non_blocking=True)
        with torch.cuda.stream(streams[1]):
            hDs[1].copy_(bufs[1][2], non_blocking=True)

    for i in range(4):
        copies(i)
    torch.cuda.synchronize(dev)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(dev)
    c0.record(streams[0])
    streams[1].wait_event(c0)
    for i in range(args.e2e_steps):
        copies(i)
    streams[0].wait_stream(streams[1])
    c1.record(streams[0])
    torch.cuda.synchronize(dev)
    copy_ms = dist.max(c0.elapsed_time(c1), dev)
    copy_bound = aggregate(flops, args.e2e_steps, copy_ms, world)
    for gg in gs:
        st, detail = gg.device_status()
        if st != binding.OK:
            raise RuntimeError(f"device watchdog tripped in the end-to-end loop: {detail:#x}")
    gs[1].close()

    # The timed region is seconds of back-to-back launches under the GPU's
    # power cap -- the condition of the sustained cuBLAS figure (a back-to-back
    # loop of seconds), so that is the roofline denominator; the fraction of
    # the burst figure (best single launches) is reported beside it.
    peaks, peak_src = load_peaks()
    peak_burst = peaks.get("bf16_tflops")
    peak = peaks.get("bf16_tflops_sustained")
    kernel_tag = f"gemm_ws_c{info['cta_group']}"
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    traffic = profiled_traffic(kernel_tag, args.workload)

    cpu = None
    if dist.rank == 0 and world == 1:
        rate, rows, secs, threads = oracle_rate(A, B, K, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{rows} random rows of D (of {M}), all {N} columns, K={K}: {secs:.1f} s"}

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args.workload, info),
            "pct_of_dense_bf16_peak": {
                "nominal_2250_tflops": 100.0 * value / world / NOMINAL_BF16_TFLOPS,
                f"{peak_src}_burst": 100.0 * value / world / peak_burst,
                f"{peak_src}_sustained": 100.0 * value / world / peak,
            },
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": kernel_tag, "kernel_ms": kernel_ms,
                         "timed_seconds": kernel_ms * args.steps * 1e-3,
                         "peak_source": f"{peak_src} bf16_tflops_sustained (back-to-back loop of seconds under "
                                        f"the power cap, as the timed region here)",
                         "frac_of_burst_peak": achieved / peak_burst},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 2 * (M * K + N * K),
                    "d2h_bytes_per_step": 2 * M * N, "streams": 2,
                    "call": "gemm_bf16_run_host (H2D A,B + GEMM + D2H D per step)",
                    "bound": "host link", "copies_only_value": copy_bound,
                    "frac_of_copy_bound": e2e_value / copy_bound},
            "detail": {
                "launch_ms": {"mean": kernel_ms, "median": statistics.median(launch_ms), "best": min(launch_ms)},
                "tflops_best_launch": flops / (min(launch_ms) * 1e-3) / 1e12,
                "hbm_gbs_compulsory": 2.0 * (M * K + N * K + M * N) / (kernel_ms * 1e-3) / 1e9,
                "library_comparator": None if lib_tflops is None else {
                    "what": "torch.matmul(A, B.T) (cuBLAS), same operands; alternating back-to-back loops "
                            "with this kernel, each side " + str(4 * max(1, args.steps // 4)) + " launches",
                    "value": lib_tflops, "ours_in_the_same_loops": ours_alt,
                    "ratio_ours_to_library": ours_alt / lib_tflops, "unit": UNIT},
            },
            "gpu_launches": args.steps,
            "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    g.close()
    dist.close()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

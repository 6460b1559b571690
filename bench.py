#!/usr/bin/env python3
"""Throughput of the persistent warp-specialised bf16 GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-detail]

One step = one D = A * B^T over the workload's synthetic operands (default
cube8192: M = N = K = 8192, bf16, U[-1,1], seed 3, SM-pair tiles, persistent
grid).  Prints ONE JSON line on rank 0.  Under torchrun each rank drives its own
GPU on its own copy of the workload (weak scaling, no collective on the data
path); the value is the FLOPs of all ranks over the slowest rank's time.

Besides the headline workload, rank 0 at N = 1 reports in ``detail``:
  workloads  the other four synthetic workloads (cube256, cube4096, longk,
             ragged): CUDA-event time per launch, TFLOP/s, fraction of the
             nominal roofline (max of FLOPs at 2.25 PFLOP/s and compulsory bytes
             at 8 TB/s) and of the measured peak, and the CPU oracle on a
             bounded sample of each;
  skinny     decode-like shapes (16 x 8192 x 8192, 8192 x 16 x 8192,
             64 x 8192 x 8192): compulsory HBM GB/s against the measured copy
             bandwidth, and against a device copy that moves the same bytes
             (the rate HBM gives a plain streaming kernel at this size);
  sustained  the headline kernel back to back for >= 1.5 s under the power cap,
             with its SM clock.

--impl reference times the CPU oracle instead (the plain fp64 triple loop on the
host cores) on a bounded sample of rows of the same workload each step.
"""
from __future__ import annotations

import argparse
import ctypes
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
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_BYTES = 129e6
# A timed region shorter than this is a burst: the GPU has not yet settled at
# its power-capped clock, so the burst peak (best single launches) applies.
SUSTAINED_MIN_S = 1.0
SKINNY_SHAPES = [(16, 8192, 8192), (8192, 16, 8192), (64, 8192, 8192)]


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
    ap.add_argument("--no-detail", dest="detail", action="store_false",
                    help="skip the other workloads, the skinny shapes and the sustained loop")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="target duration of the CPU-oracle baseline sample of the headline workload")
    ap.add_argument("--cpu-seconds-detail", type=float, default=1.5,
                    help="target duration of the CPU-oracle sample of each other workload")
    ap.add_argument("--sustained-seconds", type=float, default=1.5)
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


# ------------------------------------------------------------------ roofline and peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def nominal_roofline(M: int, N: int, K: int) -> dict:
    """The roofline of D = A * B^T: the larger of 2MNK FLOPs at the nominal
    dense-bf16 tensor peak and the compulsory bytes 2(MK + NK + MN) at nominal
    HBM bandwidth, and which of the two binds."""
    flops = 2.0 * M * N * K
    nbytes = 2.0 * (M * K + N * K + M * N)
    t_flop = flops / (NOMINAL_BF16_TFLOPS * 1e12)
    t_byte = nbytes / (NOMINAL_HBM_GBS * 1e9)
    return {"flops": flops, "bytes": nbytes, "us": max(t_flop, t_byte) * 1e6,
            "bound": "tensor" if t_flop >= t_byte else "hbm"}


def measured_peak(peaks: dict, src: str, bound: str, timed_s: float) -> dict:
    """The measured denominator for a kernel: the copy bandwidth for an
    HBM-bound one; for a tensor-bound one the burst cuBLAS figure when the
    timed region is shorter than SUSTAINED_MIN_S (the clock has not settled
    under the power cap yet), else the sustained one."""
    if bound == "hbm":
        return {"peak": peaks["hbm_gbs"], "unit": "GB/s", "kind": "hbm",
                "source": f"{src} hbm_gbs (copy bandwidth)"}
    if timed_s < SUSTAINED_MIN_S:
        return {"peak": peaks["bf16_tflops"], "unit": UNIT, "kind": "burst",
                "source": f"{src} bf16_tflops (burst: the timed region lasts {timed_s:.3f} s "
                          f"< {SUSTAINED_MIN_S:.0f} s, before the clock settles under the power cap)"}
    return {"peak": peaks["bf16_tflops_sustained"], "unit": UNIT, "kind": "sustained",
            "source": f"{src} bf16_tflops_sustained (the timed region lasts {timed_s:.1f} s "
                      f">= {SUSTAINED_MIN_S:.0f} s under the power cap)"}


# ------------------------------------------------------------------ clocks
class NvmlClocks:
    """SM clock, its maximum, board power and the clock-event reasons, sampled
    every ~1 ms by a thread through read-only NVML queries (ctypes; nothing is
    ever set).  Samples are kept with their wall-clock time; summary() takes
    those inside a window."""

    CLOCK_SM = 1
    REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
               (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))

    def __init__(self, torch_device):
        self.ok = False
        self.samples = []
        self._stop = threading.Event()
        self._thread = None
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if not self._find(torch_device):
                return
            self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = self.sample() is not None
        except (OSError, AttributeError):
            self.ok = False

    def _find(self, dev) -> bool:
        import torch
        props = torch.cuda.get_device_properties(dev)
        uuid = str(getattr(props, "uuid", "") or "")
        for cand in (uuid, "GPU-" + uuid):
            if uuid and self.lib.nvmlDeviceGetHandleByUUID(cand.encode(), ctypes.byref(self.handle)) == 0:
                return True
        if hasattr(props, "pci_bus_id"):
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            fn = getattr(self.lib, "nvmlDeviceGetHandleByPciBusId_v2", None)
            if fn is not None and fn(bus.encode(), ctypes.byref(self.handle)) == 0:
                return True
        return False

    def sample(self):
        sm, smax, mw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        mask = ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, self.CLOCK_SM, ctypes.byref(sm)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.CLOCK_SM, ctypes.byref(smax))
        self.lib.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(mw))
        self._reasons(self.handle, ctypes.byref(mask))
        return (time.time(), float(sm.value), float(smax.value), mw.value / 1000.0, int(mask.value))

    def start(self, period: float = 0.001):
        if not self.ok:
            return

        def loop():
            while not self._stop.is_set():
                s = self.sample()
                if s is not None:
                    self.samples.append(s)
                time.sleep(period)

        self._stop.clear()
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)
            self._thread = None

    def summary(self, t0: float, t1: float) -> dict:
        sel = [s for s in self.samples if t0 <= s[0] <= t1]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvml"}
        reasons = sorted({name for s in sel for bit, name in self.REASONS if s[4] & bit})
        return {"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": max(s[2] for s in sel),
                "sm_mhz_min": min(s[1] for s in sel), "power_w_median": statistics.median(s[3] for s in sel),
                "reasons": reasons, "samples": len(sel), "source": "nvml (read-only queries, ~1 ms period)"}


class SmiClocks:
    """Fallback when NVML cannot be loaded: nvidia-smi samples every 100 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self, period: float = 0.1):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _reader(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvidia-smi"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi (100 ms period)"}


def clock_sampler(dev, local: int):
    s = NvmlClocks(dev)
    return s if s.ok else SmiClocks(local)


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


# ------------------------------------------------------------------ device timing
def time_back_to_back(run, n: int, stream, dev) -> float:
    """Mean ms per launch of n launches back to back, one CUDA-event pair on `stream`."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(n):
        run()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / n


def time_each_flushed(run, n: int, stream, dev, flush_buf) -> list:
    """ms of each of n launches, each bracketed by its own CUDA events on
    `stream`, with a write of flush_buf (larger than L2) before each one."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(n):
            flush_buf.fill_(i & 0xFF)
            starts[i].record(stream)
            run()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


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


def measure_shape(M, N, K, dist, seed, dev, stream, peaks, peak_src, flush_buf, label,
                  cpu_seconds=None, graph_too=False, hbm_comparator=False, library_comparator=False):
    """One problem through the C ABI: plan, warm up, time.  Inputs larger than
    L2 are timed back to back; smaller ones launch by launch with an L2 flush
    before each.  With library_comparator, torch.matmul (cuBLAS) on the same
    operands is timed the same way afterwards.  Returns a dict for the bench
    line's detail block."""
    import torch
    from warp_specialized_tma_gb300 import binding, inputs
    A, B = inputs.make_problem(M, N, K, dist, seed)
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    roof = nominal_roofline(M, N, K)
    with binding.Gemm(dev.index) as g:
        info = g.plan(M, N, K)

        def run():
            g.run(dA, dB, dD, stream)

        for _ in range(5):
            run()
        torch.cuda.synchronize(dev)
        # about 30 ms of kernel time, at least 20 launches
        probe = time_back_to_back(run, 3, stream, dev)
        n = int(min(2000, max(20, 30.0 / max(probe, 1e-3))))
        big = 2.0 * (M * K + N * K) > L2_BYTES
        graph_us = None
        if big:
            ms = time_back_to_back(run, n, stream, dev)
            l2 = "inputs larger than L2; back to back"
        else:
            each = time_each_flushed(run, min(n, 200), stream, dev, flush_buf)
            ms = statistics.fmean(each)
            l2 = "L2 flushed before each launch; per-launch CUDA events"
        if graph_too:
            # captured on torch's side stream: the launches go to the current
            # stream, whichever that is during capture
            graph = torch.cuda.CUDAGraph()
            reps = 200
            with torch.cuda.graph(graph):
                for _ in range(reps):
                    g.run(dA, dB, dD)
            graph.replay()
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            graph_us = e0.elapsed_time(e1) / reps * 1e3
            del graph
        st, detail = g.device_status()
        if st != binding.OK:
            raise RuntimeError(f"device watchdog tripped on {label}: {detail:#x}")
    achieved_tflops = roof["flops"] / (ms * 1e-3) / 1e12
    gbs = roof["bytes"] / (ms * 1e-3) / 1e9
    pk = measured_peak(peaks, peak_src, roof["bound"], ms * n * 1e-3)
    out = {
        "M": M, "N": N, "K": K, "dist": dist, "seed": seed,
        "kernel": f"gemm_thin<{info['thin']}>" if info["thin"] else f"gemm_ws_c{info['cta_group']}",
        "launches": n, "us_per_launch": ms * 1e3, "tflops": achieved_tflops, "hbm_gbs_compulsory": gbs,
        "roofline_us_nominal": roof["us"], "bound": roof["bound"],
        "frac_of_nominal_roofline": roof["us"] / (ms * 1e3),
        "frac_of_measured_peak": (achieved_tflops if roof["bound"] == "tensor" else gbs) / pk["peak"],
        "measured_peak": pk["peak"], "measured_peak_unit": pk["unit"], "measured_peak_kind": pk["kind"],
        "l2": l2,
        "plan": {k: info[k] for k in ("cta_group", "grid_ctas", "stages", "tiles", "sk_tiles", "sk_head",
                                      "repack", "thin")},
    }
    if hbm_comparator:
        # A device copy that moves the same number of bytes (half the bytes
        # read, half written) at this transfer size: what HBM delivers to a
        # plain streaming kernel with the same fixed costs of a launch.
        half = int(roof["bytes"] // 4)  # bf16 elements read = elements written = bytes / 4
        src = torch.empty(half, dtype=torch.bfloat16, device=dev)
        dst = torch.empty_like(src)
        cms = time_back_to_back(lambda: dst.copy_(src), 20, stream, dev)
        cgbs = 4.0 * half / (cms * 1e-3) / 1e9
        out["copy_same_bytes"] = {"what": "dst.copy_(src) moving the same bytes (half read, half written), "
                                          "back to back", "us": cms * 1e3, "gbs": cgbs,
                                  "ours_over_copy": gbs / cgbs}
        del src, dst
    if library_comparator:
        # Not an oracle and not part of the library: the vendor GEMM on the same
        # operands under the same timing protocol, for context.
        dD2 = torch.empty_like(dD)

        def lib_run():
            torch.matmul(dA, dB.t(), out=dD2)

        for _ in range(5):
            lib_run()
        torch.cuda.synchronize(dev)
        if big:
            lms = time_back_to_back(lib_run, n, stream, dev)
        else:
            lms = statistics.fmean(time_each_flushed(lib_run, min(n, 200), stream, dev, flush_buf))
        out["library_comparator"] = {"what": "torch.matmul(A, B.T) (cuBLAS), same operands, same protocol ("
                                             + l2 + "), timed after ours",
                                     "us_per_launch": lms * 1e3,
                                     "tflops": roof["flops"] / (lms * 1e-3) / 1e12,
                                     "ours_over_library_time": ms / lms}
        del dD2
    if graph_us is not None:
        out["graph_replay_us_per_launch"] = graph_us
        out["graph_replay_note"] = "200 launches replayed from one CUDA graph, back to back (inputs stay in L2)"
    if cpu_seconds:
        rate, rows, secs, threads = oracle_rate(A, B, K, cpu_seconds)
        out["cpu_oracle"] = {"value": rate, "unit": UNIT, "cores": threads,
                             "sample": f"{rows} random rows of D (of {M}), all {N} columns: {secs:.2f} s"}
    del dA, dB, dD
    return out


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
    roof = nominal_roofline(M, N, K)
    A, B = inputs.make_workload(args.workload)
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    big = 2.0 * (M * K + N * K) > L2_BYTES
    flush_buf = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=dev)

    g = binding.Gemm(local)
    info = g.plan(M, N, K)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 3)):
        g.run(dA, dB, dD, stream)
    st, detail = g.device_status()
    if st != binding.OK:
        raise RuntimeError(f"device watchdog tripped during warm-up: {detail:#x}")

    clocks = clock_sampler(dev, local)
    clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_begin.record(stream)
    for i in range(args.steps):
        if not big:
            flush_buf.fill_(i & 0xFF)  # inputs fit in L2: flush it between steps
        starts[i].record(stream)
        g.run(dA, dB, dD, stream)
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    dist.barrier()
    clock_info = clocks.summary(wall0, wall1)

    st, detail = g.device_status()
    if st != binding.OK:
        raise RuntimeError(f"device watchdog tripped in the timed region: {detail:#x}")
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_ms = statistics.fmean(launch_ms)
    ms_total = t_begin.elapsed_time(t_end) if big else kernel_ms * args.steps
    max_ms = dist.max(ms_total, dev)
    value = aggregate(flops, args.steps, max_ms, world)
    timed_s = max_ms * 1e-3

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
    # Loops of this pattern run in one of two modes on GB300: the two streams'
    # copies overlap (~1.48 ms per step), or, in about one loop in ten in
    # isolation and more often right after heavy GEMM load, they serialise
    # (~2.47 ms per step) -- whatever the copy call (plain torch copies do the
    # same).  So the loop is timed five times and the median is reported, with
    # every run kept.
    def e2e_loop():
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
        return dist.max(e0.elapsed_time(e1), dev)

    e2e_runs = [aggregate(flops, args.e2e_steps, e2e_loop(), world) for _ in range(5)]
    e2e_value = statistics.median(e2e_runs)

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
        ours_fn = lambda: g.run(dA, dB, dD, stream)  # noqa: E731
        lib_fn = lambda: torch.matmul(dA, dB.t(), out=dD2)  # noqa: E731
        for c in range(4):
            for fn in ((ours_fn, lib_fn) if c % 2 == 0 else (lib_fn, ours_fn)):
                ms = time_back_to_back(fn, chunk, stream, dev) * chunk
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

    def copy_loop():
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
        return dist.max(c0.elapsed_time(c1), dev)

    copy_runs = [aggregate(flops, args.e2e_steps, copy_loop(), world) for _ in range(5)]
    copy_bound = statistics.median(copy_runs)
    for gg in gs:
        st, detail = gg.device_status()
        if st != binding.OK:
            raise RuntimeError(f"device watchdog tripped in the end-to-end loop: {detail:#x}")
    gs[1].close()
    del bufs[1], hDs

    peaks, peak_src = load_peaks()
    pk = measured_peak(peaks, peak_src, roof["bound"], kernel_ms * args.steps * 1e-3)
    kernel_tag = f"gemm_ws_c{info['cta_group']}"
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    traffic = profiled_traffic(kernel_tag, args.workload)

    # The same kernel back to back for >= sustained_seconds: the rate once the
    # clock has settled under the power cap, with the clock it ran at.
    sustained = None
    if args.detail and dist.rank == 0 and world == 1:
        n = max(1, int(math.ceil(args.sustained_seconds / max(kernel_ms * 1e-3, 1e-6))))
        torch.cuda.synchronize(dev)
        s0 = time.time()
        ms = time_back_to_back(lambda: g.run(dA, dB, dD, stream), n, stream, dev)
        s1 = time.time()
        sc = clocks.summary(s0 + 0.25 * (s1 - s0), s1)  # the settled part of the loop
        tfl = flops / (ms * 1e-3) / 1e12
        sustained = {"launches": n, "seconds": ms * n * 1e-3, "tflops": tfl,
                     "frac_of_sustained_peak": tfl / peaks["bf16_tflops_sustained"],
                     "frac_of_nominal": tfl / NOMINAL_BF16_TFLOPS,
                     "clocks_last_three_quarters": sc}
        st, detail = g.device_status()
        if st != binding.OK:
            raise RuntimeError(f"device watchdog tripped in the sustained loop: {detail:#x}")
    clocks.stop()

    cpu = None
    if dist.rank == 0 and world == 1:
        rate, rows, secs, threads = oracle_rate(A, B, K, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{rows} random rows of D (of {M}), all {N} columns, K={K}: {secs:.1f} s"}

    # The other workloads and the skinny shapes (rank 0 at N = 1 only).
    workloads = skinny = None
    if args.detail and dist.rank == 0 and world == 1:
        g.close()
        del dA, dB, dD
        torch.cuda.empty_cache()
        workloads = {}
        for name, wl in inputs.WORKLOADS.items():
            if name == args.workload:
                continue
            workloads[name] = measure_shape(wl["M"], wl["N"], wl["K"], wl["dist"], wl["seed"], dev, stream,
                                            peaks, peak_src, flush_buf, name,
                                            cpu_seconds=args.cpu_seconds_detail, graph_too=(name == "cube256"),
                                            library_comparator=args.comparator)
        skinny = {}
        for (m, n_, k) in SKINNY_SHAPES:
            skinny[f"{m}x{n_}x{k}"] = measure_shape(m, n_, k, "uniform", 3, dev, stream, peaks, peak_src,
                                                    flush_buf, f"{m}x{n_}x{k}", hbm_comparator=True,
                                                    library_comparator=args.comparator)

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args.workload, info),
            "pct_of_dense_bf16_peak": {
                "nominal_2250_tflops": 100.0 * value / world / NOMINAL_BF16_TFLOPS,
                f"{peak_src}_burst": 100.0 * value / world / peaks["bf16_tflops"],
                f"{peak_src}_sustained": 100.0 * value / world / peaks["bf16_tflops_sustained"],
                "applicable": pk["kind"],
            },
            "roofline": {"bound": roof["bound"], "achieved": achieved, "peak": pk["peak"], "unit": pk["unit"],
                         "frac": achieved / pk["peak"], "traffic": traffic,
                         "kernel": kernel_tag, "kernel_ms": kernel_ms,
                         "timed_seconds": timed_s, "peak_kind": pk["kind"], "peak_source": pk["source"],
                         "frac_of_nominal_roofline": roof["us"] / (kernel_ms * 1e3),
                         "roofline_us_nominal": roof["us"],
                         "algorithmic_flops_per_launch": flops,
                         "algorithmic_bytes_per_launch": roof["bytes"]},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 2 * (M * K + N * K),
                    "d2h_bytes_per_step": 2 * M * N, "streams": 2,
                    "call": "gemm_bf16_run_host (H2D A,B + GEMM + D2H D per step)",
                    "bound": "host link", "copies_only_value": copy_bound,
                    "frac_of_copy_bound": e2e_value / copy_bound,
                    "runs": e2e_runs, "copies_only_runs": copy_runs,
                    "note": "median of 5 timed loops of e2e_steps steps each"},
            "detail": {
                "launch_ms": {"mean": kernel_ms, "median": statistics.median(launch_ms), "best": min(launch_ms)},
                "tflops_best_launch": flops / (min(launch_ms) * 1e-3) / 1e12,
                "hbm_gbs_compulsory": roof["bytes"] / (kernel_ms * 1e-3) / 1e9,
                "library_comparator": None if lib_tflops is None else {
                    "what": "torch.matmul(A, B.T) (cuBLAS), same operands; alternating back-to-back loops "
                            "with this kernel, each side " + str(4 * max(1, args.steps // 4)) + " launches",
                    "value": lib_tflops, "ours_in_the_same_loops": ours_alt,
                    "ratio_ours_to_library": ours_alt / lib_tflops, "unit": UNIT},
                "sustained": sustained,
                "workloads": workloads,
                "skinny": skinny,
            },
            # the GEMM per step, plus the operand copy kernel when the plan repacks
            "gpu_launches": args.steps * (2 if info["repack"] else 1),
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

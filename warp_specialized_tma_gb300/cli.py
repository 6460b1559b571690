"""Run and time one GEMM workload through the C ABI.

    python -m warp_specialized_tma_gb300.cli --workload cube8192 --iters 20 \
        [--set cta_group=2 --set stages=6 ...] [--shape M N K]

Prints the resolved plan, the mean CUDA-event time per launch, the TFLOP/s and
the fraction of the roofline (the larger of the FLOPs at 2.25 PFLOP/s and the
compulsory bytes at 8 TB/s).  This is the command the ncu summaries under
profiles/ were taken with.  With --cublas, torch.matmul (cuBLAS) on the same
operands is timed after the library, the same number of launches, as a
comparator; it is not part of the library.
"""
from __future__ import annotations

import argparse
import json
import sys

import torch

from . import binding, inputs
from . import build as libbuild

NOMINAL_TFLOPS = 2250.0   # GB300 dense bf16 tensor peak
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workload", default="cube8192", choices=list(inputs.WORKLOADS))
    ap.add_argument("--shape", type=int, nargs=3, metavar=("M", "N", "K"),
                    help="override the workload's shape (its distribution and seed are kept)")
    ap.add_argument("--iters", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--set", action="append", default=[], metavar="OPTION=VALUE",
                    help=f"library option, one of {sorted(binding.OPTIONS)}")
    ap.add_argument("--device", type=int, default=0)
    ap.add_argument("--graph", action="store_true",
                    help="time the launches replayed from one CUDA graph (no host launch cost per launch)")
    ap.add_argument("--cublas", action="store_true",
                    help="also time torch.matmul(A, B.T) (cuBLAS) on the same operands, after the library's launches")
    args = ap.parse_args(argv)

    w = dict(inputs.WORKLOADS[args.workload])
    if args.shape:
        w["M"], w["N"], w["K"] = args.shape
    M, N, K = w["M"], w["N"], w["K"]
    opts = {}
    for kv in args.set:
        k, v = kv.split("=", 1)
        opts[k] = int(v)

    libbuild.build()
    torch.cuda.set_device(args.device)
    dev = torch.device("cuda", args.device)
    A, B = inputs.make_problem(M, N, K, w["dist"], w["seed"])
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(args.device, **opts) as g:
        info = g.plan(M, N, K)
        for _ in range(args.warmup):
            g.run(dA, dB, dD)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if args.graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(args.iters):
                    g.run(dA, dB, dD)
            graph.replay()  # warm-up of the graph itself
            torch.cuda.synchronize(dev)
            e0.record()
            graph.replay()
            e1.record()
        else:
            e0.record()
            for _ in range(args.iters):
                g.run(dA, dB, dD)
            e1.record()
        torch.cuda.synchronize(dev)
        st, detail = g.device_status()
    ms = e0.elapsed_time(e1) / max(args.iters, 1)
    cublas_ms = None
    if args.cublas:
        dD2 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        for _ in range(args.warmup):
            torch.matmul(dA, dB.t(), out=dD2)
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(args.iters):
            torch.matmul(dA, dB.t(), out=dD2)
        e1.record()
        torch.cuda.synchronize(dev)
        cublas_ms = e0.elapsed_time(e1) / max(args.iters, 1)
    flops = 2.0 * M * N * K
    nbytes = 2.0 * (M * K + N * K + M * N)  # compulsory: read A and B, write D once
    # roofline time: the larger of the FLOPs at the dense-bf16 tensor peak and
    # the compulsory bytes at HBM bandwidth (nominal 2.25 PFLOP/s and 8 TB/s)
    roof_us = max(flops / NOMINAL_TFLOPS / 1e12, nbytes / NOMINAL_HBM_GBS / 1e9) * 1e6
    out = {"M": M, "N": N, "K": K, "options": opts, "graph": args.graph, "plan": info, "ms_per_launch": ms,
           "tflops": flops / (ms * 1e-3) / 1e12, "hbm_gbs_compulsory": nbytes / (ms * 1e-3) / 1e9,
           "roofline_us_nominal": roof_us,
           "roofline_bound": "tensor" if flops / NOMINAL_TFLOPS / 1e12 >= nbytes / NOMINAL_HBM_GBS / 1e9 else "hbm",
           "frac_of_roofline_nominal": roof_us / (ms * 1e3), "status": st, "detail": detail}
    if cublas_ms is not None:
        out["cublas_ms_per_launch"] = cublas_ms
        out["cublas_tflops"] = flops / (cublas_ms * 1e-3) / 1e12
    print(json.dumps(out))
    return 0 if st == binding.OK else 1


if __name__ == "__main__":
    sys.exit(main())

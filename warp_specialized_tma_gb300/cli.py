"""Run and time one GEMM workload through the C ABI.

    python -m warp_specialized_tma_gb300.cli --workload cube8192 --iters 20 \
        [--set cta_group=2 --set stages=6 ...] [--shape M N K]

Prints the resolved plan and the mean CUDA-event time per launch.  This is the
command the ncu summaries under profiles/ were taken with.
"""
from __future__ import annotations

import argparse
import json
import sys

import torch

from . import binding, inputs
from . import build as libbuild


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
        e0.record()
        for _ in range(args.iters):
            g.run(dA, dB, dD)
        e1.record()
        torch.cuda.synchronize(dev)
        st, detail = g.device_status()
    ms = e0.elapsed_time(e1) / max(args.iters, 1)
    out = {"M": M, "N": N, "K": K, "options": opts, "plan": info, "ms_per_launch": ms,
           "tflops": 2.0 * M * N * K / (ms * 1e-3) / 1e12, "status": st, "detail": detail}
    print(json.dumps(out))
    return 0 if st == binding.OK else 1


if __name__ == "__main__":
    sys.exit(main())

"""Ablation ladder of the GEMM pipeline on one workload.

    python -m warp_specialized_tma_gb300.ablation --workload cube8192 [--rounds 5]

Each rung adds one design element, from the non-specialised loop that guards the
stage ring with __syncthreads up to the default kernel:

  sync_war    one elected thread loads + issues MMAs, __syncthreads WAR guard
  mbar_war    same loop, "empty" mbarrier WAR guard (tcgen05.commit arrives)
  ws          warp-specialised (producer / MMA / epilogue warps), one tile per CTA
  +persistent grid = resident CTAs, grid-stride tile loop, ring runs across tiles
  +tmem2      two TMEM accumulators: the epilogue overlaps the next tile
  +setmaxnreg producer warps give registers to the epilogue warps
  +2cta       an SM pair per 256x256 tile (cta_group::2)
  +streamk    tiles split along k: the partial last wave, or, with fewer tiles
              than SM pairs, every tile's tail taken by an idle SM pair
  +k-alt      consecutive whole tiles walk k in alternating directions
  +serpentine odd tile bands walk their columns right to left (the default)

With --shape M N K the workload's distribution and seed are drawn at another
shape.  With --schedules the default kernel is compared with its schedule options
instead: the ping-pong epilogue, the dynamic tile counter, and both.  With
--variant NAME:OPT=V,OPT=V (repeatable) any named option sets are compared,
e.g. --variant aligned:repack=0 --variant unaligned:repack=2.

Rungs run interleaved in shuffled order for several rounds (the GPU's power
limit moves the clock between runs) and the best and median times are printed
as one JSON line per rung.
"""
from __future__ import annotations

import argparse
import json
import random
import statistics
import sys

import torch

from . import binding, inputs
from . import build as libbuild

RUNGS = [
    ("sync_war", dict(pipeline=binding.PIPE_SYNC_WAR, serpentine=0)),
    ("mbar_war", dict(pipeline=binding.PIPE_MBAR_WAR, serpentine=0)),
    ("ws", dict(cta_group=1, persistent=0, acc_buffers=1, stream_k=0, k_order=0, serpentine=0)),
    ("+persistent", dict(cta_group=1, persistent=1, acc_buffers=1, stream_k=0, k_order=0, serpentine=0)),
    ("+tmem2", dict(cta_group=1, acc_buffers=2, stream_k=0, k_order=0, serpentine=0)),
    ("+setmaxnreg", dict(cta_group=1, acc_buffers=2, setmaxnreg=1, stream_k=0, k_order=0, serpentine=0)),
    ("+2cta", dict(cta_group=2, setmaxnreg=0, stream_k=0, k_order=0, serpentine=0)),
    ("+streamk", dict(k_order=0, serpentine=0)),
    ("+k-alt", dict(serpentine=0)),
    ("+serpentine", dict()),
]


SCHEDULE_RUNGS = [
    ("default", dict()),
    ("pingpong", dict(epi_schedule=1)),
    ("dynamic", dict(scheduler=1)),
    ("pingpong+dynamic", dict(epi_schedule=1, scheduler=1)),
]


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workload", default="cube8192", choices=list(inputs.WORKLOADS))
    ap.add_argument("--shape", type=int, nargs=3, metavar=("M", "N", "K"),
                    help="override the workload's shape (its distribution and seed are kept)")
    ap.add_argument("--rounds", type=int, default=5)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--device", type=int, default=0)
    ap.add_argument("--schedules", action="store_true", help="compare the schedule options")
    ap.add_argument("--variant", action="append", default=[], metavar="NAME:OPT=V,...",
                    help="compare named option sets instead of the ladder")
    args = ap.parse_args(argv)
    rungs = RUNGS
    if args.schedules:
        rungs = SCHEDULE_RUNGS
    if args.variant:
        rungs = []
        for spec in args.variant:
            name, _, opts = spec.partition(":")
            kv = dict(item.split("=", 1) for item in opts.split(",") if item)
            rungs.append((name, {k: int(v) for k, v in kv.items()}))

    libbuild.build()
    torch.cuda.set_device(args.device)
    dev = torch.device("cuda", args.device)
    w = inputs.WORKLOADS[args.workload]
    M, N, K = args.shape if args.shape else (w["M"], w["N"], w["K"])
    A, B = inputs.make_problem(M, N, K, w["dist"], w["seed"])
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    handles = []
    for name, opts in rungs:
        g = binding.Gemm(args.device, **opts)
        handles.append((name, g, g.plan(M, N, K)))

    def once(g) -> float:
        for _ in range(3):
            g.run(dA, dB, dD)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.iters):
            g.run(dA, dB, dD)
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.iters

    times = {name: [] for name, _, _ in handles}
    rng = random.Random(0)
    for _ in range(args.rounds):
        order = list(range(len(handles)))
        rng.shuffle(order)
        for i in order:
            name, g, _ = handles[i]
            times[name].append(once(g))
    flops = 2.0 * M * N * K
    rc = 0
    for name, g, info in handles:
        st, detail = g.device_status()
        rc |= st != binding.OK
        best, med = min(times[name]), statistics.median(times[name])
        print(json.dumps({"workload": args.workload, "shape": [M, N, K], "rung": name, "best_ms": round(best, 4),
                          "median_ms": round(med, 4), "tflops_best": round(flops / best / 1e9, 1),
                          "tflops_median": round(flops / med / 1e9, 1), "grid": info["grid_ctas"],
                          "stages": info["stages"], "sk_tiles": info["sk_tiles"], "sk_head": info["sk_head"],
                          "repack": info["repack"],
                          "status": st}))
        g.close()
    return rc


if __name__ == "__main__":
    sys.exit(main())

"""GPU parity of the thin kernel (min(M, N) <= 64) against the CPU oracle.

The thin kernel puts the large operand on the MMA's 128-row side and the small
one, rounded up to 16, 32, 48 or 64 rows, on its N side; split tiles are
summed from fp32 partials in a fixed order.  Integer-valued inputs make every
sum exact, so there the result must equal the oracle's bf16 rounding bit for
bit, in both orientations (small B: D rows are accumulator rows; small A: D
is the accumulator transposed), with padded pitches, the fused epilogue,
repeated launches of one handle and a watchdog give-up in between.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from warp_specialized_tma_gb300 import binding, inputs

from test_gemm_gpu import SENTINEL_BITS, check, rms, run_fused_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from warp_specialized_tma_gb300 import build as libbuild
    libbuild.build()
    binding.load()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def nt_of(M, N):
    small = N if N <= 64 else M
    return (small + 15) // 16 * 16


def run_thin(A, B, M, N, K, ldd=None, **opts):
    """D on the GPU with the thin kernel forced; returns (D on the CPU, plan info)."""
    ldd = N if ldd is None else ldd
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.full((M, ldd), SENTINEL_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
    opts = {"thin": 2} | opts
    with binding.Gemm(0, **opts) as g:
        info = g.plan(M, N, K, A.shape[1], B.shape[1], ldd)
        g.run(dA, dB, dD)
        st, detail = g.device_status()
        assert st == binding.OK, f"device status {st} detail {detail:#x}"
    torch.cuda.synchronize()
    return dD.cpu(), info


SHAPES = [
    # small B (D rows are accumulator rows)
    (4096, 16, 4104), (1000, 1, 130), (300, 17, 64), (2048, 48, 1000), (129, 64, 8), (8192, 40, 2048),
    # small A (D is the accumulator transposed)
    (16, 4096, 4104), (1, 1000, 130), (17, 300, 64), (48, 2048, 1000), (64, 129, 8), (40, 8192, 2048),
    # both small
    (16, 16, 512), (7, 5, 3), (64, 64, 64),
]


@pytest.mark.parametrize("split", ["sms", "auto"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_thin_exact_integers(shape, split):
    # "sms": the units split across the SMs, split tiles summed through global
    # memory; "auto": the planner's choice, clusters for most of these shapes
    M, N, K = shape
    ld = (K + 7) // 8 * 8  # rows 16-byte aligned, as TMA needs
    A, B = inputs.make_problem(M, N, K, "int2", seed=M * 7 + N * 3 + K, lda=ld, ldb=ld)
    D, info = run_thin(A, B, M, N, K, **({"thin_cluster": 0} if split == "sms" else {}))
    assert info["thin"] == nt_of(M, N) and info["cta_group"] == 1 and info["tile_m"] == 128
    if split == "sms":
        assert info["thin_cluster"] == 0
    check(D, A, B, M, N, K, exact=True)


# Clusters of C CTAs per tile, every C the option allows (clamped to the
# k-blocks), on ragged rows and k tails in both orientations: rank 0 adds the
# others' partials read through distributed shared memory.
@pytest.mark.parametrize("C", [2, 3, 5, 8])
@pytest.mark.parametrize("shape", [(16, 1000, 1000), (1000, 40, 700), (48, 2048, 4104), (300, 64, 200), (7, 129, 70)],
                         ids=lambda s: "x".join(map(str, s)))
def test_thin_cluster_sizes_exact(shape, C):
    M, N, K = shape
    ld = (K + 7) // 8 * 8
    A, B = inputs.make_problem(M, N, K, "int2", seed=C * 1000 + M + N + K, lda=ld, ldb=ld)
    D, info = run_thin(A, B, M, N, K, thin_cluster=C)
    KB = (K + 63) // 64
    assert info["thin_cluster"] == min(C, KB)
    assert info["grid_ctas"] == info["tiles"] * info["thin_cluster"]
    check(D, A, B, M, N, K, exact=True)


@pytest.mark.parametrize("C", [2, 4])
def test_thin_cluster_random_values_padded(C):
    M, N, K = 33, 777, 520
    A, B = inputs.make_problem(M, N, K, "normal", seed=93, lda=528, ldb=520)
    D, info = run_thin(A, B, M, N, K, ldd=780, thin_cluster=C)
    assert info["thin_cluster"] == C
    check(D, A, B, M, N, K)  # also checks the padding columns of D keep the sentinel


@pytest.mark.parametrize("shape,pads", [((2048, 16, 1000), (1008, 1024, 24)), ((16, 2048, 1000), (1016, 1000, 2056)),
                                        ((777, 33, 520), (520, 528, 40)), ((33, 777, 520), (528, 520, 780))],
                         ids=["smallB", "smallA", "smallB33", "smallA33"])
def test_thin_random_values_padded(shape, pads):
    M, N, K = shape
    lda, ldb, ldd = pads
    A, B = inputs.make_problem(M, N, K, "normal", seed=91, lda=lda, ldb=ldb)
    D, info = run_thin(A, B, M, N, K, ldd=ldd)
    assert info["thin"] == nt_of(M, N)
    check(D, A, B, M, N, K)  # also checks the padding columns of D keep the sentinel


@pytest.mark.parametrize("shape", [(2048, 16, 1000), (16, 2048, 1000), (300, 40, 200), (40, 300, 200)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("cluster", [0, 3])
def test_thin_fused_exact_integers(shape, cluster):
    M, N, K = shape
    A, B = inputs.make_problem(M, N, K, "int2", seed=81)
    g = torch.Generator().manual_seed(82)
    C = inputs.make_operand(M, N, None, "int2", g)
    bias = inputs.make_operand(1, N, None, "int2", g).reshape(-1)
    D = run_fused_gpu(A, B, M, N, K, C=C, bias=bias, alpha=2.0, beta=-3.0, thin=2, thin_cluster=cluster)
    _, refbf = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 2.0, -3.0, C=inputs.bits(C),
                                      bias=inputs.bits(bias))
    assert np.array_equal(inputs.bits(D), refbf)


def test_thin_fused_in_place_random_values():
    M, N, K = 24, 1500, 704
    A, B = inputs.make_problem(M, N, K, "normal", seed=83)
    g = torch.Generator().manual_seed(84)
    C = inputs.make_operand(M, N, None, "normal", g)
    bias = inputs.make_operand(1, N, None, "uniform", g).reshape(-1)
    D = run_fused_gpu(A, B, M, N, K, C=C, bias=bias, alpha=0.625, beta=1.25, inplace=True, thin=2)
    ref64, _ = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 0.625, 1.25, C=inputs.bits(C),
                                      bias=inputs.bits(bias))
    tol = 4e-3 * np.abs(ref64) + 2e-3 * math.sqrt(K) * rms(A, K) * rms(B, K) * 0.625 + 1e-6
    assert np.all(np.abs(D.double().numpy() - ref64) <= tol)


@pytest.mark.parametrize("cluster", [0, 1])
def test_thin_repeated_launches_with_split_tiles(cluster):
    # 64 tiles of 128 k-blocks, split across the SMs (every launch raises its
    # flags with a new epoch and each tile's owner adds the partials) or in
    # clusters of 2 (the automatic choice here)
    M, N, K = 16, 8192, 8192
    dev = torch.device("cuda:0")
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0, thin=2, thin_cluster=cluster) as g:
        info = g.plan(M, N, K)
        assert info["thin"] == 16 and info["tiles"] == 64 and info["grid_ctas"] > info["tiles"]
        assert info["thin_cluster"] == (0 if cluster == 0 else 2)
        for seed in (101, 102, 103):
            A, B = inputs.make_problem(M, N, K, "int2", seed=seed)
            g.run(A.to(dev), B.to(dev), dD)
            assert g.device_status()[0] == binding.OK
            check(dD.cpu(), A, B, M, N, K, exact=True)


def test_thin_plans_of_other_grids_and_a_fresh_handle_on_freed_memory():
    # The epoch and the count of CTAs that read it live on the device: plans
    # with other grid sizes (152 CTAs, then 64 for 8 tiles of 8 k-blocks) must
    # keep them consistent, and a new handle, whose workspace may reuse the
    # freed memory of an old one with higher epochs, must start clean.
    dev = torch.device("cuda:0")
    shapes = [(16, 8192, 8192), (16, 1024, 512), (8192, 24, 4096), (16, 8192, 8192)]
    for rounds in range(2):
        with binding.Gemm(0, thin=2) as g:
            for i, (M, N, K) in enumerate(shapes):
                info = g.plan(M, N, K)
                assert info["thin"] > 0
                for rep in range(2 + 3 * rounds):
                    A, B = inputs.make_problem(M, N, K, "int2", seed=200 + 10 * i + rep)
                    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                    g.run(A.to(dev), B.to(dev), dD)
                    assert g.device_status()[0] == binding.OK
                    check(dD.cpu(), A, B, M, N, K, exact=True)


@pytest.mark.parametrize("cluster", [0, 2, 4])  # across the SMs; clusters that push, and that pull, partials
def test_thin_watchdog_gives_up_and_the_handle_recovers(cluster):
    M, N, K = 16, 4096, 4096
    A, B = inputs.make_problem(M, N, K, "int2", seed=111)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0, thin=2, thin_cluster=cluster, watchdog_ns=20_000_000, fault_skip_load=3) as g:
        g.plan(M, N, K)
        g.run(dA, dB, dD)
        st, detail = g.device_status()
        assert st == binding.ERR_DEVICE_TIMEOUT and detail != 0
        g.set_option("fault_skip_load", -1)
        g.plan(M, N, K)
        g.run(dA, dB, dD)
        assert g.device_status()[0] == binding.OK
    check(dD.cpu(), A, B, M, N, K, exact=True)


def test_thin_selection():
    with binding.Gemm(0) as g:  # automatic (the default)
        assert g.plan(16, 8192, 8192)["thin"] == 16
        assert g.plan(1, 8192, 8192)["thin"] == 16
        assert g.plan(8192, 16, 4096)["thin"] == 16
        assert g.plan(8192, 17, 8192)["thin"] == 32   # up to 64 rows, either operand
        assert g.plan(64, 4096, 2048)["thin"] == 64
        assert g.plan(4096, 48, 2048)["thin"] == 48
        assert g.plan(16, 4096, 2040)["thin"] == 0    # K < 2048: the square kernel measured faster
        assert g.plan(16, 4000, 8192)["thin"] == 0    # too little to stream
        assert g.plan(65, 8192, 8192)["thin"] == 0
        assert g.plan(8192, 8192, 8192)["thin"] == 0
    with binding.Gemm(0, thin=2) as g:
        assert g.plan(33, 33, 104)["thin"] == 48
        assert g.plan(8192, 64, 8192)["thin"] == 64
        assert g.plan(8192, 65, 8192)["thin"] == 0
    with binding.Gemm(0, cta_group=1) as g:  # a square-kernel option: no automatic thin
        assert g.plan(16, 8192, 8192)["thin"] == 0
    with binding.Gemm(0, thin=2, cta_group=1) as g:
        assert g.plan(16, 8192, 8192)["thin"] == 16
    with binding.Gemm(0, thin=0) as g:
        assert g.plan(16, 8192, 8192)["thin"] == 0


def test_thin_cluster_selection():
    # automatic: clusters where tiles x C reaches 60 % of the SMs and each CTA
    # streams at most 160 k-blocks; else the units split across the SMs
    with binding.Gemm(0) as g:
        sms = g.plan(16, 8192, 8192)["num_sms"]
        assert sms == 152  # the figures below are for GB300
        assert g.plan(16, 8192, 8192)["thin_cluster"] == 2       # 64 tiles
        assert g.plan(8192, 16, 8192)["thin_cluster"] == 2
        assert g.plan(64, 8192, 8192)["thin_cluster"] == 2
        assert g.plan(16, 4096, 8192)["thin_cluster"] == 4       # 32 tiles
        assert g.plan(16, 12288, 8192)["thin_cluster"] == 1      # 96 whole tiles
        assert g.plan(16, 16384, 16384)["thin_cluster"] == 0     # 256 k-blocks per CTA: across the SMs
        assert g.plan(16, 28672, 8192)["thin_cluster"] == 0      # more tiles than SMs
        assert g.plan(16, 4096, 2048)["thin_cluster"] == 4
        info = g.plan(16, 8192, 8192)
        assert info["grid_ctas"] == 128
    with binding.Gemm(0, thin_cluster=0) as g:
        assert g.plan(16, 8192, 8192)["thin_cluster"] == 0
        assert g.plan(16, 8192, 8192)["grid_ctas"] == 152
    with binding.Gemm(0, thin_cluster=8) as g:
        info = g.plan(16, 4096, 8192)
        assert info["thin_cluster"] == 8 and info["grid_ctas"] == 256  # two waves of clusters


# The decode-like shapes bench.py reports, at full size and in the default
# (automatic) launch configuration, every element against the oracle; and the
# thin kernel at 64 small rows in both orientations.
@pytest.mark.parametrize("shape,opts", [
    ((16, 8192, 8192), {}), ((8192, 16, 8192), {}), ((64, 8192, 8192), {}),
    ((8192, 64, 8192), {}), ((64, 8192, 8192), {"thin": 2}), ((40, 16384, 16384), {"thin": 2}),
], ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else ",".join(f"{k}={x}" for k, x in v.items()) or "auto")
def test_skinny_full_size_every_element(shape, opts):
    from test_gemm_gpu import every_element
    M, N, K = shape
    for dist, exact in (("uniform", False), ("int2", True)):
        A, B = inputs.make_problem(M, N, K, dist, 3 if dist == "uniform" else 103)
        dev = torch.device("cuda:0")
        dD = torch.full((M, N), SENTINEL_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
        with binding.Gemm(0, **opts) as g:
            g.plan(M, N, K)
            g.run(A.to(dev), B.to(dev), dD)
            assert g.device_status()[0] == binding.OK
        every_element(dD.cpu(), A, B, M, N, K, exact=exact)

"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Tolerance (per element, against the oracle's unrounded fp64 sum ref64):
    |d - ref64| <= 4e-3 * |ref64| + 2e-3 * sqrt(K) * sigma_A * sigma_B
with sigma the RMS of the generated operand.  Integer-valued inputs make every
fp32 partial sum exact, so there the bf16 result must equal the oracle's bf16
rounding bit for bit.  Padding columns of D (n >= N) must never be written.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from warp_specialized_tma_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

SENTINEL_BITS = 0x7FC1  # a NaN pattern no correct kernel writes


@pytest.fixture(scope="module", autouse=True)
def _built():
    from warp_specialized_tma_gb300 import build as libbuild
    libbuild.build()
    binding.load()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def pad8(K: int) -> int:
    """Smallest leading dimension >= K whose rows start 16-byte aligned."""
    return (K + 7) // 8 * 8


def rms(t: torch.Tensor, K: int) -> float:
    v = t[:, :K].double()
    return float(v.pow(2).mean().sqrt())


def run_gpu(A, B, M, N, K, ldd=None, **opts):
    """D (CPU, M x ldd bf16) computed on the GPU through the C ABI."""
    ldd = N if ldd is None else ldd
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.full((M, ldd), SENTINEL_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
    with binding.Gemm(0, **opts) as g:
        g.plan(M, N, K, A.shape[1], B.shape[1], ldd)
        g.run(dA, dB, dD)
        st, detail = g.device_status()
        assert st == binding.OK, f"device status {st} detail {detail:#x}"
    torch.cuda.synchronize()
    return dD.cpu()


def check(D, A, B, M, N, K, rows=None, exact=False):
    """Compares rows of D with the oracle; returns the max abs error."""
    rows = np.arange(M) if rows is None else np.asarray(rows)
    ref64, refbf = oracle.gemm_rows(inputs.bits(A), inputs.bits(B), K=K, rows=rows)
    Dbits = inputs.bits(D)
    got_bits = Dbits[rows][:, :N]
    if exact:
        bad = np.argwhere(got_bits != refbf)
        assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"
    got = inputs.from_bits(np.ascontiguousarray(got_bits)).double().numpy()
    tol = 4e-3 * np.abs(ref64) + 2e-3 * math.sqrt(K) * rms(A, K) * rms(B, K)
    err = np.abs(got - ref64)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{len(bad)} elements outside tolerance, first {bad[:5].tolist()}, "
                           f"max err {np.nanmax(err):.4g}")
    # columns beyond N keep the sentinel
    if Dbits.shape[1] > N:
        assert np.all(Dbits[:, N:] == SENTINEL_BITS)
    return float(np.max(err)) if err.size else 0.0


def _ordered(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers whose differences count ulps across zero."""
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def sample_rows(M: int, tile_m: int = 128, seed: int = 0, extra: int = 16):
    """First/last row of every 128-row slab plus random rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    for s in range(0, M, tile_m):
        rows.add(s)
        rows.add(min(M - 1, s + tile_m - 1))
        rows.add(min(M - 1, s + 31 + (s // tile_m) % 64))
    rows.update(rng.integers(0, M, size=extra).tolist())
    return np.array(sorted(rows), dtype=np.int64)


# ------------------------------------------------------------------ small shapes
TINY = [(1, 1, 1), (1, 1, 8), (2, 3, 5), (5, 8, 7), (8, 8, 8), (3, 1, 4), (7, 5, 2)]


@pytest.mark.parametrize("M,N,K", TINY)
@pytest.mark.parametrize("cta_group", [1, 2])
def test_tiny_shapes(M, N, K, cta_group):
    A, B = inputs.make_problem(M, N, K, "normal", seed=M * 100 + N * 10 + K, lda=8, ldb=8)
    D = run_gpu(A, B, M, N, K, ldd=N, cta_group=cta_group)
    check(D, A, B, M, N, K)
    Ai, Bi = inputs.make_problem(M, N, K, "int2", seed=K, lda=8, ldb=8)
    check(run_gpu(Ai, Bi, M, N, K, cta_group=cta_group), Ai, Bi, M, N, K, exact=True)


MID = [(256, 256, 256), (300, 520, 200), (129, 257, 65), (640, 384, 1000), (1000, 1000, 1000)]


@pytest.mark.parametrize("M,N,K", MID)
@pytest.mark.parametrize("variant", [
    dict(cta_group=1),
    dict(cta_group=2),
    dict(cta_group=1, setmaxnreg=1),
    dict(cta_group=2, setmaxnreg=1),
    dict(cta_group=2, acc_buffers=1),
    dict(cta_group=2, stage_group=1),
    dict(cta_group=1, stage_group=1),
    dict(cta_group=1, persistent=0),
    dict(cta_group=2, persistent=0),
    dict(cta_group=1, epi_schedule=1),
    dict(cta_group=2, epi_schedule=1),
    dict(cta_group=1, scheduler=1),
    dict(cta_group=2, scheduler=1),
    dict(cta_group=2, epi_schedule=1, scheduler=1),
    dict(cta_group=2, scheduler=1, persistent=0),
    dict(cta_group=1, k_order=0),
    dict(cta_group=2, k_order=0),
    dict(pipeline=binding.PIPE_SYNC_WAR),
    dict(pipeline=binding.PIPE_MBAR_WAR),
])
def test_mid_shapes_all_variants(M, N, K, variant):
    A, B = inputs.make_problem(M, N, K, "normal", seed=M + N + K, lda=pad8(K), ldb=pad8(K))
    check(run_gpu(A, B, M, N, K, **variant), A, B, M, N, K)
    Ai, Bi = inputs.make_problem(M, N, K, "int2", seed=M + N + K + 1, lda=pad8(K), ldb=pad8(K))
    check(run_gpu(Ai, Bi, M, N, K, **variant), Ai, Bi, M, N, K, exact=True)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("max_ctas,stages,group", [(2, 2, 2), (4, 3, 1), (6, 0, 0), (4, 4, 2), (2, 4, 1)])
def test_few_ctas_many_tiles_ring_wraps(cta_group, max_ctas, stages, group):
    # few persistent CTAs walk many tiles: the ring and the accumulator
    # barriers wrap across tile boundaries many times; K = 520 gives 9 k-blocks
    # per tile, so released stage pairs straddle tile boundaries
    M, N, K = 1100, 1300, 520
    A, B = inputs.make_problem(M, N, K, "int2", seed=21)
    D = run_gpu(A, B, M, N, K, cta_group=cta_group, max_ctas=max_ctas, stages=stages, stage_group=group)
    check(D, A, B, M, N, K, exact=True)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("M,N,K,max_ctas", [
    (1024, 1024, 4096, 12),   # several split tiles, each over a few clusters
    (1000, 900, 1000, 6),     # ragged edges and a k tail inside split tiles
    (2048, 1536, 2560, 10),   # whole tiles plus split tiles
    (512, 512, 8192, 6),      # long k, owners with several contributors
])
def test_stream_k_split_tiles_exact(cta_group, M, N, K, max_ctas):
    A, B = inputs.make_problem(M, N, K, "int2", seed=M + K)
    with binding.Gemm(0, cta_group=cta_group, max_ctas=max_ctas) as g:
        info = g.plan(M, N, K)
    assert info["sk_tiles"] > 0
    D = run_gpu(A, B, M, N, K, cta_group=cta_group, max_ctas=max_ctas)
    check(D, A, B, M, N, K, exact=True)
    # the split schedule and the whole-tile schedule agree bit for bit here
    D0 = run_gpu(A, B, M, N, K, cta_group=cta_group, max_ctas=max_ctas, stream_k=0)
    assert torch.equal(D.view(torch.int16), D0.view(torch.int16))


SCHEDULES = [dict(epi_schedule=1), dict(scheduler=1), dict(epi_schedule=1, scheduler=1), dict(k_order=0),
             dict(k_order=0, scheduler=1)]


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("max_ctas,K", [(2, 520), (6, 64), (10, 200)])
def test_schedules_few_ctas_many_tiles_repeated(cta_group, sched, max_ctas, K):
    # Many items per SM (pair): the schedule ring and both epilogue groups wrap
    # many times; K = 64 gives one k-block per tile, so the producer runs
    # several tiles ahead.  Four launches on one handle: the dynamic counter
    # must be back at 0 before each.
    M, N = 1100, 1300
    A, B = inputs.make_problem(M, N, K, "int2", seed=23 + K)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    outs = []
    with binding.Gemm(0, cta_group=cta_group, max_ctas=max_ctas, **sched) as g:
        info = g.plan(M, N, K)
        assert info["epi_schedule"] == sched.get("epi_schedule", 0)
        assert info["scheduler"] == sched.get("scheduler", 0)
        assert info["k_order"] == sched.get("k_order", 1)
        for _ in range(4):
            D = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=dev)
            g.run(dA, dB, D)
            outs.append(D)
        st, detail = g.device_status()
        assert st == binding.OK, f"device status {st} detail {detail:#x}"
    torch.cuda.synchronize()
    check(outs[0].cpu(), A, B, M, N, K, exact=True)
    for D in outs[1:]:
        assert torch.equal(D.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("sched", SCHEDULES)
def test_schedules_with_stream_k_split_tiles(cta_group, sched):
    M, N, K, max_ctas = 2048, 1536, 2560, 10
    A, B = inputs.make_problem(M, N, K, "int2", seed=M + K)
    with binding.Gemm(0, cta_group=cta_group, max_ctas=max_ctas, **sched) as g:
        assert g.plan(M, N, K)["sk_tiles"] > 0
    D = run_gpu(A, B, M, N, K, cta_group=cta_group, max_ctas=max_ctas, **sched)
    check(D, A, B, M, N, K, exact=True)
    D0 = run_gpu(A, B, M, N, K, cta_group=cta_group, max_ctas=max_ctas)
    assert torch.equal(D.view(torch.int16), D0.view(torch.int16))


def test_schedule_options_are_validated():
    with binding.Gemm(0, epi_schedule=1, acc_buffers=1) as g:
        with pytest.raises(binding.GemmError) as e:
            g.plan(512, 512, 512)
        assert e.value.status == binding.ERR_INVALID_ARG
    with binding.Gemm(0, epi_schedule=1, scheduler=1, pipeline=binding.PIPE_MBAR_WAR) as g:
        info = g.plan(512, 512, 512)  # the ablation loops have neither schedule
        assert info["epi_schedule"] == 0 and info["scheduler"] == 0


def test_dynamic_scheduler_recovers_after_watchdog_timeout():
    # a load is skipped, the launch gives up part-way with tiles left in the
    # counter; the next launch on the same handle must still cover every tile
    M, N, K = 1024, 1024, 1024
    A, B = inputs.make_problem(M, N, K, "int2", seed=31)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0, watchdog_ns=20_000_000, fault_skip_load=5, scheduler=1, max_ctas=4) as g:
        g.plan(M, N, K)
        g.run(dA, dB, dD)
        st, detail = g.device_status()
        assert st == binding.ERR_DEVICE_TIMEOUT and detail & 0x80000000
        g.set_option("fault_skip_load", -1)
        g.plan(M, N, K)
        for _ in range(2):
            dD.fill_(3.0)
            g.run(dA, dB, dD)
            assert g.device_status()[0] == binding.OK
            check(dD.cpu(), A, B, M, N, K, exact=True)


@pytest.mark.parametrize("M,N,K,lda,ldb", [
    (1000, 900, 1000, 1008, 1000),   # both pitches misaligned (2016 B, 2000 B)
    (300, 520, 1001, 1008, 1064),    # k tail of one element in the copy
    (129, 257, 8, 8, 16),            # one short k-block, 16- and 32-byte pitches
    (640, 384, 4104, 4104, 4160),    # only A misaligned
])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_repacked_operands_exact(M, N, K, lda, ldb, cta_group):
    A, B = inputs.make_problem(M, N, K, "int2", seed=K + lda, lda=lda, ldb=ldb)
    with binding.Gemm(0, repack=1, cta_group=cta_group) as g:
        info = g.plan(M, N, K, lda, ldb, N)
    want = (1 if (lda * 2) % 128 else 0) | (2 if (ldb * 2) % 128 else 0)
    assert info["repack"] == want and info["packed_ld"] == (K + 63) // 64 * 64
    D = run_gpu(A, B, M, N, K, repack=1, cta_group=cta_group)
    check(D, A, B, M, N, K, exact=True)
    D0 = run_gpu(A, B, M, N, K, repack=2, cta_group=cta_group)
    assert torch.equal(D.view(torch.int16), D0.view(torch.int16))


def test_repack_copies_every_run_and_auto_rule():
    # automatic mode: A is copied when N >= 4096, B when M >= 4096
    M, N, K = 4100, 4200, 520
    A, B = inputs.make_problem(M, N, K, "int2", seed=91)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    rows = sample_rows(M, extra=8)
    with binding.Gemm(0) as g:
        assert g.plan(M, N, K)["repack"] == 3  # 1040-byte pitches
        g.run(dA, dB, dD)
        torch.cuda.synchronize()
        check(dD.cpu(), A, B, M, N, K, rows=rows, exact=True)
        # new operand values: the copy must be taken again
        A2 = (A.float() * -1).to(torch.bfloat16)
        dA.copy_(A2)
        g.run(dA, dB, dD)
        g.run_fused(dA, dB, dD, dD, None, 1.0, 1.0)  # D = A2 B^T + (A2 B^T) = 2 A2 B^T
        assert g.device_status()[0] == binding.OK
    torch.cuda.synchronize()
    check((dD.cpu().float() / 2).to(torch.bfloat16), A2, B, M, N, K, rows=rows, exact=True)
    with binding.Gemm(0) as g:
        assert g.plan(M, 1000, K)["repack"] == 2   # N < 4096: A stays, B (M >= 4096) is copied
        assert g.plan(1000, N, K)["repack"] == 1
        assert g.plan(M, N, 512)["repack"] == 0    # 1024-byte pitches are aligned


def test_ragged_workload_is_repacked_automatically():
    w = inputs.WORKLOADS["ragged"]
    with binding.Gemm(0) as g:
        info = g.plan(w["M"], w["N"], w["K"])
    assert info["repack"] == 3 and info["packed_ld"] == 4160


def test_stream_k_random_inputs_and_repeated_launches():
    # flags carry a per-launch epoch: back-to-back launches on one handle must
    # not read a previous launch's partials
    M, N, K = 1536, 1280, 3072
    A, B = inputs.make_problem(M, N, K, "normal", seed=77)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    outs = []
    with binding.Gemm(0, max_ctas=8) as g:
        assert g.plan(M, N, K)["sk_tiles"] > 0
        for i in range(3):
            D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            g.run(dA if i != 1 else dA * 2, dB, D)
            outs.append(D)
        assert g.device_status()[0] == binding.OK
    torch.cuda.synchronize()
    check(outs[0].cpu(), A, B, M, N, K)
    check(outs[2].cpu(), A, B, M, N, K)
    assert torch.equal(outs[1].cpu().float(), (outs[0].cpu().float() * 2))


# Fewer tiles than SM (pairs): every tile is split at the same k-block; the
# owner computes the head and adds the partials of the tails, which the other
# SM (pairs) share.  stream_k = 3 takes the split whatever the planner's cost
# model says.  Shapes (with the cta_group = 2 / 1 tile counts T and cluster
# counts C that max_ctas gives):
HEAD_TAIL = [
    (512, 512, 8192, 12),    # T = 4 / 8 on C = 6 / 12: a tail range holds two whole tails
    (600, 700, 8200, 20),    # ragged edges and a k tail of 8 (T = 9 / 15, C = 10 / 20)
    (256, 512, 8192, 16),    # T = 2 / 4 on C = 8 / 16: each tail split over three ranges
    (1792, 256, 8192, 16),   # T = 7 / 14 on C = 8 / 16: one range holds seven tails
]


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("M,N,K,max_ctas", HEAD_TAIL)
def test_stream_k_head_tail_exact(cta_group, M, N, K, max_ctas):
    A, B = inputs.make_problem(M, N, K, "int2", seed=M + N + K)
    with binding.Gemm(0, cta_group=cta_group, max_ctas=max_ctas, stream_k=3) as g:
        info = g.plan(M, N, K)
    T, KB = info["tiles"], info["k_blocks"]
    C = info["grid_ctas"] // cta_group
    assert T < C == max_ctas // cta_group and info["sk_tiles"] == T
    # tails are reckoned slower than heads, so a head is at least the even share
    assert -(-T * KB // C) <= info["sk_head"] < KB
    assert info["sk_slots"] >= (C - T) * cta_group
    D = run_gpu(A, B, M, N, K, cta_group=cta_group, max_ctas=max_ctas, stream_k=3)
    check(D, A, B, M, N, K, exact=True)
    # whole tiles (stream_k = 0) and the partial-wave-only setting (2, which
    # leaves these tiles whole) give the same bits
    for sk in (0, 2):
        with binding.Gemm(0, cta_group=cta_group, max_ctas=max_ctas, stream_k=sk) as g:
            assert g.plan(M, N, K)["sk_head"] == 0
        D0 = run_gpu(A, B, M, N, K, cta_group=cta_group, max_ctas=max_ctas, stream_k=sk)
        assert torch.equal(D.view(torch.int16), D0.view(torch.int16))


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("sched", SCHEDULES + [dict(acc_buffers=1), dict(acc_buffers=1, scheduler=1)])
def test_schedules_with_head_tail_split(cta_group, sched):
    # the owner folds the tails' partials into its spare accumulator only with
    # the cooperative epilogue and two accumulators; otherwise after its MMAs
    M, N, K, max_ctas = 600, 700, 8200, 20
    A, B = inputs.make_problem(M, N, K, "int2", seed=41)
    with binding.Gemm(0, cta_group=cta_group, max_ctas=max_ctas, stream_k=3, **sched) as g:
        assert g.plan(M, N, K)["sk_head"] > 0
    D = run_gpu(A, B, M, N, K, cta_group=cta_group, max_ctas=max_ctas, stream_k=3, **sched)
    check(D, A, B, M, N, K, exact=True)


def test_head_tail_random_inputs_repeated_launches_and_full_grid():
    # 2048 x 2048 x 32768 on the whole GPU (64 SM-pair tiles): launches on one
    # handle reuse every partial slot, each with its own epoch
    M, N, K = 2048, 2048, 32768
    A, B = inputs.make_problem(M, N, K, "normal", seed=4)
    A[:, ::97] *= 0.5  # not the longk workload's exact values
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    outs = []
    with binding.Gemm(0) as g:
        info = g.plan(M, N, K)
        assert info["sk_head"] > 0 and info["sk_tiles"] == info["tiles"]
        for i in range(3):
            D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            g.run(dA if i != 1 else dA * 2, dB, D)
            outs.append(D)
        assert g.device_status()[0] == binding.OK
    torch.cuda.synchronize()
    rows = sample_rows(M, extra=8)
    check(outs[0].cpu(), A, B, M, N, K, rows=rows)
    assert torch.equal(outs[2].view(torch.int16), outs[0].view(torch.int16))
    assert torch.equal(outs[1].cpu().float(), (outs[0].cpu().float() * 2))


@pytest.mark.parametrize("M,N,K,split", [
    (2048, 2048, 32768, True),    # 64 tiles, long k: the split pays (measured)
    (1024, 1024, 32768, True),    # 16 tiles
    (512, 512, 16384, True),      # 4 tiles
    (1024, 1024, 4096, True),     # 16 tiles of 64 k-blocks
    (2048, 2048, 8192, False),    # 64 tiles, short tails: the fixed cost of a split wins
    (256, 256, 256, False),
    (4096, 4096, 4096, False),    # more tiles than SM pairs: the partial-wave split instead
])
def test_head_tail_automatic_choice(M, N, K, split):
    with binding.Gemm(0) as g:
        info = g.plan(M, N, K)
    assert (info["sk_head"] > 0) == split, info
    if split:
        assert info["grid_ctas"] // info["cta_group"] > info["tiles"] == info["sk_tiles"]
    elif info["tiles"] * info["cta_group"] < info["num_sms"]:
        assert info["sk_tiles"] == 0 and info["grid_ctas"] == info["tiles"] * info["cta_group"]


def test_head_tail_fused_epilogue_exact():
    M, N, K, max_ctas = 600, 520, 8192, 20
    A, B = inputs.make_problem(M, N, K, "int2", seed=43)
    g = torch.Generator().manual_seed(44)
    C = inputs.make_operand(M, N, None, "int2", g)
    bias = inputs.make_operand(1, N, None, "int2", g).reshape(-1)
    with binding.Gemm(0, max_ctas=max_ctas, stream_k=3) as h:
        assert h.plan(M, N, K)["sk_head"] > 0
    D = run_fused_gpu(A, B, M, N, K, C=C, bias=bias, alpha=2.0, beta=-3.0, max_ctas=max_ctas, stream_k=3)
    _, refbf = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 2.0, -3.0, C=inputs.bits(C),
                                      bias=inputs.bits(bias))
    assert np.array_equal(inputs.bits(D), refbf)


def test_head_tail_watchdog_timeout_then_exact():
    # a skipped load stalls a tail range; its owner's wait for the partial is
    # bounded too, and the next launch on the handle (a new epoch) is exact
    M, N, K, max_ctas = 512, 512, 8192, 12
    A, B = inputs.make_problem(M, N, K, "int2", seed=45)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0, watchdog_ns=20_000_000, fault_skip_load=5, max_ctas=max_ctas, stream_k=3) as g:
        assert g.plan(M, N, K)["sk_head"] > 0
        g.run(dA, dB, dD)
        st, detail = g.device_status()
        assert st == binding.ERR_DEVICE_TIMEOUT and detail & 0x80000000
        g.set_option("fault_skip_load", -1)
        g.plan(M, N, K)
        for _ in range(2):
            dD.fill_(3.0)
            g.run(dA, dB, dD)
            assert g.device_status()[0] == binding.OK
            check(dD.cpu(), A, B, M, N, K, exact=True)


@pytest.mark.parametrize("N,epilogue,ldd", [
    (517, 0, 520), (517, 1, 520), (517, 2, 520), (517, 0, 523), (517, 2, 528), (517, 1, 600),
    (512, 1, 520), (520, 1, 600), (64, 1, 72), (1, 2, 1), (7, 0, 8)])
def test_epilogue_paths_and_padding(N, epilogue, ldd):
    # padding columns n >= N keep their sentinel on every path
    M, K = 333, 96
    A, B = inputs.make_problem(M, N, K, "normal", seed=5)
    D = run_gpu(A, B, M, N, K, ldd=ldd, epilogue=epilogue)
    check(D, A, B, M, N, K)


@pytest.mark.parametrize("serpentine", [0, 1])
@pytest.mark.parametrize("raster_group", [0, 1, 3, 8, 64])
def test_raster_orders(raster_group, serpentine):
    M, N, K = 1536, 1280, 128
    A, B = inputs.make_problem(M, N, K, "int2", seed=3)
    D = run_gpu(A, B, M, N, K, raster_group=raster_group, serpentine=serpentine, max_ctas=10)
    check(D, A, B, M, N, K, exact=True)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_serpentine_with_stream_k_and_pipelines(cta_group):
    # odd bands reversed, split tiles, ragged edges; and the ablation loops
    M, N, K = 2000, 1800, 700
    A, B = inputs.make_problem(M, N, K, "int2", seed=13, lda=pad8(K), ldb=pad8(K))
    check(run_gpu(A, B, M, N, K, serpentine=1, raster_group=2, max_ctas=14, cta_group=cta_group),
          A, B, M, N, K, exact=True)
    check(run_gpu(A, B, M, N, K, serpentine=1, raster_group=2, pipeline=binding.PIPE_MBAR_WAR),
          A, B, M, N, K, exact=True)


def test_identity_and_permutation_full_tiles():
    # B = I gives D = A bit for bit; A = P gives D[m, n] = B[n, perm[m]]
    K = 1024
    g = torch.Generator().manual_seed(9)
    A = inputs.make_operand(768, K, None, "normal", g)
    eye = torch.eye(K, dtype=torch.bfloat16)
    D = run_gpu(A, eye, 768, K, K)
    assert torch.equal(D.view(torch.int16), A.view(torch.int16))
    perm = torch.randperm(K, generator=g)
    P = torch.zeros((K, K), dtype=torch.bfloat16)
    P[torch.arange(K), perm] = 1.0
    Bm = inputs.make_operand(640, K, None, "uniform", g)
    D2 = run_gpu(P, Bm, K, 640, K)
    assert torch.equal(D2.view(torch.int16), Bm[:, perm].t().contiguous().view(torch.int16))


# ------------------------------------------------------------------ the five workloads
def every_element(D, A, B, M, N, K, exact=False, band=1024):
    """Every element of D against the oracle, computed in bands of rows (the
    oracle's fp64 sums of one band at a time): the tolerance count, the exact
    matches against the oracle's bf16 rounding and the ulp histogram.  With
    `exact`, every element must equal the oracle's bf16 rounding bit for bit.
    Padding columns n >= N must keep their sentinel."""
    Ab, Bb = inputs.bits(A), inputs.bits(B)
    Dbits = inputs.bits(D)
    scale = math.sqrt(K) * rms(A, K) * rms(B, K)
    st = {"elements": 0, "over_tolerance": 0, "mismatches": 0, "max_abs_err": 0.0, "max_err_over_tol": 0.0,
          "ulp_hist": {"0": 0, "1": 0, "2": 0, "3+": 0}, "max_ulp_away_from_zero": 0}
    first_bad = None
    for r0 in range(0, M, band):
        rows = np.arange(r0, min(M, r0 + band), dtype=np.int64)
        ref64, refbf = oracle.gemm_rows(Ab, Bb, K=K, rows=rows)
        got_bits = np.ascontiguousarray(Dbits[r0:r0 + rows.size, :N])
        got = inputs.from_bits(got_bits).double().numpy()
        tol = 4e-3 * np.abs(ref64) + 2e-3 * scale
        err = np.abs(got - ref64)
        over = ~(err <= tol)
        mism = got_bits != refbf
        if first_bad is None and (over.any() or (exact and mism.any())):
            idx = np.argwhere(over | (mism if exact else over))[0]
            first_bad = (int(r0 + idx[0]), int(idx[1]))
        ulp = np.abs(_ordered(got_bits) - _ordered(refbf))
        big = np.abs(ref64) >= 0.25 * scale  # a quarter of the typical magnitude or more
        st["elements"] += int(err.size)
        st["over_tolerance"] += int(over.sum())
        st["mismatches"] += int(mism.sum())
        st["max_abs_err"] = max(st["max_abs_err"], float(err.max()))
        st["max_err_over_tol"] = max(st["max_err_over_tol"], float((err / tol).max()))
        for k in (0, 1, 2):
            st["ulp_hist"][str(k)] += int((ulp == k).sum())
        st["ulp_hist"]["3+"] += int((ulp >= 3).sum())
        if big.any():
            st["max_ulp_away_from_zero"] = max(st["max_ulp_away_from_zero"], int(ulp[big].max()))
    st["exact_frac"] = st["ulp_hist"]["0"] / max(st["elements"], 1)
    st["first_bad"] = first_bad
    assert st["elements"] == M * N
    assert st["over_tolerance"] == 0, f"{st['over_tolerance']} elements outside tolerance, first {first_bad}"
    if exact:
        assert st["mismatches"] == 0, f"{st['mismatches']} mismatches, first at {first_bad}"
    if Dbits.shape[1] > N:
        assert np.all(Dbits[:, N:] == SENTINEL_BITS)
    return st


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_every_element(name):
    # the full-size workload in the launch configuration bench.py times, every
    # element of D against the oracle
    w = inputs.WORKLOADS[name]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.make_workload(name)
    D = run_gpu(A, B, M, N, K)
    st = every_element(D, A, B, M, N, K)
    print(f"parity {name}: {st}")
    # away from zero the fp32 sum is far closer than a bf16 ulp to the exact
    # one, so the result is the oracle's rounding or its neighbour
    assert st["max_ulp_away_from_zero"] <= 1


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_integer_inputs_exact(name):
    # same shapes and launch configuration, integer-valued inputs: every fp32
    # partial sum is exact, so every element must be the oracle's bit for bit
    w = inputs.WORKLOADS[name]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.make_problem(M, N, K, "int2", seed=w["seed"] + 100)
    D = run_gpu(A, B, M, N, K)
    every_element(D, A, B, M, N, K, exact=True)


def test_ragged_padded_ldd_uses_tma_store():
    w = inputs.WORKLOADS["ragged"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = inputs.make_workload("ragged")
    D = run_gpu(A, B, M, N, K, ldd=6000, epilogue=1)
    every_element(D, A, B, M, N, K)


def test_all_ones_full_size_property():
    # every entry of D is exactly K (K <= 256 keeps it representable in bf16)
    M, N, K = 4096, 4096, 256
    A = torch.ones((M, K), dtype=torch.bfloat16)
    D = run_gpu(A, A, M, N, K)
    assert torch.all(D.float() == K)


# ------------------------------------------------------------------ boundary behaviour
def test_run_before_plan_and_bad_pointers():
    dev = torch.device("cuda:0")
    buf = torch.zeros(4096, dtype=torch.bfloat16, device=dev)
    st, h = binding.gemm_bf16_create(0)
    assert st == binding.OK
    try:
        p = buf.data_ptr()
        assert binding.gemm_bf16_run(h, p, p, p) == binding.ERR_NOT_PLANNED
        assert binding.gemm_bf16_plan(h, 16, 16, 16, 16, 16, 16) == binding.OK
        assert binding.gemm_bf16_run(h, p + 2, p, p) == binding.ERR_ALIGNMENT
        assert binding.gemm_bf16_run(h, p, p + 8, p) == binding.ERR_ALIGNMENT
        assert binding.gemm_bf16_run(h, p, p, p + 1) == binding.ERR_ALIGNMENT
        assert binding.gemm_bf16_run(h, 0, p, p) == binding.ERR_INVALID_ARG
        assert binding.gemm_bf16_set_option(h, 99, 0) == binding.ERR_INVALID_ARG
        assert binding.gemm_bf16_set_option(h, binding.OPTIONS["stages"], 99) == binding.ERR_INVALID_ARG
        # forcing the TMA-store epilogue on an odd ldd is refused before launch
        assert binding.gemm_bf16_set_option(h, binding.OPTIONS["epilogue"], 1) == binding.OK
        assert binding.gemm_bf16_plan(h, 16, 15, 16, 16, 16, 15) == binding.OK
        assert binding.gemm_bf16_run(h, p, p, p) == binding.ERR_ALIGNMENT
        # the ablation loops are single-CTA only
        assert binding.gemm_bf16_set_option(h, binding.OPTIONS["pipeline"], binding.PIPE_SYNC_WAR) == binding.OK
        assert binding.gemm_bf16_set_option(h, binding.OPTIONS["cta_group"], 2) == binding.OK
        assert binding.gemm_bf16_plan(h, 16, 16, 16, 16, 16, 16) == binding.ERR_UNSUPPORTED
    finally:
        torch.cuda.synchronize()
        binding.gemm_bf16_destroy(h)


def test_handles_with_different_ring_depths_interleave():
    # the kernel's shared-memory limit is per function: plans of one handle must
    # not stop another handle's deeper ring from launching
    M, N, K = 512, 768, 256
    A, B = inputs.make_problem(M, N, K, "int2", seed=31)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    deep = binding.Gemm(0)
    deep.plan(M, N, K)
    shallow = binding.Gemm(0, stages=3)
    shallow.plan(M, N, K)
    one = binding.Gemm(0, cta_group=1, stages=2)
    one.plan(M, N, K)
    try:
        for _ in range(2):
            deep.run(dA, dB, outs[0])
            shallow.run(dA, dB, outs[1])
            one.run(dA, dB, outs[2])
        for g in (deep, shallow, one):
            assert g.device_status()[0] == binding.OK
        torch.cuda.synchronize()
        for o in outs:
            check(o.cpu(), A, B, M, N, K, exact=True)
    finally:
        for g in (deep, shallow, one):
            g.close()


@pytest.mark.parametrize("pdl", [0, 1])
def test_chained_gemms_on_one_stream_respect_order(pdl):
    # D1 = A B^T, then D2 = D1 C^T and D3 = D2-free overwrite of D1, all
    # enqueued back to back: with programmatic dependent launch each kernel's
    # global accesses must still wait for the previous kernel.  Integer inputs
    # keep both stages exact.
    M, N, K, P = 768, 512, 64, 640
    A, B = inputs.make_problem(M, N, K, "int2", seed=41)
    g2 = torch.Generator().manual_seed(42)
    C = inputs.make_operand(P, N, None, "int2", g2)
    dev = torch.device("cuda:0")
    dA, dB, dC = A.to(dev), B.to(dev), C.to(dev)
    D1 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    D2 = torch.empty((M, P), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0, pdl=pdl) as g1, binding.Gemm(0, pdl=pdl) as g2h:
        g1.plan(M, N, K)
        g2h.plan(M, P, N)
        for _ in range(5):
            g1.run(dA, dB, D1)
            g2h.run(D1, dC, D2)
            D1.zero_()            # a plain kernel between our launches
            g1.run(dA, dB, D1)
        assert g1.device_status()[0] == binding.OK and g2h.device_status()[0] == binding.OK
    torch.cuda.synchronize()
    _, d1_ref = oracle.gemm_rows(inputs.bits(A), inputs.bits(B))
    assert np.array_equal(inputs.bits(D1.cpu()), d1_ref)
    _, d2_ref = oracle.gemm_rows(d1_ref, inputs.bits(C))
    assert np.array_equal(inputs.bits(D2.cpu()), d2_ref)


def test_cuda_graph_capture_and_replay():
    # plan outside the capture (it may allocate); run() only enqueues a launch
    M, N, K = 2048, 1536, 1024
    dev = torch.device("cuda:0")
    A, B = inputs.make_problem(M, N, K, "int2", seed=51)
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0) as g:
        g.plan(M, N, K)
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            g.run(dA, dB, dD)          # warm-up outside the capture
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.run(dA, dB, dD)
        dD.zero_()
        dA.copy_(A.to(dev) * -1)       # new inputs, same buffers
        graph.replay()
        torch.cuda.synchronize(dev)
        assert g.device_status()[0] == binding.OK
    check(dD.cpu(), (A.float() * -1).to(torch.bfloat16), B, M, N, K, exact=True)


@pytest.mark.parametrize("M,N,K,what,opts", [
    (4096, 4096, 1024, "partial-wave split", {}),   # 256 tiles: 28 split tiles share flags
    (1024, 1024, 32768, "head/tail split", {}),     # 16 tiles, tails on the idle SM pairs
    (16, 8192, 8192, "thin kernel", {}),            # split tiles of the thin kernel
    (4096, 4096, 1024, "dynamic tile counter", {"scheduler": 1}),
    (4096, 4096, 1024, "ping-pong epilogue", {"epi_schedule": 1}),
])
def test_cuda_graph_replays_with_new_inputs(M, N, K, what, opts):
    # A captured launch keeps the epoch it was captured with; its split tiles'
    # flags must still mean "written by this replay" on every replay.
    dev = torch.device("cuda:0")
    gens = [inputs.make_problem(M, N, K, "int2", seed=60 + i) for i in range(3)]
    dA = torch.empty_like(gens[0][0], device=dev)
    dB = torch.empty_like(gens[0][1], device=dev)
    dD = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0, **opts) as g:
        info = g.plan(M, N, K)
        assert info["sk_tiles"] > 0 or info["thin"] > 0, (what, info)
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        dA.copy_(gens[0][0])
        dB.copy_(gens[0][1])
        with torch.cuda.stream(s):
            g.run(dA, dB, dD)          # warm-up outside the capture
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.run(dA, dB, dD)
        for A, B in gens + gens[:1]:
            dA.copy_(A)
            dB.copy_(B)
            dD.zero_()
            graph.replay()
            torch.cuda.synchronize(dev)
            assert g.device_status()[0] == binding.OK
            check(dD.cpu(), A, B, M, N, K, exact=True)


@pytest.mark.parametrize("M,N,K", [(1 << 20, 384, 128), (256, 1 << 19, 64)])
def test_very_large_m_or_n(M, N, K):
    A, B = inputs.make_problem(M, N, K, "int2", seed=61)
    D = run_gpu(A, B, M, N, K)
    rows = np.array([0, 1, 255, 256, M // 2 + 7, M - 129, M - 1])
    rows = rows[rows < M]
    check(D, A, B, M, N, K, rows=rows, exact=True)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_very_long_k(cta_group):
    # 16,385 k-blocks in one tile, the last holding 8 valid columns: every fp32
    # partial sum of integers in [-2, 2] stays below 2^24, so the result is exact
    M, N, K = 130, 130, (1 << 20) + 8
    A, B = inputs.make_problem(M, N, K, "int2", seed=67)
    D = run_gpu(A, B, M, N, K, cta_group=cta_group)
    check(D, A, B, M, N, K, rows=np.array([0, 1, 63, 127, 128, 129]), exact=True)


def run_fused_gpu(A, B, M, N, K, C=None, bias=None, alpha=1.0, beta=0.0, ldd=None, inplace=False, **opts):
    ldd = N if ldd is None else ldd
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    if inplace:
        dD = C.to(dev).clone()
        dC = dD
    else:
        dD = torch.full((M, ldd), SENTINEL_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
        dC = None if C is None else C.to(dev)
    dbias = None if bias is None else bias.to(dev)
    with binding.Gemm(0, **opts) as g:
        g.plan(M, N, K, A.shape[1], B.shape[1], ldd)
        g.run_fused(dA, dB, dD, dC, dbias, alpha, beta)
        assert g.device_status()[0] == binding.OK
    torch.cuda.synchronize()
    return dD.cpu()


@pytest.mark.parametrize("variant", [dict(), dict(cta_group=1), dict(max_ctas=14),
                                     dict(max_ctas=14, epi_schedule=1, scheduler=1),
                                     dict(pipeline=binding.PIPE_MBAR_WAR), dict(epilogue=2)])
def test_fused_epilogue_exact_integers(variant):
    M, N, K = 1100, 900, 2560
    A, B = inputs.make_problem(M, N, K, "int2", seed=71)
    g = torch.Generator().manual_seed(72)
    C = inputs.make_operand(M, N, None, "int2", g)
    bias = inputs.make_operand(1, N, None, "int2", g).reshape(-1)
    D = run_fused_gpu(A, B, M, N, K, C=C, bias=bias, alpha=2.0, beta=-3.0, **variant)
    _, refbf = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 2.0, -3.0, C=inputs.bits(C),
                                      bias=inputs.bits(bias))
    assert np.array_equal(inputs.bits(D), refbf)


@pytest.mark.parametrize("case", ["all", "c_only", "bias_only", "alpha_only", "odd_ldc", "inplace"])
def test_fused_epilogue_random_values(case):
    M, N, K = 777, 520, 1000
    A, B = inputs.make_problem(M, N, K, "normal", seed=73)
    g = torch.Generator().manual_seed(74)
    ldc = 523 if case == "odd_ldc" else N
    C = inputs.make_operand(M, N, ldc, "normal", g) if case in ("all", "c_only", "odd_ldc", "inplace") else None
    bias = inputs.make_operand(1, N, None, "uniform", g).reshape(-1) if case in ("all", "bias_only") else None
    alpha = float(np.float32(0.625 if case != "alpha_only" else -1.375))
    beta = float(np.float32(1.25))
    D = run_fused_gpu(A, B, M, N, K, C=C, bias=bias, alpha=alpha, beta=beta,
                      ldd=ldc if case == "inplace" else None, inplace=(case == "inplace"))
    ref64, _ = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), alpha, beta,
                                      C=None if C is None else inputs.bits(C),
                                      bias=None if bias is None else inputs.bits(bias))
    got = D[:, :N].double().numpy()
    tol = (4e-3 * np.abs(ref64) + 2e-3 * math.sqrt(K) * rms(A, K) * rms(B, K) * abs(alpha) + 1e-6)
    assert np.all(np.abs(got - ref64) <= tol)
    if case == "inplace":
        # columns beyond N keep C's own values
        assert torch.equal(D[:, N:].view(torch.int16), C[:, N:].view(torch.int16))


def test_fused_rejects_bad_arguments():
    dev = torch.device("cuda:0")
    buf = torch.zeros(1 << 16, dtype=torch.bfloat16, device=dev)
    p = buf.data_ptr()
    st, h = binding.gemm_bf16_create(0)
    try:
        assert binding.gemm_bf16_run_fused(h, p, p, p, p, 16, 0, 1.0, 1.0) == binding.ERR_NOT_PLANNED
        assert binding.gemm_bf16_plan(h, 16, 16, 16, 16, 16, 16) == binding.OK
        assert binding.gemm_bf16_run_fused(h, p, p, p, p, 8, 0, 1.0, 1.0) == binding.ERR_INVALID_ARG
        assert binding.gemm_bf16_run_fused(h, p, p, p, p + 1, 16, 0, 1.0, 1.0) == binding.ERR_ALIGNMENT
        assert binding.gemm_bf16_run_fused(h, p, p, p, 0, 0, p + 1, 1.0, 1.0) == binding.ERR_ALIGNMENT
    finally:
        torch.cuda.synchronize()
        binding.gemm_bf16_destroy(h)


def test_plan_info_reports_the_configuration():
    with binding.Gemm(0) as g:
        info = g.plan(8192, 8192, 8192)
        assert info["cta_group"] == 2 and info["tile_m"] == 256 and info["tile_n"] == 256
        assert info["tiles"] == 32 * 32 and info["k_blocks"] == 128
        assert info["grid_ctas"] % 2 == 0 and info["grid_ctas"] <= info["num_sms"]
        assert info["stages"] >= 4 and info["acc_buffers"] == 2
        assert info["regs_per_thread"] * info["threads_per_cta"] <= 65536


@pytest.mark.parametrize("variant", [dict(cta_group=1), dict(cta_group=2),
                                     dict(pipeline=binding.PIPE_MBAR_WAR)])
def test_watchdog_reports_timeout_and_context_survives(variant):
    # the producer skips one load: the MMA warp's bounded wait runs out, the
    # kernel returns early with a status word instead of hanging
    M, N, K = 512, 512, 1024
    A, B = inputs.make_problem(M, N, K, "normal", seed=2)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0, watchdog_ns=20_000_000, fault_skip_load=3, **variant) as g:
        g.plan(M, N, K)
        g.run(dA, dB, dD)
        st, detail = g.device_status()
        assert st == binding.ERR_DEVICE_TIMEOUT
        assert detail & 0x80000000
    torch.cuda.synchronize()
    # the context is still usable: a normal run afterwards is correct
    check(run_gpu(A, B, M, N, K, **variant), A, B, M, N, K)


@pytest.mark.parametrize("stream_k", [0, 1])
def test_watchdog_limit_scales_with_k(stream_k):
    # 1 us asked for, but a wait for a whole tile's accumulator (1024 k-blocks,
    # ~0.3 ms) is legitimate: plan raises the limit to 2 us per k-block
    M, N, K = 512, 512, 65536
    A, B = inputs.make_problem(M, N, K, "int2", seed=81)
    D = run_gpu(A, B, M, N, K, watchdog_ns=1000, stream_k=stream_k)
    check(D, A, B, M, N, K, rows=sample_rows(M, extra=4), exact=True)


def test_tensormap_failure_is_reported_before_launch():
    # an encode failure (forced by the test hook) comes back as TENSORMAP and
    # launches nothing; the handle works again once the hook is off
    M, N, K = 300, 260, 200
    A, B = inputs.make_problem(M, N, K, "int2", seed=83, lda=pad8(K), ldb=pad8(K))
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.full((M, N), SENTINEL_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
    with binding.Gemm(0, fault_tensormap=1) as g:
        g.plan(M, N, K, pad8(K), pad8(K), N)
        for _ in range(2):
            with pytest.raises(binding.GemmError) as e:
                g.run(dA, dB, dD)
            assert e.value.status == binding.ERR_TENSORMAP
        torch.cuda.synchronize()
        assert bool((dD.view(torch.int16) == SENTINEL_BITS).all())
        assert g.device_status()[0] == binding.OK
        g.set_option("fault_tensormap", 0)
        g.run(dA, dB, dD)
        assert g.device_status()[0] == binding.OK
    torch.cuda.synchronize()
    check(dD.cpu(), A, B, M, N, K, exact=True)


@pytest.mark.parametrize("K,padded_ab,ldd", [(300, True, 600), (296, False, 608), (296, False, 600)])
def test_run_host_end_to_end(K, padded_ab, ldd):
    # padded rows take a pitched copy, contiguous rows one linear copy; padding
    # columns of D are not copied back (the host keeps its sentinel there)
    M, N = 700, 600
    ld = pad8(K) + 8 if padded_ab else K
    A, B = inputs.make_problem(M, N, K, "normal", seed=4, lda=ld, ldb=ld)
    hA, hB = A.pin_memory(), B.pin_memory()
    hD = torch.full((M, ldd), SENTINEL_BITS, dtype=torch.int16).view(torch.bfloat16).pin_memory()
    dev = torch.device("cuda:0")
    dA = torch.empty_like(A, device=dev)
    dB = torch.empty_like(B, device=dev)
    dD = torch.empty((M, ldd), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0) as g:
        g.plan(M, N, K, ld, ld, ldd)
        g.run_host(hA, hB, hD, dA, dB, dD)
        torch.cuda.synchronize()
        assert g.device_status()[0] == binding.OK
    check(hD, A, B, M, N, K)


def test_gemm_convenience_matches_oracle():
    A, B = inputs.make_problem(384, 640, 320, "uniform", seed=8)
    D = binding.gemm(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    check(D.cpu(), A, B, 384, 640, 320)


# ------------------------------------------------------------------ random shapes and options
def _random_case(i: int):
    rng = np.random.default_rng(1000 + i)
    logu = lambda lo, hi: int(round(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
    if i % 2 == 0:  # edge-heavy: many tiny and thin shapes
        M, N = logu(1, 3000), logu(1, 3000)
    else:  # several tiles, where the k splits happen
        M, N = int(rng.integers(200, 3001)), int(rng.integers(200, 3001))
    K = 8 * logu(1, 2048)
    opts = dict(cta_group=int(rng.integers(0, 3)), stream_k=int(rng.integers(0, 4)),
                epi_schedule=int(rng.integers(0, 2)), scheduler=int(rng.integers(0, 2)),
                k_order=int(rng.integers(0, 2)))
    if rng.random() < 0.5:
        opts["max_ctas"] = 2 * int(rng.integers(1, 21))
    ldd = N + (int(rng.integers(1, 10)) if rng.random() < 0.3 else 0)
    pad = 8 * int(rng.integers(1, 4)) if rng.random() < 0.3 else 0
    return M, N, K, ldd, pad, opts


@pytest.mark.parametrize("i", range(64))
def test_random_shapes_and_options_exact(i):
    # integer inputs keep every fp32 partial sum exact, so any split of k, any
    # schedule and any tile order must give the oracle's bits
    M, N, K, ldd, pad, opts = _random_case(i)
    A, B = inputs.make_problem(M, N, K, "int2", seed=2000 + i, lda=K + pad, ldb=K + pad)
    with binding.Gemm(0, **opts) as g:
        info = g.plan(M, N, K, K + pad, K + pad, ldd)
    if opts["stream_k"] == 0:
        assert info["sk_tiles"] == 0 and info["sk_head"] == 0
    if opts["stream_k"] == 2:
        assert info["sk_head"] == 0
    clusters = info["grid_ctas"] // info["cta_group"]
    if info["sk_head"]:
        assert info["sk_tiles"] == info["tiles"] < clusters and 0 < info["sk_head"] < info["k_blocks"]
    D = run_gpu(A, B, M, N, K, ldd=ldd, **opts)
    check(D, A, B, M, N, K, rows=sample_rows(M, extra=8, seed=i), exact=True)


def test_binding_rejects_tensors_off_the_handles_device():
    # the library dereferences raw pointers on the handle's device only; the
    # binding refuses host tensors for run() and device tensors as run_host's
    # host side before anything reaches the library
    M, N, K = 64, 64, 64
    A, B = inputs.make_problem(M, N, K, "int2", seed=87)
    dev = torch.device("cuda:0")
    dA, dB = A.to(dev), B.to(dev)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    with binding.Gemm(0) as g:
        assert g.device == 0
        g.plan(M, N, K)
        with pytest.raises(ValueError):
            g.run(A, dB, dD)
        with pytest.raises(ValueError):
            g.run_host(dA, B, torch.empty((M, N), dtype=torch.bfloat16), dA, dB, dD)
        g.run(dA, dB, dD)
        assert g.device_status()[0] == binding.OK
    torch.cuda.synchronize()
    check(dD.cpu(), A, B, M, N, K, exact=True)

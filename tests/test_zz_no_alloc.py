"""The allocation-free entry point, for callers that cannot allocate device
memory (pool-owned memory, loops that cannot afford an allocation).

gemm_bf16_run_noalloc must give the same D as gemm_bf16_run on the same
operands, within the tolerance the other GPU tests use, on two calls in a row
(the second call reuses the shared scratch array the first one left behind).
On integer-valued inputs every fp32 partial sum is exact, so there both entry
points must equal the oracle bit for bit on every element; that case has more
output tiles than SM pairs, so each SM pair walks several tiles (double-buffered
accumulators, alternating k direction, serpentine raster).  The status word
goes to page-locked host memory, which keeps its copy asynchronous; pageable
memory is refused.  This file is named to be collected last, so that a run
stopping at the first failure has already run every other test.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from warp_specialized_tma_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

SENTINEL_BITS = 0x7FC1


def _rms(t, K):
    return float(t[:, :K].double().pow(2).mean().sqrt())


def _with_handle(A, B, M, N, K, ldd, dev):
    D = torch.full((M, ldd), SENTINEL_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
    with binding.Gemm(dev.index) as g:
        g.plan(M, N, K, A.shape[1], B.shape[1], ldd)
        g.run(A, B, D)
        assert g.device_status()[0] == binding.OK
    return D


def _noalloc(A, B, M, N, K, ldd, dev):
    D = torch.full((M, ldd), SENTINEL_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
    status = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    st = binding.gemm_bf16_run_noalloc(M, N, K, A.shape[1], B.shape[1], ldd, A.data_ptr(), B.data_ptr(),
                                       D.data_ptr(), torch.cuda.current_stream(dev).cuda_stream,
                                       status.data_ptr())
    assert st == binding.OK, binding.gemm_bf16_strerror(st)
    torch.cuda.synchronize(dev)
    assert int(status[0]) == 0
    return D


@pytest.fixture(scope="module")
def dev():
    from warp_specialized_tma_gb300 import build as libbuild
    libbuild.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def test_noalloc_matches_the_handle_entry_point_twice(dev):
    cases = [(1000, 777, 520, 780, "normal", 11), (640, 1024, 256, 1024, "uniform", 12)]
    for (M, N, K, ldd, dist, seed) in cases:   # two calls in a row
        A, B = inputs.make_problem(M, N, K, dist, seed)
        dA, dB = A.to(dev), B.to(dev)
        ref = _with_handle(dA, dB, M, N, K, ldd, dev).cpu()
        got = _noalloc(dA, dB, M, N, K, ldd, dev).cpu()
        r = inputs.bits(ref).astype(np.int64)
        gbits = inputs.bits(got).astype(np.int64)
        # padding columns untouched by both
        assert np.all(gbits[:, N:] == SENTINEL_BITS) and np.all(r[:, N:] == SENTINEL_BITS)
        a = got[:, :N].double().numpy()
        b = ref[:, :N].double().numpy()
        tol = 4e-3 * np.abs(b) + 2e-3 * math.sqrt(K) * _rms(A, K) * _rms(B, K)
        assert np.all(np.abs(a - b) <= tol)
        # and against the oracle on every element
        ref64, _ = oracle.gemm_rows(inputs.bits(A), inputs.bits(B))
        tol_o = 4e-3 * np.abs(ref64) + 2e-3 * math.sqrt(K) * _rms(A, K) * _rms(B, K)
        assert np.all(np.abs(a - ref64) <= tol_o)


def test_noalloc_integer_inputs_exact_with_many_tiles_per_sm_pair(dev):
    # 11 x 10 = 110 tiles of 256 x 256 against at most 76 SM pairs: every pair
    # walks a second tile; ragged M and N, a k tail, and TMA-stored D
    M, N, K = 2600, 2504, 1000
    A, B = inputs.make_problem(M, N, K, "int2", seed=41)
    dA, dB = A.to(dev), B.to(dev)
    _, refbf = oracle.gemm_rows(inputs.bits(A), inputs.bits(B))
    for _ in range(2):   # two calls in a row on the shared scratch
        got = inputs.bits(_noalloc(dA, dB, M, N, K, N, dev).cpu())
        bad = np.argwhere(got != refbf)
        assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"
    hnd = inputs.bits(_with_handle(dA, dB, M, N, K, N, dev).cpu())
    assert np.array_equal(hnd, got)


def test_noalloc_rejects_bad_arguments_before_launch(dev):
    buf = torch.zeros(4096, dtype=torch.bfloat16, device=dev)
    p = buf.data_ptr()
    assert binding.gemm_bf16_run_noalloc(0, 8, 8, 8, 8, 8, p, p, p) == binding.ERR_INVALID_ARG
    assert binding.gemm_bf16_run_noalloc(8, 8, 12, 12, 16, 8, p, p, p) == binding.ERR_ALIGNMENT
    assert binding.gemm_bf16_run_noalloc(8, 8, 8, 8, 8, 8, p + 2, p, p) == binding.ERR_ALIGNMENT
    assert binding.gemm_bf16_run_noalloc(8, 8, 8, 8, 8, 8, 0, p, p) == binding.ERR_INVALID_ARG
    # a pageable status word would make the call block until the GEMM is done
    pageable = ctypes.c_uint32(0xFFFFFFFF)
    assert binding.gemm_bf16_run_noalloc(8, 8, 8, 8, 8, 8, p, p, p,
                                         status=ctypes.addressof(pageable)) == binding.ERR_INVALID_ARG
    assert pageable.value == 0xFFFFFFFF
    # device memory is accepted
    word = torch.full((1,), -1, dtype=torch.int32, device=dev)
    assert binding.gemm_bf16_run_noalloc(8, 8, 8, 8, 8, 8, p, p, p, status=word.data_ptr()) == binding.OK
    torch.cuda.synchronize(dev)
    assert int(word.cpu()[0]) == 0

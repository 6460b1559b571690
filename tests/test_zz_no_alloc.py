"""The allocation-free entry point, for callers that cannot allocate device
memory (pool-owned memory, loops that cannot afford an allocation).

gemm_bf16_run_noalloc must give the same D as gemm_bf16_run on the same
operands, within the tolerance the other GPU tests use, on two calls in a row
(the second call reuses the shared scratch array the first one left behind).
This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
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
    status = ctypes.c_uint32(0xFFFFFFFF)
    st = binding.gemm_bf16_run_noalloc(M, N, K, A.shape[1], B.shape[1], ldd, A.data_ptr(), B.data_ptr(),
                                       D.data_ptr(), torch.cuda.current_stream(dev).cuda_stream, status)
    assert st == binding.OK, binding.gemm_bf16_strerror(st)
    torch.cuda.synchronize(dev)
    assert status.value == 0
    return D


def test_noalloc_matches_the_handle_entry_point_twice():
    from warp_specialized_tma_gb300 import build as libbuild
    libbuild.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
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
        # and both agree with the oracle on a few rows
        rows = [0, M // 2, M - 1]
        ref64, _ = oracle.gemm_rows(inputs.bits(A), inputs.bits(B), rows=rows)
        tol_o = 4e-3 * np.abs(ref64) + 2e-3 * math.sqrt(K) * _rms(A, K) * _rms(B, K)
        assert np.all(np.abs(a[rows] - ref64) <= tol_o)


def test_noalloc_rejects_bad_arguments_before_launch():
    dev = torch.device("cuda:0")
    buf = torch.zeros(4096, dtype=torch.bfloat16, device=dev)
    p = buf.data_ptr()
    assert binding.gemm_bf16_run_noalloc(0, 8, 8, 8, 8, 8, p, p, p) == binding.ERR_INVALID_ARG
    assert binding.gemm_bf16_run_noalloc(8, 8, 12, 12, 16, 8, p, p, p) == binding.ERR_ALIGNMENT
    assert binding.gemm_bf16_run_noalloc(8, 8, 8, 8, 8, 8, p + 2, p, p) == binding.ERR_ALIGNMENT
    assert binding.gemm_bf16_run_noalloc(8, 8, 8, 8, 8, 8, 0, p, p) == binding.ERR_INVALID_ARG

"""CPU oracle for D = A * B^T over bf16 operands -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline
leg and its reference arm) may import this package.  The product library under
``warp_specialized_tma_gb300/`` never imports it and shares no code with it.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64, one rounding to bf16
at the end); this module only builds it with gcc and marshals numpy arrays.
What it follows: Fuser issue #3941 "Allow separate sub-DAG for load and compute
warp groups with warp-specialized circular buffering", Pseudo-code (the compute
warp group sums the A/B tile products over cta-k, then converts the fp32 sums to
bf16 before the store).  Parity status: pinned (tests/test_oracle.py).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


_STAMP = _LIB + ".stamp"
_CMD = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def _stamp() -> str:
    """The source's sha256, the host architecture and the compiler command: a
    library built from other source or on another machine never matches."""
    with open(_SRC, "rb") as fh:
        digest = hashlib.sha256(fh.read()).hexdigest()
    return f"{digest} machine={platform.machine()} cmd={' '.join(_CMD)}"


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into liboracle.so (gcc, OpenMP, no fp contraction)."""
    if not force and os.path.exists(_LIB) and os.path.exists(_STAMP):
        with open(_STAMP) as fh:
            if fh.read().strip() == _stamp():
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(_CMD + ["-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    with open(_STAMP, "w") as fh:
        fh.write(_stamp())
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_gemm_rows.restype = ctypes.c_int
        lib.oracle_gemm_rows.argtypes = [u16p, ctypes.c_int64, u16p, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         i64p, ctypes.c_int64, f64p, u16p]
        lib.oracle_gemm_fused_rows.restype = ctypes.c_int
        lib.oracle_gemm_fused_rows.argtypes = [u16p, ctypes.c_int64, u16p, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               i64p, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                               u16p, ctypes.c_int64, u16p, f64p, u16p]
        lib.oracle_bf16_from_f64.restype = ctypes.c_uint16
        lib.oracle_bf16_from_f64.argtypes = [ctypes.c_double]
        lib.oracle_f64_from_bf16.restype = ctypes.c_double
        lib.oracle_f64_from_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_from_f64_array.restype = None
        lib.oracle_bf16_from_f64_array.argtypes = [f64p, u16p, ctypes.c_int64]
        lib.oracle_f64_from_bf16_array.restype = None
        lib.oracle_f64_from_bf16_array.argtypes = [u16p, f64p, ctypes.c_int64]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_set_threads.restype = None
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def gemm_rows(A: np.ndarray, B: np.ndarray, K: int | None = None, rows=None):
    """Rows of D = A * B^T.

    ``A`` is an (M, lda) uint16 array of bf16 patterns and ``B`` an (N, ldb)
    one; only the first ``K`` columns of each are read (default: all).
    ``rows`` selects m indices (default: all rows).  Returns ``(ref64, refbf16)``
    with shapes (len(rows), N): the fp64 sum and its single bf16 rounding.
    """
    lib = _load()
    A = np.ascontiguousarray(_u16(A))
    B = np.ascontiguousarray(_u16(B))
    if A.ndim != 2 or B.ndim != 2:
        raise ValueError("A and B must be 2-D")
    M, lda = A.shape
    N, ldb = B.shape
    K = min(lda, ldb) if K is None else int(K)
    if K > lda or K > ldb:
        raise ValueError("K exceeds a leading dimension")
    if rows is None:
        rows_arr = None
        nrows = M
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    ref64 = np.empty((nrows, N), dtype=np.float64)
    refbf16 = np.empty((nrows, N), dtype=np.uint16)
    rc = lib.oracle_gemm_rows(_ptr(A, ctypes.c_uint16), lda, _ptr(B, ctypes.c_uint16), ldb,
                              M, N, K,
                              None if rows_arr is None else _ptr(rows_arr, ctypes.c_int64),
                              nrows, _ptr(ref64, ctypes.c_double),
                              _ptr(refbf16, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle_gemm_rows rejected its arguments")
    return ref64, refbf16


def gemm_fused_rows(A: np.ndarray, B: np.ndarray, alpha: float, beta: float, C=None, bias=None,
                    K: int | None = None, rows=None):
    """Rows of D = alpha * (A * B^T) + beta * C + bias (bias broadcast over rows).

    ``C`` is an (M, ldc) uint16 array of bf16 patterns or None; ``bias`` an (N,)
    uint16 array or None; alpha and beta are the fp32 values the GPU receives
    (pass Python floats that are exactly fp32, e.g. via numpy.float32).
    Returns ``(ref64, refbf16)`` like :func:`gemm_rows`.
    """
    lib = _load()
    A = np.ascontiguousarray(_u16(A))
    B = np.ascontiguousarray(_u16(B))
    M, lda = A.shape
    N, ldb = B.shape
    K = min(lda, ldb) if K is None else int(K)
    if C is not None:
        C = np.ascontiguousarray(_u16(C))
        if C.shape[0] != M or C.shape[1] < N:
            raise ValueError("C must be M x ldc with ldc >= N")
        ldc = C.shape[1]
    else:
        ldc = 0
    if bias is not None:
        bias = np.ascontiguousarray(_u16(bias)).reshape(-1)
        if bias.size < N:
            raise ValueError("bias must have N entries")
    if rows is None:
        rows_arr = None
        nrows = M
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    ref64 = np.empty((nrows, N), dtype=np.float64)
    refbf16 = np.empty((nrows, N), dtype=np.uint16)
    rc = lib.oracle_gemm_fused_rows(
        _ptr(A, ctypes.c_uint16), lda, _ptr(B, ctypes.c_uint16), ldb, M, N, K,
        None if rows_arr is None else _ptr(rows_arr, ctypes.c_int64), nrows,
        float(alpha), float(beta),
        None if C is None else _ptr(C, ctypes.c_uint16), ldc,
        None if bias is None else _ptr(bias, ctypes.c_uint16),
        _ptr(ref64, ctypes.c_double), _ptr(refbf16, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle_gemm_fused_rows rejected its arguments")
    return ref64, refbf16


def bf16_from_f64(x) -> np.ndarray:
    """Round fp64 values to bf16 patterns (nearest, ties to even)."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_bf16_from_f64_array(_ptr(x, ctypes.c_double), _ptr(out, ctypes.c_uint16), x.size)
    return out


def f64_from_bf16(h) -> np.ndarray:
    """Widen bf16 patterns to fp64 (exact)."""
    lib = _load()
    h = np.ascontiguousarray(_u16(h))
    out = np.empty(h.shape, dtype=np.float64)
    lib.oracle_f64_from_bf16_array(_ptr(h, ctypes.c_uint16), _ptr(out, ctypes.c_double), h.size)
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))

"""Thin Python binding over the C ABI of ``include/gemm_bf16.h``.

Argument marshalling only: every step of the GEMM runs in ``libgemm_bf16.so``
(the CUDA kernels for sm_103a).  The functions named ``gemm_bf16_*`` mirror the
C entry points one to one and return the C status code; ``Gemm`` wraps a handle
for torch tensors and raises ``GemmError`` on a non-zero status.  There is no
fallback: if the library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgemm_bf16.so")

# status codes (gemm_bf16_status)
OK = 0
ERR_INVALID_ARG = -1
ERR_ALIGNMENT = -2
ERR_NOT_PLANNED = -3
ERR_CUDA = -4
ERR_TENSORMAP = -5
ERR_DEVICE_TIMEOUT = -6
ERR_UNSUPPORTED = -7

# pipelines (gemm_bf16_pipeline)
PIPE_WS = 0
PIPE_SYNC_WAR = 1
PIPE_MBAR_WAR = 2

# options (gemm_bf16_option)
OPTIONS = {
    "pipeline": 1,
    "cta_group": 2,
    "persistent": 3,
    "acc_buffers": 4,
    "setmaxnreg": 5,
    "stages": 6,
    "raster_group": 7,
    "epilogue": 8,
    "max_ctas": 9,
    "watchdog_ns": 10,
    "fault_skip_load": 11,
    "stage_group": 12,
    "stream_k": 13,
    "pdl": 14,
    "epi_schedule": 15,
    "scheduler": 16,
    "repack": 17,
    "k_order": 18,
    "serpentine": 19,
    "fault_tensormap": 20,
    "thin": 21,
    "thin_cluster": 22,
}

# the C entry points and their signatures
_H = ctypes.c_void_p
_SIGNATURES = {
    "gemm_bf16_create": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(_H)]),
    "gemm_bf16_destroy": (ctypes.c_int, [_H]),
    "gemm_bf16_set_option": (ctypes.c_int, [_H, ctypes.c_int, ctypes.c_int64]),
    "gemm_bf16_get_option": (ctypes.c_int, [_H, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]),
    "gemm_bf16_check_problem": (ctypes.c_int, [ctypes.c_int64] * 6),
    "gemm_bf16_plan": (ctypes.c_int, [_H] + [ctypes.c_int64] * 6),
    "gemm_bf16_plan_info": (ctypes.c_int, [_H, ctypes.c_void_p]),
    "gemm_bf16_run": (ctypes.c_int, [_H, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "gemm_bf16_run_host": (ctypes.c_int, [_H] + [ctypes.c_void_p] * 7),
    "gemm_bf16_run_fused": (ctypes.c_int, [_H, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                           ctypes.c_float, ctypes.c_float, ctypes.c_void_p]),
    "gemm_bf16_device_status": (ctypes.c_int, [_H, ctypes.POINTER(ctypes.c_uint32)]),
    "gemm_bf16_run_noalloc": (ctypes.c_int, [ctypes.c_int64] * 6 + [ctypes.c_void_p] * 5),
    "gemm_bf16_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "gemm_bf16_version": (ctypes.c_char_p, []),
}


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("tiles", ctypes.c_int64),
        ("k_blocks", ctypes.c_int64),
        ("grid_ctas", ctypes.c_int32),
        ("threads_per_cta", ctypes.c_int32),
        ("cta_group", ctypes.c_int32),
        ("pipeline", ctypes.c_int32),
        ("persistent", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("acc_buffers", ctypes.c_int32),
        ("setmaxnreg", ctypes.c_int32),
        ("tile_m", ctypes.c_int32),
        ("tile_n", ctypes.c_int32),
        ("tile_k", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("epilogue_tma_allowed", ctypes.c_int32),
        ("raster_group", ctypes.c_int32),
        ("regs_per_thread", ctypes.c_int32),
        ("stage_group", ctypes.c_int32),
        ("sk_tiles", ctypes.c_int32),
        ("epi_schedule", ctypes.c_int32),
        ("scheduler", ctypes.c_int32),
        ("repack", ctypes.c_int32),
        ("packed_ld", ctypes.c_int32),
        ("k_order", ctypes.c_int32),
        ("serpentine", ctypes.c_int32),
        ("sk_head", ctypes.c_int32),
        ("sk_slots", ctypes.c_int32),
        ("thin", ctypes.c_int32),
        ("thin_cluster", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {gemm_bf16_strerror(status)} (status {status})")


_lib = None
_lock = threading.Lock()


def load() -> ctypes.CDLL:
    """Loads libgemm_bf16.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with "
                                  "`python -m warp_specialized_tma_gb300.build` (needs nvcc)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


# ------------------------------------------------------------------ C mirror
def gemm_bf16_create(device: int = -1):
    h = _H()
    st = load().gemm_bf16_create(int(device), ctypes.byref(h))
    return st, h


def gemm_bf16_destroy(h) -> int:
    return load().gemm_bf16_destroy(h)


def gemm_bf16_set_option(h, key: int, value: int) -> int:
    return load().gemm_bf16_set_option(h, int(key), int(value))


def gemm_bf16_get_option(h, key: int):
    v = ctypes.c_int64()
    st = load().gemm_bf16_get_option(h, int(key), ctypes.byref(v))
    return st, v.value


def gemm_bf16_check_problem(M, N, K, lda, ldb, ldd) -> int:
    return load().gemm_bf16_check_problem(int(M), int(N), int(K), int(lda), int(ldb), int(ldd))


def gemm_bf16_plan(h, M, N, K, lda, ldb, ldd) -> int:
    return load().gemm_bf16_plan(h, int(M), int(N), int(K), int(lda), int(ldb), int(ldd))


def gemm_bf16_plan_info(h):
    info = PlanInfo()
    st = load().gemm_bf16_plan_info(h, ctypes.byref(info))
    return st, info


def gemm_bf16_run(h, A: int, B: int, D: int, stream: int = 0) -> int:
    return load().gemm_bf16_run(h, ctypes.c_void_p(A), ctypes.c_void_p(B), ctypes.c_void_p(D),
                                ctypes.c_void_p(stream))


def gemm_bf16_run_fused(h, A: int, B: int, D: int, C: int, ldc: int, bias: int, alpha: float, beta: float,
                        stream: int = 0) -> int:
    return load().gemm_bf16_run_fused(h, ctypes.c_void_p(A), ctypes.c_void_p(B), ctypes.c_void_p(D),
                                      ctypes.c_void_p(C), int(ldc), ctypes.c_void_p(bias),
                                      float(alpha), float(beta), ctypes.c_void_p(stream))


def gemm_bf16_run_host(h, hA, hB, hD, dA, dB, dD, stream: int = 0) -> int:
    return load().gemm_bf16_run_host(h, *(ctypes.c_void_p(p) for p in (hA, hB, hD, dA, dB, dD)),
                                     ctypes.c_void_p(stream))


def gemm_bf16_device_status(h):
    w = ctypes.c_uint32()
    st = load().gemm_bf16_device_status(h, ctypes.byref(w))
    return st, w.value


def gemm_bf16_run_noalloc(M, N, K, lda, ldb, ldd, A: int, B: int, D: int, stream: int = 0,
                          status: int | None = None) -> int:
    """Allocation-free GEMM on the current device.  `status` is None or the
    address of a uint32 in page-locked host memory or device memory, which
    receives the watchdog word once the stream has synchronised."""
    return load().gemm_bf16_run_noalloc(int(M), int(N), int(K), int(lda), int(ldb), int(ldd),
                                        ctypes.c_void_p(A), ctypes.c_void_p(B), ctypes.c_void_p(D),
                                        ctypes.c_void_p(stream),
                                        None if status is None else ctypes.c_void_p(int(status)))


def gemm_bf16_strerror(status: int) -> str:
    return load().gemm_bf16_strerror(int(status)).decode()


def gemm_bf16_version() -> str:
    return load().gemm_bf16_version().decode()


# ------------------------------------------------------------------ torch wrapper
def _check(st: int, what: str) -> None:
    if st != OK:
        raise GemmError(st, what)


def _stream_handle(stream, device=None) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ld(t, rows: int, what: str) -> int:
    if t.dim() != 2 or t.stride(1) != 1 or t.shape[0] != rows:
        raise ValueError(f"{what} must be a {rows} x ld row-major matrix")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


class Gemm:
    """One handle: plan once, run many times on torch tensors.

    ``Gemm(device=0, cta_group=2, ...)`` takes any option of OPTIONS as a keyword.
    """

    def __init__(self, device: int = -1, **options):
        import torch
        st, h = gemm_bf16_create(device)
        _check(st, "gemm_bf16_create")
        self.h = h
        # the device the handle is bound to: the library dereferences the raw
        # pointers it is given on this device only
        self.device = int(device) if device >= 0 else torch.cuda.current_device()
        self.shape = None
        for k, v in options.items():
            self.set_option(k, v)

    def set_option(self, name: str, value: int) -> None:
        _check(gemm_bf16_set_option(self.h, OPTIONS[name], int(value)), f"set_option({name}={value})")

    def get_option(self, name: str) -> int:
        st, v = gemm_bf16_get_option(self.h, OPTIONS[name])
        _check(st, f"get_option({name})")
        return v

    def plan(self, M, N, K, lda=None, ldb=None, ldd=None) -> dict:
        lda = K if lda is None else lda
        ldb = K if ldb is None else ldb
        ldd = N if ldd is None else ldd
        _check(gemm_bf16_plan(self.h, M, N, K, lda, ldb, ldd), "gemm_bf16_plan")
        self.shape = (M, N, K, lda, ldb, ldd)
        return self.info()

    def info(self) -> dict:
        st, info = gemm_bf16_plan_info(self.h)
        _check(st, "gemm_bf16_plan_info")
        return info.as_dict()

    def _on_device(self, *tensors) -> None:
        for t in tensors:
            if t.device.type != "cuda" or t.device.index != self.device:
                raise ValueError(f"tensors must be on cuda:{self.device}, the handle's device (got {t.device})")

    def _validate(self, A, B, D) -> None:
        import torch
        if self.shape is None:
            raise GemmError(ERR_NOT_PLANNED, "run")
        M, N, K, lda, ldb, ldd = self.shape
        for t, what in ((A, "A"), (B, "B"), (D, "D")):
            if t.dtype != torch.bfloat16:
                raise TypeError(f"{what} must be bf16")
        if A.shape[1] < K or B.shape[1] < K or D.shape[1] < N:
            raise ValueError("operand narrower than the plan")
        if (_ld(A, M, "A") != lda and M > 1) or (_ld(B, N, "B") != ldb and N > 1) or \
                (_ld(D, M, "D") != ldd and M > 1):
            raise ValueError("operand leading dimensions differ from the plan")

    def run(self, A, B, D, stream=None) -> None:
        """D[:M, :N] = A[:, :K] @ B[:, :K].T on device tensors (asynchronous)."""
        self._validate(A, B, D)
        if not (A.is_cuda and B.is_cuda and D.is_cuda):
            raise ValueError("run() takes device tensors; use run_host() for host operands")
        self._on_device(A, B, D)
        _check(gemm_bf16_run(self.h, A.data_ptr(), B.data_ptr(), D.data_ptr(), _stream_handle(stream, self.device)),
               "gemm_bf16_run")

    def run_fused(self, A, B, D, C=None, bias=None, alpha: float = 1.0, beta: float = 0.0, stream=None) -> None:
        """D = alpha * A @ B.T + beta * C + bias (C: M x ldc bf16 or None; bias: N bf16 or None)."""
        import torch
        self._validate(A, B, D)
        M, N = self.shape[0], self.shape[1]
        ldc = 0
        if C is not None:
            if C.dtype != torch.bfloat16 or not C.is_cuda:
                raise TypeError("C must be a bf16 device tensor")
            ldc = _ld(C, M, "C")
        if bias is not None and (bias.dtype != torch.bfloat16 or not bias.is_cuda or bias.numel() < N):
            raise TypeError("bias must be a bf16 device tensor with N values")
        self._on_device(A, B, D, *(t for t in (C, bias) if t is not None))
        _check(gemm_bf16_run_fused(self.h, A.data_ptr(), B.data_ptr(), D.data_ptr(),
                                   0 if C is None else C.data_ptr(), ldc,
                                   0 if bias is None else bias.data_ptr(), alpha, beta,
                                   _stream_handle(stream, self.device)), "gemm_bf16_run_fused")

    def run_host(self, hA, hB, hD, dA, dB, dD, stream=None) -> None:
        """Copies hA, hB to dA, dB, runs, copies the result to hD (all enqueued on `stream`)."""
        self._validate(hA, hB, hD)
        self._validate(dA, dB, dD)
        if hA.is_cuda or hB.is_cuda or hD.is_cuda:
            raise ValueError("run_host() takes host tensors hA, hB, hD")
        self._on_device(dA, dB, dD)
        _check(gemm_bf16_run_host(self.h, hA.data_ptr(), hB.data_ptr(), hD.data_ptr(), dA.data_ptr(),
                                  dB.data_ptr(), dD.data_ptr(), _stream_handle(stream, self.device)),
               "gemm_bf16_run_host")

    def device_status(self):
        """(status, detail word) of the device watchdog; synchronises the last stream."""
        return gemm_bf16_device_status(self.h)

    def close(self) -> None:
        if getattr(self, "h", None) is not None:
            gemm_bf16_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


_handles: dict = {}


def gemm(A, B, out=None, stream=None, **options):
    """D = A @ B.T for bf16 device matrices A (M x K) and B (N x K), via a cached handle."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    dev = A.device.index if A.device.index is not None else torch.cuda.current_device()
    key = (dev, tuple(sorted(options.items())))
    g = _handles.get(key)
    if g is None:
        g = _handles[key] = Gemm(dev, **options)
    shape = (M, N, K, _ld(A, M, "A") if M > 1 else K, _ld(B, N, "B") if N > 1 else K,
             _ld(out, M, "D") if M > 1 else N)
    if g.shape != shape:
        g.plan(*shape)
    g.run(A, B, out, stream)
    return out

"""A GB300-native persistent, warp-specialised, TMA-fed bf16 GEMM (D = A * B^T).

The compute path is hand-written CUDA for sm_103a behind a C ABI
(``include/gemm_bf16.h``, built into ``libgemm_bf16.so``); ``binding`` is a thin
ctypes layer over that ABI.  Import ``warp_specialized_tma_gb300.binding`` for
the GEMM; this package import itself loads nothing.
"""

__all__ = ["binding", "inputs"]

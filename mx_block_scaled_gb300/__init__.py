"""MX block-scaled NT GEMM for one NVIDIA GB300 (sm_103a).

C[M,N] = A[M,K] * B[N,K]^T with MXFP8 (E4M3) or MXFP4 (E2M1, two codes per
byte) operands, one E8M0 scale per 32 values along K, FP32 accumulation and
FP32 or BF16 output.  The compute path is the C-ABI library ``libmxgemm.so``
(hand-written CUDA for sm_103a); :mod:`.binding` is its thin ctypes front end.
:mod:`.inputs` generates seeded synthetic operands.
"""

import importlib

__all__ = ["binding", "inputs", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)

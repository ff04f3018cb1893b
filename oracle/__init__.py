"""CPU oracle for the MX block-scaled NT GEMM.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The product path (the package
``mx_block_scaled_gb300``) never imports it, and it never imports the package.
"""
from .mxref import (  # noqa: F401
    FMT_MXFP8,
    FMT_MXFP4,
    build,
    decode_table,
    gemm,
    grouped_gemm,
    bf16_gemm,
    bf16_to_f64,
    num_threads,
    quantize,
    placement_scan,
    placement_eval,
    placement_tuple,
    placement_values,
    IN_F32,
    IN_BF16,
)

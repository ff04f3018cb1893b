"""Helpers for the GPU parity tests: upload operands, call the C ABI, compare."""
from __future__ import annotations

import numpy as np

from mx_block_scaled_gb300.inputs import FMT_MXFP4, FMT_MXFP8, pack_fp4

OUT_F32 = 1
OUT_BF16 = 2


def lib():
    from mx_block_scaled_gb300 import build
    build.build()
    from mx_block_scaled_gb300 import binding
    return binding


def small_int_codes(rng, rows, K, fmt):
    """Codes of values in {0, +-0.5, +-1, +-2} with scales in [125, 129]: every partial
    sum of a K <= 2048 product is exact in FP32, so the GPU must match bit for bit."""
    vals = np.array([0x00, 0x30, 0x38, 0x40, 0xB0, 0xB8, 0xC0], np.uint8) if fmt == FMT_MXFP8 else \
        np.array([0x0, 0x1, 0x2, 0x4, 0x9, 0xA, 0xC], np.uint8)
    codes = vals[rng.integers(0, len(vals), size=(rows, K))]
    if fmt == FMT_MXFP4:
        codes = pack_fp4(codes)
    scales = rng.integers(125, 130, size=(rows, K // 32), dtype=np.uint8)
    return codes, scales


def to_dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def gpu_gemm_device(fmt, A, SA, B, SB, K, out=OUT_F32, flags=0):
    """Run C = A * B^T through mxgemm_run; return C as a CUDA tensor (no host copy)."""
    import torch
    b = lib()
    M, N = A.shape[0], B.shape[0]
    plan = b.Plan(M, N, K, fmt, out, flags)
    C = plan.run(to_dev(A), to_dev(SA), to_dev(B), to_dev(SB))
    b.check_device_status()
    torch.cuda.synchronize()
    return C


def gpu_gemm(fmt, A, SA, B, SB, K, out=OUT_F32, flags=0, run_flags=0, return_plan=False):
    """Run C = A * B^T through mxgemm_run; returns C as float64 numpy (and the plan text)."""
    import torch
    b = lib()
    M, N = A.shape[0], B.shape[0]
    plan = b.Plan(M, N, K, fmt, out, flags)
    dA, dB, dSA, dSB = to_dev(A), to_dev(B), to_dev(SA), to_dev(SB)
    C = plan.run(dA, dSA, dB, dSB, run_flags=run_flags)
    b.check_device_status()
    torch.cuda.synchronize()
    res = C.float().double().cpu().numpy()
    if return_plan:
        return res, plan.describe()
    return res


def tolerance(C_ref, S, out):
    """|C - C_ref| bound: 1e-5 * sum|a*b| for FP32 accumulation in any order,
    plus 2^-8 * |C_ref| for the BF16 rounding of the output."""
    tol = 1e-5 * S
    if out == OUT_BF16:
        tol = tol + 2.0 ** -8 * np.abs(C_ref)
    return tol


def assert_within(C, C_ref, S, out, what=""):
    nan = np.isnan(C_ref)
    assert (np.isnan(C) == nan).all(), f"{what}: NaN pattern differs"
    err = np.abs(C - C_ref)[~nan]
    tol = tolerance(C_ref, S, out)[~nan]
    bad = err > tol
    if bad.any():
        idx = np.argwhere((np.abs(C - C_ref) > tolerance(C_ref, S, out)) & ~nan)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first {idx.tolist()}; "
                             f"worst err/tol {np.max(err / np.maximum(tol, 1e-300)):.3g}")
    return float(np.max(err / np.maximum(tol, 1e-300))) if err.size else 0.0


def sample_indices(n, seed, count=32):
    """First/last index, the first and last of a few seeded 128-blocks, and random picks."""
    rng = np.random.default_rng(seed)
    idx = {0, n - 1}
    for blk in rng.integers(0, (n + 127) // 128, size=4):
        idx.add(int(blk) * 128)
        idx.add(min(n - 1, int(blk) * 128 + 127))
    idx.update(int(i) for i in rng.integers(0, n, size=count))
    return np.array(sorted(idx), dtype=np.int64)


def tile_sample_indices(n, seed, block=128):
    """One seeded index inside every `block`-wide block of [0, n), plus the first
    and the last index.  Where the tiles of a plan are 128 or 256 rows (or
    columns) wide and start on multiples of 128 -- every plan of a shape with
    more than 256 rows on that side -- sampled rows over all columns (or sampled
    columns over all rows) touch every tile of the plan, split-K slabs and
    stream-K cut tiles included."""
    rng = np.random.default_rng(seed)
    nb = (n + block - 1) // block
    starts = np.arange(nb, dtype=np.int64) * block
    widths = np.minimum(block, n - starts)
    idx = starts + np.floor(rng.random(nb) * widths).astype(np.int64)
    return np.unique(np.concatenate([idx, [0, n - 1]])).astype(np.int64)


FMTS = {"mxfp8": FMT_MXFP8, "mxfp4": FMT_MXFP4}

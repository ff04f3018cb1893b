"""Seeded synthetic inputs for the MX block-scaled NT GEMM.

This module only *produces* operands: packed element codes and E8M0 scale
bytes, from seeded random numbers.  It holds no part of the GEMM itself (no
decoding, no products, no accumulation), so the CUDA path and the CPU oracle
can both be fed from it without sharing any of the method's arithmetic.

The workloads restate the serving shapes of the FlyDSL article (English digest,
section "Whole-request experiments are closer to serving, with narrow
conditions": Llama-3.1-8B, Qwen3-32B and Llama-3.3-70B at TP=1) as projection
GEMMs C[M,N] = A[M,K] * B[N,K]^T with M tokens and (N, K) the weight shape.
There is no dataset and no trained weight: values are N(0,1) draws.

Quantisation recipe (the step before the GEMM; the article times the GEMM from
already-quantised inputs, section "Performance numbers need their baselines"):
  * per row, per 32-value block along K: amax = max |x|;
  * scale exponent s = floor(log2 amax) - e_max with e_max = 8 for E4M3 (448 =
    1.75 * 2^8) and 2 for E2M1 (6 = 1.5 * 2^2), clamped to [-127, 127]; the
    E8M0 code is s + 127; an all-zero block gets code 127;
  * v = x / 2^s (exact), rounded to the element grid with round-half-to-even,
    magnitudes above the largest finite value saturate (448 or 6); the sign of
    a zero is kept.
floor(log2 amax) comes from frexp, never from a floating-point log2.
"""
from __future__ import annotations

import os

import numpy as np

FMT_MXFP8 = 1
FMT_MXFP4 = 2
FMT_BY_NAME = {"mxfp8": FMT_MXFP8, "mxfp4": FMT_MXFP4}
OUT_F32 = 1
OUT_BF16 = 2
OUT_BY_NAME = {"f32": OUT_F32, "bf16": OUT_BF16}

_CHUNK = 1 << 20  # elements per quantisation chunk (bounds host memory per thread)

# E2M1 magnitude (x2) -> 3-bit code: 0,.5,1,1.5,2,3,4,6 -> 0..7
_E2M1_CODE_OF_TWICE = np.full(13, 255, dtype=np.uint8)
for _code, _twice in enumerate((0, 1, 2, 3, 4, 6, 8, 12)):
    _E2M1_CODE_OF_TWICE[_twice] = _code


def row_bytes(fmt: int, K: int) -> int:
    """Bytes per operand row: K for MXFP8, K/2 for MXFP4."""
    return K if fmt == FMT_MXFP8 else K // 2


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes [rows, K] into bytes [rows, K/2]; element 2i in the low nibble."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    return (c[:, 0::2] & 15) | ((c[:, 1::2] & 15) << 4)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_fp4`."""
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 15
    out[:, 1::2] = p >> 4
    return out


def _round_to_grid(v: np.ndarray, min_exp: int, mbits: int, vmax: float) -> np.ndarray:
    """Round-half-even v onto a binary grid with `mbits` fraction bits, exponent
    floor `min_exp` (subnormal spacing 2^(min_exp-mbits)), saturating at vmax."""
    _, e = np.frexp(v)
    q = np.maximum(e - 1, min_exp) - mbits
    r = np.ldexp(np.rint(np.ldexp(v, -q)), q)
    return np.clip(r, -vmax, vmax)


def _encode_e4m3(r: np.ndarray) -> np.ndarray:
    mag = np.abs(r)
    sign = np.signbit(r).astype(np.uint8) << 7
    m, e = np.frexp(mag)  # mag = m * 2^e, m in [0.5, 1)
    normal = mag >= 2.0 ** -6
    ef = np.where(normal, e + 6, 0)
    mf = np.where(normal, np.rint((2.0 * m - 1.0) * 8.0), np.rint(mag * 512.0))
    return sign | (ef.astype(np.uint8) << 3) | mf.astype(np.uint8)


def _encode_e2m1(r: np.ndarray) -> np.ndarray:
    twice = np.rint(np.abs(r) * 2.0).astype(np.int64)
    code = _E2M1_CODE_OF_TWICE[twice]
    return code | (np.signbit(r).astype(np.uint8) << 3)


def _quantize_rows(x, fmt, codes, scales, r0, r1):
    K = x.shape[1]
    e_max, min_exp, mbits, vmax = ((8, -6, 3, 448.0) if fmt == FMT_MXFP8 else (2, 0, 1, 6.0))
    xb = x[r0:r1].astype(np.float64).reshape(r1 - r0, K // 32, 32)
    amax = np.abs(xb).max(axis=2)
    _, e = np.frexp(amax)
    s = np.where(amax > 0, e - 1 - e_max, 0)
    s = np.clip(s, -127, 127)
    scales[r0:r1] = (s + 127).astype(np.uint8)
    v = np.ldexp(xb, -s[:, :, None])
    r = _round_to_grid(v, min_exp, mbits, vmax).reshape(r1 - r0, K)
    codes[r0:r1] = _encode_e4m3(r) if fmt == FMT_MXFP8 else _encode_e2m1(r)


def quantize_mx(x: np.ndarray, fmt: int):
    """Quantise float data [rows, K] to MX codes and E8M0 scales.

    Returns ``(codes, scales)``: codes are [rows, K] uint8 for MXFP8 or packed
    [rows, K/2] for MXFP4; scales are [rows, K/32] uint8.  Row chunks are
    quantised on a thread pool (each chunk independently, so the result does not
    depend on the thread count).
    """
    rows, K = x.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    codes = np.empty((rows, K), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    step = max(1, _CHUNK // K)
    spans = [(r0, min(rows, r0 + step)) for r0 in range(0, rows, step)]
    if len(spans) == 1:
        _quantize_rows(x, fmt, codes, scales, *spans[0])
    else:
        from concurrent.futures import ThreadPoolExecutor
        workers = min(len(spans), os.cpu_count() or 1, 32)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(lambda sp: _quantize_rows(x, fmt, codes, scales, *sp), spans))
    if fmt == FMT_MXFP4:
        codes = pack_fp4(codes)
    return codes, scales


def normal_f32(rng: np.random.Generator, rows: int, K: int) -> np.ndarray:
    return rng.standard_normal((rows, K), dtype=np.float32)


def with_outlier_blocks(x: np.ndarray, rng: np.random.Generator, frac: float = 0.01,
                        factor: float = 256.0) -> np.ndarray:
    """Multiply round(frac * #blocks) distinct 32-blocks (chosen uniformly) by `factor`."""
    rows, K = x.shape
    nblk = rows * (K // 32)
    k = int(round(frac * nblk))
    idx = rng.choice(nblk, size=k, replace=False)
    y = x.reshape(nblk, 32).copy()
    y[idx] *= np.float32(factor)
    return y.reshape(rows, K)


def uniform_codes(rng: np.random.Generator, rows: int, K: int, fmt: int):
    """Independent uniform codes over the whole code space, every scale 127 (x1.0)."""
    if fmt == FMT_MXFP4:
        codes = pack_fp4(rng.integers(0, 16, size=(rows, K), dtype=np.uint8))
    else:
        codes = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    return codes, np.full((rows, K // 32), 127, dtype=np.uint8)


def finite_uniform_codes(rng: np.random.Generator, rows: int, K: int, fmt: int,
                         scale_lo: int = 127, scale_hi: int = 127):
    """Uniform codes without the E4M3 NaN codes, scales uniform in [lo, hi]."""
    if fmt == FMT_MXFP8:
        codes = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
        nan = (codes & 0x7F) == 0x7F
        codes[nan] &= 0xFE  # 0x7F -> 0x7E (448), 0xFF -> 0xFE (-448)
    else:
        codes = pack_fp4(rng.integers(0, 16, size=(rows, K), dtype=np.uint8))
    scales = rng.integers(scale_lo, scale_hi + 1, size=(rows, K // 32), dtype=np.uint8)
    return codes, scales


# ---------------------------------------------------------------------------
# Workloads: projection shapes of the three served models, plus two small and
# square cases.  A's seed is [cfg, shape index, 0]; B's is [cfg, (N,K) index, 1]
# so that every M of one weight shape sees the same weight.
# ---------------------------------------------------------------------------

def _shapes(ms, nks):
    return [(m, n, k) for m in ms for (n, k) in nks]


WORKLOADS = {
    # 256^3 MXFP4, uniform codes, unit scales, FP32 out: every partial sum is a
    # multiple of 1/4 below 2^14, so any FP32 summation order is exact.
    "mxfp4_uniform_256": dict(cfg=0, fmts=("mxfp4",), out="f32", values="uniform",
                              nks=[(256, 256)], ms=[256]),
    # 4096^3 MXFP8 from N(0,1), BF16 out.
    "mxfp8_square_4096": dict(cfg=1, fmts=("mxfp8",), out="bf16", values="normal",
                              nks=[(4096, 4096)], ms=[4096]),
    # Llama-3.1-8B projections (QKV, O, gate+up, down), MXFP4.
    "llama31_8b": dict(cfg=2, fmts=("mxfp4",), out="bf16", values="normal",
                       nks=[(6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336)],
                       ms=[256, 2048, 8192]),
    # Llama-3.3-70B projections, MXFP8 and MXFP4, decode and prefill token counts.
    "llama33_70b": dict(cfg=3, fmts=("mxfp8", "mxfp4"), out="bf16", values="normal",
                        nks=[(10240, 8192), (8192, 8192), (57344, 8192), (8192, 28672)],
                        ms=[8, 64, 256, 16384]),
    # Qwen3-32B projections with 1% outlier blocks (x2^8) stressing the E8M0 range.
    "qwen3_32b": dict(cfg=4, fmts=("mxfp8", "mxfp4"), out="bf16", values="normal_outliers",
                      nks=[(10240, 5120), (5120, 8192), (51200, 5120), (5120, 25600)],
                      ms=[128, 4096]),
}


def workload_cases(name: str):
    """Yield (fmt_name, shape_index, nk_index, M, N, K) for every case of a workload."""
    w = WORKLOADS[name]
    for fmt in w["fmts"]:
        si = 0
        for m in w["ms"]:
            for nki, (n, k) in enumerate(w["nks"]):
                yield fmt, si, nki, m, n, k
                si += 1


def make_operand(name: str, which: str, index: int, rows: int, K: int, fmt: int):
    """Codes and scales of operand `which` ('A' or 'B') for a workload case.

    `index` is the shape index for A and the (N,K) index for B.
    """
    w = WORKLOADS[name]
    rng = np.random.default_rng([w["cfg"], index, 0 if which == "A" else 1])
    if w["values"] == "uniform":
        return uniform_codes(rng, rows, K, fmt)
    x = normal_f32(rng, rows, K)
    if w["values"] == "normal_outliers":
        x = with_outlier_blocks(x, rng)
    return quantize_mx(x, fmt)


# ---------------------------------------------------------------------------
# Grouped (mixture-of-experts) workloads.  The FlyDSL page (English digest,
# "Performance numbers need their baselines") times 24 grouped GEMMs covering
# uniform groups, projection-dimension changes and uneven expert loads, without
# listing them; these synthetic cases stand in for those three axes with
# expert shapes of common MoE layers: 8 experts with (N, K) = (28672, 4096)
# gate+up and (4096, 14336) down projections, and 64 fine-grained experts with
# (1536, 2048) / (2048, 768).  Tokens are N(0,1) rows quantised like the dense
# workloads; group sizes are uniform or drawn from a seeded Zipf-like law.
# ---------------------------------------------------------------------------

MOE_WORKLOADS = {
    # name: groups, total token rows, (N, K) per expert, load ("uniform" or "zipf")
    "moe8_uniform_prefill": dict(groups=8, rows=8192, nks=[(28672, 4096), (4096, 14336)], load="uniform"),
    "moe64_uneven_prefill": dict(groups=64, rows=8192, nks=[(1536, 2048), (2048, 768)], load="zipf"),
    "moe64_uneven_decode": dict(groups=64, rows=256, nks=[(1536, 2048), (2048, 768)], load="zipf"),
    "moe8_uneven_decode": dict(groups=8, rows=64, nks=[(28672, 4096), (4096, 14336)], load="zipf"),
}


def group_sizes(groups: int, rows: int, load: str, seed) -> np.ndarray:
    """Rows per group summing to `rows`: equal shares, or a Zipf-like draw
    (weights 1/rank^1.2 over a seeded permutation of the groups; some groups
    may receive no rows)."""
    if load == "uniform":
        base = np.full(groups, rows // groups, dtype=np.int64)
        base[: rows - base.sum()] += 1
        return base
    rng = np.random.default_rng(seed)
    w = 1.0 / np.arange(1, groups + 1) ** 1.2
    w = w[rng.permutation(groups)]
    counts = rng.multinomial(rows, w / w.sum()).astype(np.int64)
    return counts


def group_offsets(sizes) -> np.ndarray:
    """Offsets [0, s0, s0+s1, ...] (groups + 1 entries, int64)."""
    return np.concatenate([[0], np.cumsum(np.asarray(sizes, dtype=np.int64))]).astype(np.int64)


def moe_cases(name: str):
    """Yield (fmt_name, nk_index, groups, rows, N, K, sizes) for a grouped workload (both formats)."""
    w = MOE_WORKLOADS[name]
    for fmt in ("mxfp8", "mxfp4"):
        for nki, (n, k) in enumerate(w["nks"]):
            sizes = group_sizes(w["groups"], w["rows"], w["load"], [len(name), nki, w["groups"]])
            yield fmt, nki, w["groups"], w["rows"], n, k, sizes

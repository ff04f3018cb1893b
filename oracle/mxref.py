"""ctypes front end of the C oracle in ``oracle/mxref.c``.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This module marshals
numpy arrays into the C routine and compiles it with gcc when the shared object
is missing or older than its source.  No arithmetic of the method lives here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FMT_MXFP8 = 1
FMT_MXFP4 = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxref.c")
_SO = os.path.join(_HERE, "_build", "libmxref.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mxref.c`` into ``oracle/_build/libmxref.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
           "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.mxref_gemm.restype = ctypes.c_int
            lib.mxref_gemm.argtypes = [
                ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.mxref_decode_table.restype = ctypes.c_int
            lib.mxref_decode_table.argtypes = [ctypes.c_int, ctypes.c_void_p]
            lib.mxref_num_threads.restype = ctypes.c_int
            lib.mxref_placement_scan.restype = ctypes.c_int
            lib.mxref_placement_scan.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                                 ctypes.c_void_p, ctypes.c_void_p]
            lib.mxref_placement_eval.restype = ctypes.c_int
            lib.mxref_placement_eval.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                                 ctypes.c_void_p]
            lib.mxref_placement_values.restype = ctypes.c_int
            lib.mxref_placement_values.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
            lib.mxref_quantize.restype = ctypes.c_int
            lib.mxref_quantize.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            _lib = lib
    return _lib


def decode_table(which: str) -> np.ndarray:
    """Return the oracle's decode table: 'e4m3' (256), 'e2m1' (16) or 'e8m0' (256)."""
    idx = {"e4m3": 1, "e2m1": 2, "e8m0": 3}[which]
    out = np.empty(256, dtype=np.float64)
    n = _load().mxref_decode_table(idx, out.ctypes.data)
    return out[:n].copy()


def num_threads() -> int:
    return int(_load().mxref_num_threads())


def _u8(x, shape):
    a = np.ascontiguousarray(x, dtype=np.uint8)
    if a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def gemm(fmt: int, A, SA, B, SB, K: int, rows=None, cols=None,
         with_abs: bool = True, nthreads: int = 0):
    """Reference C = A * B^T (binary64) and S = sum |a*b| (same scaling).

    ``A``: M x (K or K/2) uint8 codes; ``SA``: M x K/32 uint8 E8M0 scales;
    likewise ``B``/``SB`` with N rows.  ``rows``/``cols`` select a subset of the
    output (index arrays); the result then has shape (len(rows), len(cols)).
    Returns ``(C, S)`` (``S`` is None when ``with_abs`` is False).
    """
    rb = K if fmt == FMT_MXFP8 else K // 2
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    M, N = A.shape[0], B.shape[0]
    A = _u8(A, (M, rb))
    B = _u8(B, (N, rb))
    SA = _u8(SA, (M, K // 32))
    SB = _u8(SB, (N, K // 32))
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    C = np.empty((nr, nc), dtype=np.float64)
    S = np.empty((nr, nc), dtype=np.float64) if with_abs else None
    rc = _load().mxref_gemm(
        fmt, M, N, K, A.ctypes.data, SA.ctypes.data, B.ctypes.data, SB.ctypes.data,
        None if r is None else r.ctypes.data, nr,
        None if c is None else c.ctypes.data, nc,
        C.ctypes.data, None if S is None else S.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError("mxref_gemm rejected its arguments")
    return C, S


IN_F32 = 1
IN_BF16 = 2


def quantize(fmt: int, x, in_dtype: int = IN_F32):
    """Reference MX quantiser: x [rows, K] (float32, or uint16 BF16 bit patterns when
    in_dtype == IN_BF16) -> (codes, row-major scales)."""
    x = np.ascontiguousarray(x, dtype=np.float32 if in_dtype == IN_F32 else np.uint16)
    rows, K = x.shape
    codes = np.zeros((rows, K if fmt == FMT_MXFP8 else K // 2), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    rc = _load().mxref_quantize(fmt, in_dtype, rows, K, x.ctypes.data, codes.ctypes.data, scales.ctypes.data)
    if rc != 0:
        raise ValueError("mxref_quantize rejected its arguments")
    return codes, scales


def grouped_gemm(fmt: int, offsets, A, SA, B, SB, N: int, K: int, rows=None, with_abs: bool = True,
                 nthreads: int = 0):
    """Reference grouped GEMM (mixture-of-experts layout): group e owns rows
    [offsets[e], offsets[e+1]) of A (and of C) and weight rows [e*N, (e+1)*N) of B;
    C[r, :] = A[r] * B_e^T for every row r of group e.  Written as one call of the
    pinned per-group reference :func:`gemm` per group (its plain definition).

    ``offsets``: G+1 non-decreasing row offsets.  ``rows`` (optional): which rows
    of C to compute.  Returns ``(C, S)`` over those rows (all rows by default);
    rows outside every group stay 0.
    """
    off = [int(v) for v in np.asarray(offsets).reshape(-1)]
    T = A.shape[0]
    rsel = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    C = np.zeros((rsel.size, N), dtype=np.float64)
    S = np.zeros((rsel.size, N), dtype=np.float64) if with_abs else None
    for e in range(len(off) - 1):
        lo, hi = off[e], off[e + 1]
        pick = np.nonzero((rsel >= lo) & (rsel < hi))[0]
        if pick.size == 0:
            continue
        Be, SBe = B[e * N:(e + 1) * N], SB[e * N:(e + 1) * N]
        Ce, Se = gemm(fmt, A[lo:hi], SA[lo:hi], Be, SBe, K, rows=rsel[pick] - lo, with_abs=with_abs,
                      nthreads=nthreads)
        C[pick] = Ce
        if with_abs:
            S[pick] = Se
    return C, S


def bf16_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> binary64, exactly: a BF16 value is the FP32
    value whose upper 16 bits are the pattern and whose lower 16 bits are zero."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):  # NaN patterns widen to NaN
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_gemm(A_bits, B_bits, rows=None, cols=None, with_abs: bool = True):
    """Reference BF16 NT GEMM: C = A * B^T and S = |A| * |B|^T in binary64 from
    BF16 operands (the FlyDSL page's BF16 "NT GEMM" set, section "Performance
    numbers need their baselines").  Every product of two BF16 values is exact
    in binary64; the sums go through one binary64 matrix product (error far below
    the FP32-accumulation bound the parity tests allow)."""
    A = bf16_to_f64(A_bits)
    B = bf16_to_f64(B_bits)
    if rows is not None:
        A = A[np.asarray(rows, dtype=np.int64)]
    if cols is not None:
        B = B[np.asarray(cols, dtype=np.int64)]
    C = A @ B.T
    S = np.abs(A) @ np.abs(B).T if with_abs else None
    return C, S


def placement_scan(k: int, sa, sb):
    """Reference scale-placement checker (see ``mxref_placement_scan``): for each
    scale pair, counts [pre != post, pre == rn_exact, post == rn_exact] over all
    16^(2k) E2M1 tuples and the first tuple where pre and post differ (-1: none)."""
    sa = np.ascontiguousarray(sa, dtype=np.int32)
    sb = np.ascontiguousarray(sb, dtype=np.int32)
    n = sa.size
    counts = np.zeros((n, 3), dtype=np.int64)
    first = np.zeros(n, dtype=np.int64)
    if _load().mxref_placement_scan(k, sa.ctypes.data, sb.ctypes.data, n, counts.ctypes.data, first.ctypes.data):
        raise ValueError("mxref_placement_scan rejected its arguments")
    return counts, first


def placement_tuple(k: int, a_codes, b_codes) -> int:
    """Tuple number of E2M1 codes (element 0 first): a_i at bits 4i, b_i at 4(k+i)."""
    t = 0
    for i, c in enumerate(a_codes):
        t |= int(c) << (4 * i)
    for i, c in enumerate(b_codes):
        t |= int(c) << (4 * (k + i))
    return t


def placement_eval(k: int, sa: int, sb: int, t: int):
    """(pre, post, rn) of tuple t as binary32 values (see ``mxref_placement_scan``)."""
    out = np.zeros(3, dtype=np.float32)
    if _load().mxref_placement_eval(k, sa, sb, t, out.ctypes.data):
        raise ValueError("mxref_placement_eval rejected its arguments")
    return tuple(float(v) for v in out)


def placement_values(k: int, sa: int, sb: int) -> np.ndarray:
    """[16^(2k), 3] float32: pre, post and rn of every tuple of one scale pair (k <= 3)."""
    out = np.zeros((1 << (8 * k), 3), dtype=np.float32)
    if _load().mxref_placement_values(k, sa, sb, out.ctypes.data):
        raise ValueError("mxref_placement_values rejected its arguments")
    return out

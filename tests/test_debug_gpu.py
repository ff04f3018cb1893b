"""The debug build (libmxgemm_debug.so, compiled with MXGEMM_DEBUG) on the GPU.

Every plain global load and store of its GEMM kernels is bounds-checked, C is
pre-filled with NaN, and a run returns the device status word.  On valid plans
of every kind (single-CTA and CTA-pair tiles, swap-AB, split-K, stream-K, MXFP8,
MXFP4, BF16) no check may fire, no element of C may keep the NaN fill, and C
must equal the oracle's product exactly (small-integer codes, FP32 out).  The
bounds self-test then shows a check firing: the kernel is told that C ends one
row early, skips those stores without faulting, and reports it."""
import ctypes

import numpy as np
import pytest

from gpu_util import OUT_F32, lib, small_int_codes, to_dev
from mx_block_scaled_gb300.inputs import FMT_MXFP4, FMT_MXFP8

pytestmark = pytest.mark.gpu

FMT_BF16 = 3
SINGLE, PAIR, SK, NOSK = 1 << 5, 1 << 4, 1 << 7, 1 << 16


@pytest.fixture(scope="module")
def dbg():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3)
    b = lib()
    d = b.load_library(b.DEBUG_LIB_PATH)
    assert d.mxgemm_debug_build() == 1
    return d


def _operands(fmt, M, N, K, seed):
    rng = np.random.default_rng(seed)
    if fmt == FMT_BF16:
        import torch
        a = rng.integers(-8, 9, (M, K)).astype(np.float32)
        b = rng.integers(-8, 9, (N, K)).astype(np.float32)
        ta = torch.from_numpy(a).bfloat16().view(torch.uint8).numpy().reshape(M, 2 * K)
        tb = torch.from_numpy(b).bfloat16().view(torch.uint8).numpy().reshape(N, 2 * K)
        return ta, None, tb, None, a.astype(np.float64) @ b.astype(np.float64).T
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    return A, SA, B, SB, None


def _plan(d, M, N, K, fmt, flags):
    h = ctypes.c_void_p()
    st = d.mxgemm_plan_create(ctypes.byref(h), M, N, K, fmt, OUT_F32, flags)
    assert st == 0, st
    buf = ctypes.create_string_buffer(512)
    d.mxgemm_plan_describe(h, buf, 512)
    return h, buf.value.decode()


def _run(d, entry, fmt, M, N, K, flags, seed, oracle_mod):
    import torch
    A, SA, B, SB, ref = _operands(fmt, M, N, K, seed)
    if ref is None:
        ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    h, desc = _plan(d, M, N, K, fmt, flags)
    ws_bytes = d.mxgemm_workspace_bytes(h)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    dA, dB = to_dev(A), to_dev(B)
    dSA = to_dev(SA) if SA is not None else None
    dSB = to_dev(SB) if SB is not None else None
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = entry(h, dA.data_ptr(), dSA.data_ptr() if dSA is not None else None, dB.data_ptr(),
               dSB.data_ptr() if dSB is not None else None, C.data_ptr(), ws.data_ptr(), ws_bytes, 0, stream)
    torch.cuda.synchronize()
    d.mxgemm_plan_destroy(h)
    return st, C.double().cpu().numpy(), ref, desc


CASES = [
    (FMT_MXFP8, 300, 520, 1152, SINGLE, "mode=single"),
    (FMT_MXFP8, 520, 1024, 4096, PAIR, "sa=in-kernel"),
    (FMT_MXFP8, 1000, 512, 3072, PAIR | SK, "mode=pair"),
    (FMT_MXFP8, 1024, 1536, 4096, SINGLE | SK, "mode=single"),
    (FMT_MXFP8, 200, 328, 2048, SINGLE | (3 << 8), "split_k=3"),
    (FMT_MXFP8, 8, 1280, 4096, SK, "swap_ab=1"),
    (FMT_MXFP8, 33, 8192, 1024, 0, "swap_ab=1"),
    (FMT_MXFP4, 383, 640, 1536, PAIR, "mode=pair"),
    (FMT_MXFP4, 136, 256, 512, SINGLE, "mode=single"),
    (FMT_MXFP4, 64, 2048, 4096, SK, "swap_ab=1"),
    (FMT_BF16, 264, 392, 512, 0, "fmt=bf16"),
    (FMT_BF16, 300, 768, 1024, PAIR, "mode=pair"),
    (FMT_MXFP8, 256, 1000, 1536, 1 << 17, "tile=256x192"),
    (FMT_MXFP4, 300, 2000, 2048, 1 << 17, "tile=256x192"),
    (FMT_MXFP8, 100, 1000, 8192, 0, "swap_ab=1"),
    (FMT_MXFP8, 8, 10240, 2048, 0, " lean"),
    (FMT_MXFP4, 8, 1280, 16384, 0, " lean"),
]


@pytest.mark.parametrize("fmt,M,N,K,flags,expect", CASES)
def test_debug_build_runs_clean_and_writes_every_element(dbg, oracle_mod, fmt, M, N, K, flags, expect):
    st, C, ref, desc = _run(dbg, dbg.mxgemm_run, fmt, M, N, K, flags, M + N + K, oracle_mod)
    assert expect in desc, desc
    assert st == 0, (st, desc)
    assert not np.isnan(C).any(), (int(np.isnan(C).sum()), desc)
    assert (C == ref).all(), desc
    assert dbg.mxgemm_device_status(None, 1) == 0


ONE_SPLIT = 1 << 8  # split-K forced to 1: C is written by the GEMM kernel itself


@pytest.mark.parametrize("fmt,M,N,K,flags", [(FMT_MXFP8, 300, 520, 1152, SINGLE | ONE_SPLIT),
                                             (FMT_MXFP8, 520, 1024, 4096, PAIR | ONE_SPLIT),
                                             (FMT_MXFP8, 1000, 512, 3072, PAIR | SK),
                                             (FMT_MXFP4, 383, 640, 1536, PAIR | ONE_SPLIT)])
def test_bounds_check_skips_and_reports_an_out_of_range_store(dbg, oracle_mod, fmt, M, N, K, flags):
    st, C, ref, desc = _run(dbg, dbg.mxgemm_selftest_bounds, fmt, M, N, K, flags, 7 * M + K, oracle_mod)
    assert st == -9, (st, desc)  # MXGEMM_ERR_DEVICE_BOUNDS
    assert np.isnan(C[M - 1]).all(), desc  # the last row kept its NaN fill
    assert (C[: M - 1] == ref[: M - 1]).all(), desc
    assert dbg.mxgemm_device_status(None, 1) == -9  # sticky until cleared
    assert dbg.mxgemm_device_status(None, 1) == 0


SWAP = 1 << 3
GROUPED_CASES = [
    # (fmt, group sizes, N, K, leading gap rows, plan flags, expected plan text)
    (FMT_MXFP8, [0, 1, 127, 128, 129, 300], 384, 512, 3, 0, "mode=single"),
    (FMT_MXFP8, [5, 0, 33, 0, 200], 128, 1024, 7, SWAP, "swap_ab=1"),
    (FMT_MXFP8, [300, 0, 600, 37], 256, 1024, 0, PAIR, "mode=pair"),
    (FMT_MXFP4, [300, 0, 600, 37], 512, 1024, 5, PAIR, "mode=pair"),
]


@pytest.mark.parametrize("fmt,sizes,N,K,lead,flags,expect", GROUPED_CASES)
def test_debug_build_grouped_runs_clean(dbg, oracle_mod, fmt, sizes, N, K, lead, flags, expect):
    """The grouped GEMM (single-CTA, swap-AB and CTA-pair tiles) in the debug
    build: no bounds check fires, every row inside a group equals the oracle's
    grouped product, and rows outside every group keep their NaN fill."""
    import torch
    from mx_block_scaled_gb300.inputs import group_offsets
    offsets = [lead + int(o) for o in group_offsets(sizes)]
    T, G = offsets[-1] + 4, len(sizes)
    rng = np.random.default_rng([fmt, T, N, K])
    A, SA = small_int_codes(rng, T, K, fmt)
    B, SB = small_int_codes(rng, G * N, K, fmt)
    ref, _ = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K)
    h = ctypes.c_void_p()
    assert dbg.mxgemm_grouped_plan_create(ctypes.byref(h), G, T, N, K, fmt, OUT_F32, flags) == 0
    buf = ctypes.create_string_buffer(512)
    dbg.mxgemm_grouped_plan_describe(h, buf, 512)
    desc = buf.value.decode()
    ws_bytes = dbg.mxgemm_grouped_workspace_bytes(h)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    d_off = torch.tensor(np.asarray(offsets, dtype=np.int64), device="cuda")
    dA, dSA, dB, dSB = to_dev(A), to_dev(SA), to_dev(B), to_dev(SB)
    C = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    st = dbg.mxgemm_grouped_run(h, d_off.data_ptr(), dA.data_ptr(), dSA.data_ptr(), dB.data_ptr(), dSB.data_ptr(),
                                C.data_ptr(), ws.data_ptr(), ws_bytes, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    dbg.mxgemm_grouped_plan_destroy(h)
    assert expect in desc, desc
    assert st == 0, (st, desc)
    got = C.double().cpu().numpy()
    inside = np.zeros(T, bool)
    for e in range(G):
        inside[offsets[e]:offsets[e + 1]] = True
    assert (got[inside] == ref[inside]).all(), desc
    assert np.isnan(got[~inside]).all(), desc
    assert dbg.mxgemm_device_status(None, 1) == 0

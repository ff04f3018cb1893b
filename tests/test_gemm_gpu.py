"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Exact equality wherever every partial sum is representable in FP32 (then any
FP32 accumulation order gives the same bits); elsewhere the bound
|C - C_ref| <= 1e-5 * sum|a*b| (+ 2^-8 |C_ref| for BF16 output).
"""
import numpy as np
import pytest

from golden_io import load_handworked
from gpu_util import (OUT_BF16, OUT_F32, assert_within, gpu_gemm, gpu_gemm_device, lib, small_int_codes,
                      tile_sample_indices, to_dev)
from mx_block_scaled_gb300.inputs import (FMT_MXFP4, FMT_MXFP8, finite_uniform_codes, make_operand,
                                          pack_fp4, workload_cases)

pytestmark = pytest.mark.gpu

# plan flags: 256-row tiles on CTA pairs / 128-row tiles on single CTAs
PAIR, SINGLE = 1 << 4, 1 << 5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    cap = torch.cuda.get_device_capability()
    assert cap == (10, 3), f"expected an sm_103 GPU, got {cap}"
    lib()


# ---- scale relayout: byte-exact against the documented index formula --------

def relayout_reference(S, rows, K):
    kb = K // 32
    nrb, nkt = (rows + 127) // 128, K // 128
    out = np.full((nrb, nkt, 512), 127, np.uint8)
    for r in range(rows):
        R, rr = divmod(r, 128)
        q, p = divmod(rr, 32)
        for j in range(kb):
            T, c = divmod(j, 4)
            out[R, T, p * 16 + q * 4 + c] = S[r, j]
    return out.reshape(-1)


@pytest.mark.parametrize("rows", [1, 8, 127, 128, 129, 300])
@pytest.mark.parametrize("K", [128, 256, 28672])
def test_relayout_matches_index_formula(rows, K):
    import torch
    b = lib()
    rng = np.random.default_rng(rows * 7 + K)
    S = rng.integers(0, 256, size=(rows, K // 32), dtype=np.uint8)
    out = b.relayout_scales(to_dev(S), rows, K)
    torch.cuda.synchronize()
    ref = relayout_reference(S, rows, K) if rows * K <= 300 * 256 else None
    got = out.cpu().numpy()
    assert got.size == b.mxgemm_sf_bytes(rows, K)
    if ref is not None:
        assert (got == ref).all()
    else:  # vectorised form of the same formula for the large K
        kb = K // 32
        r = np.arange(rows)[:, None]
        j = np.arange(kb)[None, :]
        pos = ((r // 128) * (K // 128) + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4
        assert (got[pos] == S).all()


# ---- element formats and descriptors: all code pairs ---------------------------

@pytest.mark.parametrize("k_pos", [0, 45, 127])
def test_all_fp8_code_pairs(oracle_mod, k_pos):
    K = 128
    A = np.zeros((256, K), np.uint8)
    A[:, k_pos] = np.arange(256)
    S = np.full((256, K // 32), 127, np.uint8)
    C = gpu_gemm(FMT_MXFP8, A, S, A, S, K, OUT_F32)
    ref, _ = oracle_mod.gemm(FMT_MXFP8, A, S, A, S, K)
    assert (np.isnan(C) == np.isnan(ref)).all()
    ok = ~np.isnan(ref)
    assert (C[ok] == ref[ok]).all()


@pytest.mark.parametrize("k_pos", [0, 1, 70, 127])
def test_all_fp4_code_pairs(oracle_mod, k_pos):
    K = 128
    codes = np.zeros((16, K), np.uint8)
    codes[:, k_pos] = np.arange(16)
    A = pack_fp4(codes)
    S = np.full((16, K // 32), 127, np.uint8)
    C = gpu_gemm(FMT_MXFP4, A, S, A, S, K, OUT_F32)
    ref, _ = oracle_mod.gemm(FMT_MXFP4, A, S, A, S, K)
    assert (C == ref).all()


@pytest.mark.parametrize("case", load_handworked(), ids=lambda c: c["name"])
def test_handworked_dot_products(case):
    C = gpu_gemm(case["fmt"], case["A"], case["SA"], case["B"], case["SB"], 128, OUT_F32)
    assert C[0, 0] == float(case["expected"])


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_identity_b_returns_dequantised_a(oracle_mod, fmt):
    K = 256
    rng = np.random.default_rng(21)
    A, SA = finite_uniform_codes(rng, 200, K, fmt, 120, 134)
    one = 0x38 if fmt == FMT_MXFP8 else 0x2
    eye = np.where(np.eye(K, dtype=bool), one, 0).astype(np.uint8)
    B = eye if fmt == FMT_MXFP8 else pack_fp4(eye)
    SB = np.full((K, K // 32), 127, np.uint8)
    C = gpu_gemm(fmt, A, SA, B, SB, K, OUT_F32)
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    assert (C == ref).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_per_block_scale_sweep(oracle_mod, fmt):
    """Each A row has exactly one nonzero 32-block; rows cycle over all blocks, and
    every (row, block) and (column, block) has its own scale: pins the scale
    addressing (TMEM scale columns, scale ids, relayout) element by element."""
    K, M, N = 1024, 300, 272
    rng = np.random.default_rng(22)
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    w = 32 if fmt == FMT_MXFP8 else 16  # bytes of one 32-block in a row
    Ab = A.copy()
    for m in range(M):
        j = m % (K // 32)
        keep = np.zeros(Ab.shape[1], bool)
        keep[j * w:(j + 1) * w] = True
        Ab[m, ~keep] = 0
    C = gpu_gemm(fmt, Ab, SA, B, SB, K, OUT_F32)
    ref, _ = oracle_mod.gemm(fmt, Ab, SA, B, SB, K)
    assert (C == ref).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
@pytest.mark.parametrize("flags", [0, SINGLE, PAIR])
@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (8, 129, 256), (127, 255, 384), (129, 8, 128),
                                   (255, 127, 384), (130, 300, 640), (64, 512, 1024), (385, 264, 384)])
def test_edge_shapes_exact(oracle_mod, fmt, flags, M, N, K):
    if flags == PAIR and (M < 128 or N < 128):
        pytest.skip("pair tiles are for shapes with at least 128 rows on each side")
    rng = np.random.default_rng(M * 1000 + N + K)
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    for out in (OUT_F32, OUT_BF16):
        C = gpu_gemm(fmt, A, SA, B, SB, K, out, flags=flags)
        if out == OUT_F32:
            assert (C == ref).all(), f"M={M} N={N} K={K}"
        else:
            import torch
            expect = torch.from_numpy(ref.astype(np.float32)).bfloat16().double().numpy()
            assert (C == expect).all(), f"M={M} N={N} K={K} bf16"


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
@pytest.mark.parametrize("flags", [0, 1 << 2, 1 << 3, (1 << 2) | 1, (1 << 2) | 2, (3 << 8), (1 << 3) | (5 << 8),
                                   SINGLE, SINGLE | 2, PAIR | 1, PAIR | 2, PAIR | 1 | (3 << 8), PAIR | 2 | (2 << 8),
                                   PAIR | (1 << 3), PAIR | (1 << 3) | 1])
def test_plan_variants_agree_with_oracle(oracle_mod, fmt, flags):
    """Forced tile width / swap-AB / split-K variants all reproduce the oracle."""
    M, N, K = 200, 384, 2048
    rng = np.random.default_rng(23)
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    C, desc = gpu_gemm(fmt, A, SA, B, SB, K, OUT_F32, flags=flags, return_plan=True)
    assert (C == ref).all(), desc


SK = 1 << 7  # stream-K plan flag


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
@pytest.mark.parametrize("mode", [SINGLE, PAIR])
@pytest.mark.parametrize("M,N,K", [(1024, 1536, 4096), (2560, 2304, 1024), (300, 520, 1152), (8, 8192, 2048)])
def test_stream_k_exact(oracle_mod, fmt, mode, M, N, K):
    """Tiles whose k-stages are spread over several CTAs or CTA pairs (stream-K,
    fixed up in the kernel) give the exact result, as does the default
    decomposition."""
    if mode == PAIR and min(M, N) < 128:
        pytest.skip("cluster modes are for shapes with at least 128 rows on each side")
    rng = np.random.default_rng(M + 7 * N + K)
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    C, desc = gpu_gemm(fmt, A, SA, B, SB, K, OUT_F32, flags=SK | mode, return_plan=True)
    # pair tiles need MXFP4 rows of whole 128-byte K-slices (K % 256 == 0)
    assert ("mode=pair" in desc) == (mode == PAIR and (fmt != FMT_MXFP4 or K % 256 == 0)), desc
    assert "streamk=" in desc and "/0 " not in desc.split("streamk=")[1][:12], desc
    assert (C == ref).all(), desc
    C2, desc2 = gpu_gemm(fmt, A, SA, B, SB, K, OUT_BF16, return_plan=True)
    import torch
    expect = torch.from_numpy(ref.astype(np.float32)).bfloat16().double().numpy()
    assert (C2 == expect).all(), desc2
    C3 = gpu_gemm(fmt, A, SA, B, SB, K, OUT_BF16, flags=SK | mode)  # stream-K, BF16 out
    assert (C3 == expect).all(), desc


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
@pytest.mark.parametrize("M,N,K,forced", [(8, 1280, 4096, True), (64, 2048, 4096, True), (1, 384, 1024, True),
                                          (33, 8192, 1024, True), (8, 20480, 1024, True),
                                          (8, 10240, 16384, False), (8, 1280, 32768, False)])
def test_decode_stream_k_exact(oracle_mod, fmt, M, N, K, forced):
    """Weight-streaming decode shapes (swap-AB, 32- or 64-token tiles) with the
    k-stages of the tiles beyond the full waves spread over every SM (stream-K),
    cutting tiles into up to ~8 segments whose partial sums the epilogue of the
    last CTA adds in k order: exact, FP32 and BF16 out.  Short k-loops get
    stream-K from the plan flag (their default plan splits K); 80 tiles of 64
    k-stages and 10 tiles of 128 k-stages get it by default.  The default plan
    of every shape is exact too."""
    rng = np.random.default_rng([M, N, K, fmt])
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    import torch
    expect = torch.from_numpy(ref.astype(np.float32)).bfloat16().double().numpy()
    flags = SK if forced else 0
    C, desc = gpu_gemm(fmt, A, SA, B, SB, K, OUT_F32, flags=flags, return_plan=True)
    assert "swap_ab=1" in desc and "/0 " not in desc.split("streamk=")[1][:16], desc
    assert (C == ref).all(), desc
    C2 = gpu_gemm(fmt, A, SA, B, SB, K, OUT_BF16, flags=flags)
    assert (C2 == expect).all(), desc
    if forced:
        C3, desc3 = gpu_gemm(fmt, A, SA, B, SB, K, OUT_F32, return_plan=True)
        assert "swap_ab=1" in desc3, desc3
        assert (C3 == ref).all(), desc3


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_prelayout_scales_give_the_same_result(fmt):
    import torch
    b = lib()
    M, N, K = 160, 320, 512
    rng = np.random.default_rng(24)
    A, SA = finite_uniform_codes(rng, M, K, fmt, 110, 140)
    B, SB = finite_uniform_codes(rng, N, K, fmt, 110, 140)
    plan = b.Plan(M, N, K, fmt, OUT_F32)
    dA, dB, dSA, dSB = to_dev(A), to_dev(B), to_dev(SA), to_dev(SB)
    C1 = plan.run(dA, dSA, dB, dSB)
    tSA, tSB = b.relayout_scales(dSA, M, K), b.relayout_scales(dSB, N, K)
    C2 = plan.run(dA, tSA, dB, tSB, run_flags=b.MXGEMM_RUN_SA_PRELAYOUT | b.MXGEMM_RUN_SB_PRELAYOUT)
    C3 = plan.run(dA, dSA, dB, tSB, run_flags=b.MXGEMM_RUN_SB_PRELAYOUT)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2) and torch.equal(C1, C3)


@pytest.mark.parametrize("M,N,K,flags", [(136, 256, 512, PAIR), (383, 640, 1536, PAIR), (520, 1024, 4096, PAIR),
                                         (520, 1024, 4096, PAIR | SK), (300, 768, 2048, PAIR | (3 << 8)),
                                         (1000, 512, 3072, PAIR | SK)])
def test_in_kernel_scale_layout_exact(oracle_mod, M, N, K, flags):
    """MXFP8 pair plans with K % 512 == 0 lay out the row-major activation
    scales inside the GEMM (the odd CTA of each pair builds both CTAs' chunks):
    ragged pair tiles (rows past M), many scale groups per tile, stream-K
    segments and split-K slabs that start inside a group all give the oracle's
    result, bit-identical to the pre-laid-out path."""
    import torch
    b = lib()
    rng = np.random.default_rng([M, N, K, flags])
    A, SA = small_int_codes(rng, M, K, FMT_MXFP8)
    B, SB = small_int_codes(rng, N, K, FMT_MXFP8)
    ref, _ = oracle_mod.gemm(FMT_MXFP8, A, SA, B, SB, K)
    plan = b.Plan(M, N, K, FMT_MXFP8, OUT_F32, flags)
    assert "sa=in-kernel" in plan.describe(), plan.describe()
    dA, dB, dSA, dSB = to_dev(A), to_dev(B), to_dev(SA), to_dev(SB)
    C1 = plan.run(dA, dSA, dB, dSB)
    tSA = b.relayout_scales(dSA, M, K)
    C2 = plan.run(dA, tSA, dB, dSB, run_flags=b.MXGEMM_RUN_SA_PRELAYOUT)
    b.check_device_status()
    torch.cuda.synchronize()
    assert torch.equal(C1, C2), plan.describe()
    assert (C1.double().cpu().numpy() == ref).all(), plan.describe()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_nan_scale_makes_its_rows_nan(oracle_mod, fmt):
    """E8M0 code 0xFF is NaN: every output fed by such a block is NaN, the rest is exact."""
    M, N, K = 160, 288, 256
    rng = np.random.default_rng(31)
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    SA[5, 2] = 0xFF
    SB[200, 7] = 0xFF
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    assert np.isnan(ref[5]).all() and np.isnan(ref[:, 200]).all()
    C = gpu_gemm(fmt, A, SA, B, SB, K, OUT_F32)
    assert (np.isnan(C) == np.isnan(ref)).all()
    ok = ~np.isnan(ref)
    assert (C[ok] == ref[ok]).all()


# ---- invariants at full workload size (GPU vs GPU, no oracle cost) ------------

@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_incrementing_every_a_scale_doubles_c_exactly(fmt):
    import torch
    b = lib()
    M, N, K = 4096, 4096, 4096
    A, SA = make_operand("mxfp8_square_4096", "A", 0, M, K, fmt)
    B, SB = make_operand("mxfp8_square_4096", "B", 0, N, K, fmt)
    assert SA.max() < 254
    for out in (OUT_F32, OUT_BF16):
        plan = b.Plan(M, N, K, fmt, out)
        dA, dB, dSB = to_dev(A), to_dev(B), to_dev(SB)
        C1 = plan.run(dA, to_dev(SA), dB, dSB)
        C2 = plan.run(dA, to_dev(SA + 1), dB, dSB)
        torch.cuda.synchronize()
        assert torch.equal(C2.float(), 2 * C1.float())


# ---- the workloads ---------------------------------------------------------------

def test_mxfp4_uniform_256_is_bit_exact(oracle_mod):
    M = N = K = 256
    A, SA = make_operand("mxfp4_uniform_256", "A", 0, M, K, FMT_MXFP4)
    B, SB = make_operand("mxfp4_uniform_256", "B", 0, N, K, FMT_MXFP4)
    ref, _ = oracle_mod.gemm(FMT_MXFP4, A, SA, B, SB, K)
    C = gpu_gemm(FMT_MXFP4, A, SA, B, SB, K, OUT_F32)
    assert (C == ref).all()


def test_mxfp8_square_4096_full(oracle_mod):
    M = N = K = 4096
    A, SA = make_operand("mxfp8_square_4096", "A", 0, M, K, FMT_MXFP8)
    B, SB = make_operand("mxfp8_square_4096", "B", 0, N, K, FMT_MXFP8)
    C = gpu_gemm(FMT_MXFP8, A, SA, B, SB, K, OUT_BF16)
    ref, S = oracle_mod.gemm(FMT_MXFP8, A, SA, B, SB, K)
    assert_within(C, ref, S, OUT_BF16, "mxfp8 4096^3")


def _all_workload_cases():
    """Every shape of the model workloads, grouped so that consecutive cases share
    the weight operand B: (workload, fmt, shape index, (N,K) index, M, N, K)."""
    from mx_block_scaled_gb300.inputs import WORKLOADS
    out = []
    for name in ("llama31_8b", "llama33_70b", "qwen3_32b"):
        cases = list(workload_cases(name))
        cases.sort(key=lambda c: (c[0], c[2], c[3]))
        out += [(name, c[0], c[1], c[2], c[3], c[4], c[5]) for c in cases]
    assert len(out) == sum(len(w["fmts"]) * len(w["ms"]) * len(w["nks"])
                           for n, w in WORKLOADS.items() if n in ("llama31_8b", "llama33_70b", "qwen3_32b"))
    return out


_WEIGHTS = {}


def _weights(name, fmt, nki, N, K):
    key = (name, fmt, nki)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()  # one weight resident at a time: cases are grouped by weight
        _WEIGHTS[key] = make_operand(name, "B", nki, N, K, fmt)
    return _WEIGHTS[key]


@pytest.mark.parametrize("name,fmt,si,nki,M,N,K", _all_workload_cases(),
                         ids=[f"{c[0]}-{c[1]}-M{c[4]}-N{c[5]}-K{c[6]}" for c in _all_workload_cases()])
def test_workload_full_size_sampled(oracle_mod, name, fmt, si, nki, M, N, K):
    """Full-size model shapes in the default launch configuration, within the bound:
    for M <= 256 every element of C; otherwise one seeded row inside every 128-row
    tile (all columns) and one seeded column inside every 128-column tile (all
    rows), so that every output tile of the plan -- split-K slabs and stream-K
    cut tiles included -- has elements compared with the oracle."""
    f = FMT_MXFP8 if fmt == "mxfp8" else FMT_MXFP4
    A, SA = make_operand(name, "A", si, M, K, f)
    B, SB = _weights(name, f, nki, N, K)
    import torch
    C = gpu_gemm_device(f, A, SA, B, SB, K, OUT_BF16)
    if M <= 256:
        got = C.double().cpu().numpy()
        del C
        ref, S = oracle_mod.gemm(f, A, SA, B, SB, K)
        worst = assert_within(got, ref, S, OUT_BF16, f"{name} full C")
        _record_parity_stat(name=name, format=fmt, M=M, N=N, K=K, rows=M, cols=N, full=True,
                            worst_err_over_bound=worst)
        return
    rows = tile_sample_indices(M, si)
    cols = tile_sample_indices(N, nki + 100)
    C_rows = C[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    C_cols = C[:, torch.from_numpy(cols).cuda()].double().cpu().numpy()
    del C
    ref_r, S_r = oracle_mod.gemm(f, A, SA, B, SB, K, rows=rows)
    worst_r = assert_within(C_rows, ref_r, S_r, OUT_BF16, f"{name} rows")
    ref_c, S_c = oracle_mod.gemm(f, A, SA, B, SB, K, cols=cols)
    worst_c = assert_within(C_cols, ref_c, S_c, OUT_BF16, f"{name} cols")
    _record_parity_stat(name=name, format=fmt, M=M, N=N, K=K, rows=len(rows), cols=len(cols), full=False,
                        worst_err_over_bound=max(worst_r, worst_c))


def _record_parity_stat(**rec):
    """Append the worst |C - C_ref| / bound of a case to the JSON-lines file named by
    MXGEMM_PARITY_STATS (unset: nothing is written)."""
    import json
    import os
    path = os.environ.get("MXGEMM_PARITY_STATS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


# ---- failure path: a stalled kernel returns an error instead of hanging --------

def test_stalled_kernel_times_out_and_context_survives():
    import torch
    b = lib()
    M = N = K = 256
    plan = b.Plan(M, N, K, FMT_MXFP8, OUT_F32)
    A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    S = torch.full((b.mxgemm_sf_bytes(M, K),), 127, dtype=torch.uint8, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert b.mxgemm_device_status(stream, True) == b.MXGEMM_OK
    st = b.mxgemm_selftest_stall(plan.handle, A.data_ptr(), S.data_ptr(), A.data_ptr(), S.data_ptr(),
                                 C.data_ptr(), plan.workspace.data_ptr(), plan.ws_bytes, stream)
    assert st == b.MXGEMM_OK
    assert b.mxgemm_device_status(stream, True) == b.MXGEMM_ERR_DEVICE_TIMEOUT
    assert b.mxgemm_device_status(stream, True) == b.MXGEMM_OK
    # the context is still usable: a normal run afterwards is correct
    A1 = torch.full((M, K), 0x38, dtype=torch.uint8, device="cuda")
    Srow = torch.full((M, K // 32), 127, dtype=torch.uint8, device="cuda")
    out = plan.run(A1, Srow, A1, Srow)
    b.check_device_status()
    assert torch.all(out == float(K))


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
@pytest.mark.parametrize("plan_flags", [0, SK])
def test_prepare_then_run_equals_run(oracle_mod, fmt, plan_flags):
    """mxgemm_prepare (scale relayout into the workspace + stream-K counter reset)
    followed by mxgemm_run with MXGEMM_RUN_PREPARED gives the same exact result
    as mxgemm_run alone, for every choice of pre-laid-out operands, and again
    on a second prepared run over the same workspace."""
    import torch
    b = lib()
    M, N, K = 1024, 1536, 4096
    rng = np.random.default_rng([fmt, plan_flags, 3])
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    plan = b.Plan(M, N, K, fmt, OUT_F32, plan_flags)
    if plan_flags & SK:
        assert "/0 " not in plan.describe().split("streamk=")[1][:12], plan.describe()
    dA, dB, dSA, dSB = to_dev(A), to_dev(B), to_dev(SA), to_dev(SB)
    tSA, tSB = b.relayout_scales(dSA, M, K), b.relayout_scales(dSB, N, K)
    C0 = plan.run(dA, dSA, dB, dSB)
    torch.cuda.synchronize()
    assert (C0.double().cpu().numpy() == ref).all()
    for rf in (0, b.MXGEMM_RUN_SB_PRELAYOUT, b.MXGEMM_RUN_SA_PRELAYOUT,
               b.MXGEMM_RUN_SA_PRELAYOUT | b.MXGEMM_RUN_SB_PRELAYOUT):
        sa_pre = rf & b.MXGEMM_RUN_SA_PRELAYOUT
        sb_pre = rf & b.MXGEMM_RUN_SB_PRELAYOUT
        for _ in range(2):
            plan.prepare(None if sa_pre else dSA, None if sb_pre else dSB, rf)
            # a plan that lays out row-major SA inside the GEMM (sa=in-kernel) reads SA in run
            sa_arg = tSA if sa_pre else (dSA if "sa=in-kernel" in plan.describe() else None)
            C = plan.run(dA, sa_arg, dB, tSB if sb_pre else None, run_flags=rf | b.MXGEMM_RUN_PREPARED)
            b.check_device_status()
            torch.cuda.synchronize()
            assert (C.double().cpu().numpy() == ref).all(), (rf, plan.describe())


@pytest.mark.parametrize("fmt,M,N,K,expect", [
    ("mxfp8", 4096, 4096, 4096, ["tile=256x256", "mode=pair", "streamk=228+28/56", "sa=in-kernel"]),
    ("mxfp8", 16384, 8192, 8192, ["tile=256x256", "mode=pair", "sa=in-kernel"]),
    ("mxfp8", 8, 10240, 8192, ["tile=128x32", "mode=single", "swap_ab=1", "streamk=0+80/152", "lean"]),
    ("mxfp8", 64, 8192, 8192, ["tile=128x64", "swap_ab=1", "split_k=2", "streamk=64+0/0", "!lean"]),
    ("bf16", 8, 8192, 8192, ["tile=128x32", "swap_ab=1", "!lean"]),
    ("mxfp8", 8, 8192, 28672, ["tile=128x32", "swap_ab=1", "streamk=0+64/152"]),
    ("mxfp8", 128, 5120, 8192, ["tile=256x128", "mode=pair", "swap_ab=1"]),
    ("mxfp8", 128, 10240, 5120, ["tile=256x192", "mode=pair", "swap_ab=0"]),
    ("mxfp4", 8, 10240, 8192, ["tile=128x32", "swap_ab=1", "streamk=80+0/0"]),
    ("mxfp4", 4096, 4096, 4096, ["tile=256x256", "mode=pair", "sa=relayout"]),
    ("mxfp4", 256, 6144, 4096, ["tile=128x256", "mode=single"]),
    ("mxfp4", 256, 10240, 8192, ["tile=256x192", "mode=pair"]),
    ("mxfp4", 256, 8192, 8192, ["tile=256x192", "mode=pair", "split_k=1"]),
    ("bf16", 128, 10240, 5120, ["tile=128x128", "mode=single"]),
    ("bf16", 128, 51200, 5120, ["mode=pair"]),
    ("bf16", 256, 6144, 4096, ["tile=256x128", "mode=pair"]),
    ("bf16", 256, 10240, 8192, ["tile=256x192", "mode=pair"]),
    ("mxfp8", 256, 10240, 8192, ["tile=256x192", "mode=pair", "split_k=1"]),
    ("mxfp8", 256, 8192, 8192, ["tile=256x256", "mode=pair", "split_k=2"]),
])
def test_default_plans_follow_the_heuristic(fmt, M, N, K, expect):
    """The planner's choices on representative shapes, as the design documents them
    (pair tiles for MXFP8 from 128 tokens, MXFP4 pair tiles from half a wave, 192-wide
    pair tiles where 256-wide ones fill less than a wave and cannot split two ways,
    BF16 small-token tile rules, swap-AB decode with stream-K over every SM on wide
    or long k-loops and split-K otherwise, the lean kernel form for MX decode of at
    most 32 tokens)."""
    b = lib()
    f = {"mxfp8": FMT_MXFP8, "mxfp4": FMT_MXFP4, "bf16": b.MXGEMM_FMT_BF16}[fmt]
    plan = b.Plan(M, N, K, f, OUT_BF16)
    d = plan.describe()
    sms = __import__("torch").cuda.get_device_properties(0).multi_processor_count
    for e in expect:
        if "streamk=" in e and sms != 152:
            continue  # the stream-K split depends on the SM count
        if e.startswith("!"):
            assert e[1:] not in d, (e, d)
        else:
            assert e in d, (e, d)


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
@pytest.mark.parametrize("M,N,K", [(8, 1280, 4096), (8, 10240, 2048), (1, 384, 1024), (32, 2048, 8192)])
def test_static_weight_early_loads_exact(oracle_mod, fmt, M, N, K):
    """MXGEMM_RUN_B_STATIC on the lean decode form (the weight's first ring and
    first scale group loaded before the grid-dependency wait): back-to-back calls,
    each the programmatic dependent of the one before, and a CUDA-graph replay of
    them give the oracle's product exactly, as does a call without the flag."""
    import torch
    b = lib()
    rng = np.random.default_rng([M, N, K, fmt, 5])
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    plan = b.Plan(M, N, K, fmt, OUT_F32)
    assert "lean" in plan.describe(), plan.describe()
    dA, dSA, dB, dSB = to_dev(A), to_dev(SA), to_dev(B), to_dev(SB)
    flags = b.MXGEMM_RUN_B_STATIC
    outs = [plan.run(dA, dSA, dB, dSB, run_flags=flags) for _ in range(4)]
    outs.append(plan.run(dA, dSA, dB, dSB))
    b.check_device_status()
    torch.cuda.synchronize()
    for C in outs:
        assert (C.double().cpu().numpy() == ref).all(), plan.describe()
    Cs = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for C in Cs:
            plan.run(dA, dSA, dB, dSB, C=C, run_flags=flags)
    g.replay()
    torch.cuda.synchronize()
    b.check_device_status()
    for C in Cs:
        assert (C.double().cpu().numpy() == ref).all(), plan.describe()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
@pytest.mark.parametrize("M,N,K", [(256, 1000, 1536), (300, 2000, 1152), (200, 4096, 2048), (129, 776, 4096)])
def test_pair_192_wide_tiles_exact(oracle_mod, fmt, M, N, K):
    """256 x 192 CTA-pair tiles (MXGEMM_PLAN_FORCE_BN192; planned by default where
    256-wide pair tiles fill less than a wave and cannot split two ways): every
    other tile starts 64 rows into a 128-row scale chunk, so its MMAs
    read the B scales two TMEM columns in, and the last tile's second chunk lies
    past the end of B; ragged M and N, in-kernel and relayout activation scales."""
    if fmt == FMT_MXFP4 and K % 256 != 0:
        pytest.skip("MXFP4 pair tiles need K % 256 == 0")
    rng = np.random.default_rng([M, N, K, fmt, 192])
    A, SA = small_int_codes(rng, M, K, fmt)
    B, SB = small_int_codes(rng, N, K, fmt)
    ref, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    flags = (1 << 17) | ((1 << 8) if fmt == FMT_MXFP8 else 0)  # FORCE_BN192; MXFP8: one split
    C, desc = gpu_gemm(fmt, A, SA, B, SB, K, OUT_F32, flags=flags, return_plan=True)
    assert "tile=256x192" in desc, desc
    assert (C == ref).all(), desc
    C2, desc2 = gpu_gemm(fmt, A, SA, B, SB, K, OUT_BF16, flags=1 << 17, return_plan=True)
    import torch
    expect = torch.from_numpy(ref.astype(np.float32)).bfloat16().double().numpy()
    assert (C2 == expect).all(), desc2


@pytest.mark.parametrize("M,N,K", [(128, 640, 8192), (100, 1000, 8192), (65, 384, 16384)])
def test_swap_pair_default_for_mid_token_counts_exact(oracle_mod, M, N, K):
    """MXFP8 with 65-128 tokens and K >= 8192 plans swap-AB on CTA pairs (the weight
    in the 256-row role, the tokens as one 128-wide tile): exact against the oracle,
    row-major and pre-laid-out scales, FP32 and BF16 out."""
    b = lib()
    rng = np.random.default_rng([M, N, K, 65])
    A, SA = small_int_codes(rng, M, K, FMT_MXFP8)
    B, SB = small_int_codes(rng, N, K, FMT_MXFP8)
    ref, _ = oracle_mod.gemm(FMT_MXFP8, A, SA, B, SB, K)
    C, desc = gpu_gemm(FMT_MXFP8, A, SA, B, SB, K, OUT_F32, return_plan=True)
    assert "mode=pair" in desc and "swap_ab=1" in desc and "tile=256x128" in desc, desc
    assert (C == ref).all(), desc
    import torch
    plan = b.Plan(M, N, K, FMT_MXFP8, OUT_BF16)
    tSA = b.relayout_scales(to_dev(SA), M, K)
    tSB = b.relayout_scales(to_dev(SB), N, K)
    C2 = plan.run(to_dev(A), tSA, to_dev(B), tSB,
                  run_flags=b.MXGEMM_RUN_SA_PRELAYOUT | b.MXGEMM_RUN_SB_PRELAYOUT)
    b.check_device_status()
    expect = torch.from_numpy(ref.astype(np.float32)).bfloat16().double().numpy()
    assert (C2.double().cpu().numpy() == expect).all(), desc


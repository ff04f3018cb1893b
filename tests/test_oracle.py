"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: the element
formats' published values (via PyTorch's independent float8 decoders and the
E2M1 magnitude set), hand-worked dot products, exact rational arithmetic,
an independent binary64 matmul, and algebraic invariants of the definition.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from mx_block_scaled_gb300.inputs import (FMT_MXFP4, FMT_MXFP8, finite_uniform_codes,
                                          pack_fp4, unpack_fp4)
from golden_io import load_handworked

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---- independent decoders (third-party: PyTorch's float8 dtypes) -------------

def torch_e4m3(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_e8m0(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e8m0fnu).to(torch.float32).to(torch.float64).numpy()


def e2m1_from_set(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    mag = np.array(E2M1_MAGNITUDES)[c & 7]
    return np.where(c & 8, -mag, mag)


def dequant(fmt, codes, scales, K):
    """Dequantised operand via the independent decoders: value * 2^(scale-127)."""
    if fmt == FMT_MXFP8:
        v = torch_e4m3(codes)
    else:
        v = e2m1_from_set(unpack_fp4(codes))
    s = torch_e8m0(scales)
    return v * np.repeat(s, 32, axis=1)


# ---- decode tables -----------------------------------------------------------

def test_e2m1_table_is_the_mx_magnitude_set(oracle_mod):
    t = oracle_mod.decode_table("e2m1")
    assert t.shape == (16,)
    assert list(t[:8]) == E2M1_MAGNITUDES            # codes 0..7, increasing
    assert list(-t[8:]) == E2M1_MAGNITUDES           # sign bit is bit 3
    assert np.signbit(t[8]) and t[8] == 0.0          # 0x8 is -0
    assert sorted(set(np.abs(t))) == E2M1_MAGNITUDES
    assert np.isfinite(t).all()                      # no NaN / inf in E2M1


def test_e4m3_table_matches_torch_float8_e4m3fn(oracle_mod):
    t = oracle_mod.decode_table("e4m3")
    ref = torch_e4m3(np.arange(256))
    nan = np.isnan(ref)
    assert (np.isnan(t) == nan).all()
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert (t[~nan] == ref[~nan]).all()
    assert np.signbit(t[~nan]).tolist() == np.signbit(ref[~nan]).tolist()
    assert np.nanmax(t) == 448.0 and np.nanmin(t) == -448.0
    assert t[0x01] == 2.0 ** -9                      # smallest subnormal


def test_e8m0_table_matches_torch_float8_e8m0fnu(oracle_mod):
    t = oracle_mod.decode_table("e8m0")
    ref = torch_e8m0(np.arange(256))
    assert np.isnan(t[255]) and np.isnan(ref[255])
    assert (t[:255] == ref[:255]).all()
    assert t[127] == 1.0 and t[0] == 2.0 ** -127 and t[254] == 2.0 ** 127


# ---- hand-worked dot products (tests/golden/handworked_dot.txt) -------------

@pytest.mark.parametrize("case", load_handworked(), ids=lambda c: c["name"])
def test_handworked_dot_products(oracle_mod, case):
    C, S = oracle_mod.gemm(case["fmt"], case["A"], case["SA"], case["B"], case["SB"], 128)
    assert Fraction(C[0, 0]) == case["expected"]
    assert S[0, 0] >= abs(C[0, 0])


# ---- brute force over all code pairs ----------------------------------------

@pytest.mark.parametrize("k_pos", [0, 77, 127])
def test_all_fp8_code_pairs(oracle_mod, k_pos):
    K = 128
    A = np.zeros((256, K), np.uint8)
    A[:, k_pos] = np.arange(256)
    B = A.copy()
    SA = np.full((256, K // 32), 127, np.uint8)
    C, _ = oracle_mod.gemm(FMT_MXFP8, A, SA, B, SA, K)
    d = torch_e4m3(np.arange(256))
    ref = np.outer(d, d)
    assert (np.isnan(C) == np.isnan(ref)).all()
    ok = ~np.isnan(ref)
    assert (C[ok] == ref[ok]).all()


@pytest.mark.parametrize("k_pos", [0, 1, 76, 127])
def test_all_fp4_code_pairs(oracle_mod, k_pos):
    K = 128
    codes = np.zeros((16, K), np.uint8)
    codes[:, k_pos] = np.arange(16)
    A = pack_fp4(codes)
    # B gets a non-unit scale on the block holding k_pos: result scales by 2^3.
    SA = np.full((16, K // 32), 127, np.uint8)
    SB = SA.copy()
    SB[:, k_pos // 32] = 130
    C, _ = oracle_mod.gemm(FMT_MXFP4, A, SA, A, SB, K)
    d = e2m1_from_set(np.arange(16))
    assert (C == np.outer(d, d) * 8.0).all()


# ---- structure: identity B, single block, transposition ---------------------

@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_identity_b_returns_dequantised_a(oracle_mod, fmt):
    K = 128
    rng = np.random.default_rng(11)
    A, SA = finite_uniform_codes(rng, 40, K, fmt, 110, 140)
    one = 0x38 if fmt == FMT_MXFP8 else 0x2
    eye = np.where(np.eye(K, dtype=bool), one, 0).astype(np.uint8)
    B = eye if fmt == FMT_MXFP8 else pack_fp4(eye)
    SB = np.full((K, K // 32), 127, np.uint8)
    C, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    assert (C == dequant(fmt, A, SA, K)).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_non_square_matches_independent_matmul(oracle_mod, fmt):
    """Random codes and scales, M != N: catches transposed operands, wrong scale
    indices and dropped blocks.  Reference: independent decoders + binary64 matmul."""
    K, M, N = 512, 37, 53
    rng = np.random.default_rng(12)
    A, SA = finite_uniform_codes(rng, M, K, fmt, 100, 150)
    B, SB = finite_uniform_codes(rng, N, K, fmt, 100, 150)
    C, S = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    ref = dequant(fmt, A, SA, K) @ dequant(fmt, B, SB, K).T
    refS = np.abs(dequant(fmt, A, SA, K)) @ np.abs(dequant(fmt, B, SB, K)).T
    assert np.allclose(S, refS, rtol=1e-13, atol=0)
    assert (np.abs(C - ref) <= 1e-13 * S).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_exact_rational_on_tiny_inputs(oracle_mod, fmt):
    """Exact result in rationals; the oracle must be within (K/32) ulp-of-S of it."""
    K, M, N = 256, 3, 4
    rng = np.random.default_rng(13)
    A, SA = finite_uniform_codes(rng, M, K, fmt, 90, 160)
    B, SB = finite_uniform_codes(rng, N, K, fmt, 90, 160)
    C, S = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    a, b = dequant(fmt, A, SA, K), dequant(fmt, B, SB, K)
    for m in range(M):
        for n in range(N):
            exact = sum((Fraction(x) * Fraction(y) for x, y in zip(a[m], b[n])), Fraction(0))
            err = abs(Fraction(C[m, n]) - exact)
            assert err <= Fraction(K // 32) * Fraction(2) ** -52 * Fraction(S[m, n])


def test_single_block_contribution_is_exact(oracle_mod):
    """Zero all blocks but j: C equals that block's exact contribution."""
    K, M, N = 256, 8, 6
    rng = np.random.default_rng(14)
    A, SA = finite_uniform_codes(rng, M, K, FMT_MXFP8, 120, 135)
    B, SB = finite_uniform_codes(rng, N, K, FMT_MXFP8, 120, 135)
    for j in range(K // 32):
        Aj = np.zeros_like(A)
        Aj[:, 32 * j:32 * j + 32] = A[:, 32 * j:32 * j + 32]
        C, _ = oracle_mod.gemm(FMT_MXFP8, Aj, SA, B, SB, K)
        a = torch_e4m3(A[:, 32 * j:32 * j + 32])
        b = torch_e4m3(B[:, 32 * j:32 * j + 32])
        scale = np.outer(torch_e8m0(SA[:, j]), torch_e8m0(SB[:, j]))
        assert (C == (a @ b.T) * scale).all()   # 32-term sums: exact in binary64


# ---- invariants ---------------------------------------------------------------

@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_incrementing_every_a_scale_doubles_c_exactly(oracle_mod, fmt):
    K, M, N = 384, 19, 23
    rng = np.random.default_rng(15)
    A, SA = finite_uniform_codes(rng, M, K, fmt, 1, 252)
    B, SB = finite_uniform_codes(rng, N, K, fmt, 1, 252)
    C1, S1 = oracle_mod.gemm(fmt, A, SA, B, SB, K)
    C2, S2 = oracle_mod.gemm(fmt, A, SA + 1, B, SB, K)
    assert (C2 == 2 * C1).all() and (S2 == 2 * S1).all()


def test_nan_scale_poisons_its_row_only(oracle_mod):
    K, M, N = 128, 4, 5
    rng = np.random.default_rng(16)
    A, SA = finite_uniform_codes(rng, M, K, FMT_MXFP8)
    B, SB = finite_uniform_codes(rng, N, K, FMT_MXFP8)
    SA[2, 3] = 0xFF
    C, _ = oracle_mod.gemm(FMT_MXFP8, A, SA, B, SB, K)
    assert np.isnan(C[2]).all()
    assert np.isfinite(np.delete(C, 2, axis=0)).all()


def test_row_and_column_sampling_matches_full(oracle_mod):
    K, M, N = 256, 30, 41
    rng = np.random.default_rng(17)
    A, SA = finite_uniform_codes(rng, M, K, FMT_MXFP4, 120, 130)
    B, SB = finite_uniform_codes(rng, N, K, FMT_MXFP4, 120, 130)
    C, S = oracle_mod.gemm(FMT_MXFP4, A, SA, B, SB, K)
    rows = np.array([29, 0, 7, 7])
    cols = np.array([40, 3])
    Cs, Ss = oracle_mod.gemm(FMT_MXFP4, A, SA, B, SB, K, rows=rows, cols=cols)
    assert (Cs == C[np.ix_(rows, cols)]).all() and (Ss == S[np.ix_(rows, cols)]).all()


def test_rejects_bad_arguments(oracle_mod):
    A = np.zeros((2, 64), np.uint8)
    S = np.full((2, 2), 127, np.uint8)
    with pytest.raises(ValueError):
        oracle_mod.gemm(FMT_MXFP8, A, S, A, S, 64, rows=np.array([2]))
    with pytest.raises(ValueError):
        oracle_mod.gemm(7, A, S, A, S, 64)

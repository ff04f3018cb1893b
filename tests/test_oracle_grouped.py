"""Pins for the oracle's grouped (mixture-of-experts) GEMM (no GPU).

The grouped GEMM is the per-group MX GEMM of the FlyDSL page's grouped-GEMM cases
(English digest, "Performance numbers need their baselines": uniform groups,
projection-dimension changes, uneven expert loads).  Pinned against the dense
reference on stacked and block-diagonal forms, which fix the row/weight pairing
independently of how the grouped routine walks the groups.
"""
import numpy as np
import pytest

from mx_block_scaled_gb300.inputs import FMT_MXFP4, FMT_MXFP8, finite_uniform_codes


def _operands(fmt, T, G, N, K, seed):
    rng = np.random.default_rng(seed)
    A, SA = finite_uniform_codes(rng, T, K, fmt, 120, 134)
    B, SB = finite_uniform_codes(rng, G * N, K, fmt, 120, 134)
    return A, SA, B, SB


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_one_group_is_the_dense_gemm(oracle_mod, fmt):
    A, SA, B, SB = _operands(fmt, 37, 1, 24, 128, 1)
    C, S = oracle_mod.grouped_gemm(fmt, [0, 37], A, SA, B, SB, 24, 128)
    Cd, Sd = oracle_mod.gemm(fmt, A, SA, B, SB, 128)
    assert (C == Cd).all() and (S == Sd).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_each_row_uses_its_own_experts_weight(oracle_mod, fmt):
    """Against the dense product with every expert's weight: row r of group e must
    equal column block e of the dense result (catches an off-by-one group or a
    shifted weight block)."""
    G, N, K = 5, 16, 256
    offsets = [0, 3, 3, 20, 21, 40]           # includes an empty group and a one-row group
    A, SA, B, SB = _operands(fmt, 40, G, N, K, 2)
    C, _ = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K)
    D, _ = oracle_mod.gemm(fmt, A, SA, B, SB, K)   # [40, G*N]
    for e in range(G):
        for r in range(offsets[e], offsets[e + 1]):
            assert (C[r] == D[r, e * N:(e + 1) * N]).all(), (e, r)


def test_rows_outside_groups_are_zero_and_row_selection_matches(oracle_mod):
    fmt, G, N, K = FMT_MXFP8, 3, 8, 128
    offsets = [2, 10, 10, 30]                 # rows 0, 1 and 30..31 belong to no group
    A, SA, B, SB = _operands(fmt, 32, G, N, K, 3)
    C, S = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K)
    assert (C[[0, 1, 30, 31]] == 0).all() and (S[[0, 1, 30, 31]] == 0).all()
    rows = np.array([31, 5, 2, 29, 0])
    Cr, Sr = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K, rows=rows)
    assert (Cr == C[rows]).all() and (Sr == S[rows]).all()


def test_block_diagonal_form(oracle_mod):
    """Grouped = dense GEMM of A with a block-diagonal arrangement: zero every
    K-block of A except those of the row's own group's slot and concatenate the
    expert weights along K."""
    fmt, G, N, K = FMT_MXFP8, 3, 8, 128
    offsets = [0, 4, 9, 12]
    A, SA, B, SB = _operands(fmt, 12, G, N, K, 4)
    C, _ = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K)
    # A' [12, G*K]: row r of group e holds A[r] in K-slot e, zeros elsewhere
    A2 = np.zeros((12, G * K), np.uint8)
    SA2 = np.full((12, G * K // 32), 127, np.uint8)
    for e in range(G):
        for r in range(offsets[e], offsets[e + 1]):
            A2[r, e * K:(e + 1) * K] = A[r]
            SA2[r, e * K // 32:(e + 1) * K // 32] = SA[r]
    # B' [N, G*K]: weight e's row n in K-slot e
    B2 = np.concatenate([B[e * N:(e + 1) * N] for e in range(G)], axis=1)
    SB2 = np.concatenate([SB[e * N:(e + 1) * N] for e in range(G)], axis=1)
    D, _ = oracle_mod.gemm(fmt, A2, SA2, B2, SB2, G * K)
    assert (C == D).all()

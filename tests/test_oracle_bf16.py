"""Pins for the oracle's BF16 NT GEMM (no GPU): the decode against PyTorch's
independent bfloat16 type for every bit pattern, exact integer and rational
products, and the transpose convention."""
from fractions import Fraction

import numpy as np
import torch


def test_decode_of_every_bf16_pattern_matches_torch(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()
    assert (np.signbit(ours[~nan]) == np.signbit(ref[~nan])).all()


def _bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_small_integer_products_are_exact(oracle_mod):
    rng = np.random.default_rng(1)
    A = rng.integers(-8, 9, size=(7, 96)).astype(np.float32)
    B = rng.integers(-8, 9, size=(5, 96)).astype(np.float32)
    C, S = oracle_mod.bf16_gemm(_bits(A), _bits(B))
    exact = A.astype(np.int64) @ B.astype(np.int64).T
    assert (C == exact).all()
    assert (S == np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64).T).all()


def test_rational_values_against_fractions(oracle_mod):
    vals = [0.5, -0.25, 1.5, 3.0, -0.125, 2.0 ** -20, 2.0 ** 20, -7.0]
    rng = np.random.default_rng(2)
    A = np.array(vals, np.float32)[rng.integers(0, len(vals), size=(3, 64))]
    B = np.array(vals, np.float32)[rng.integers(0, len(vals), size=(4, 64))]
    C, _ = oracle_mod.bf16_gemm(_bits(A), _bits(B))
    for i in range(3):
        for j in range(4):
            ref = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(A[i], B[j]))
            assert C[i, j] == float(ref)


def test_nt_convention_and_selection(oracle_mod):
    """C[i, j] = row i of A dotted with row j of B (B is N x K, not K x N)."""
    A = np.zeros((2, 64), np.float32)
    B = np.zeros((3, 64), np.float32)
    A[1, 5] = 2.0
    B[2, 5] = 3.0
    C, _ = oracle_mod.bf16_gemm(_bits(A), _bits(B))
    expect = np.zeros((2, 3))
    expect[1, 2] = 6.0
    assert (C == expect).all()
    Cs, _ = oracle_mod.bf16_gemm(_bits(A), _bits(B), rows=[1], cols=[2, 0])
    assert Cs.tolist() == [[6.0, 0.0]]

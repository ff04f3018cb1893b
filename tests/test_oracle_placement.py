"""Pins for the oracle's scale-placement checker (no GPU).

The checker follows "Deciding Scale Placement in MXFP4 Dot Products with Integer
Arithmetic" (AI-compiler daily digest of 2026-10-22, item 2): pre-scaling (scale
each element, then multiply and sum in binary32) against post-scaling (sum the
exact products in binary32, then apply the scales).  The page does not print the
study's bound, so the bound itself is not pinned; the checker is pinned by
hand-worked tuples and by closed forms derived below.
"""
import math

import numpy as np
import pytest

from golden_io import load_placement_handworked

CASES = load_placement_handworked()


def _same(x, y):
    return (math.isnan(x) and math.isnan(y)) or x == y


@pytest.mark.parametrize("case", CASES, ids=[f"k{c['k']}-{c['sa']}-{c['sb']}-{c['a']}-{c['b']}" for c in CASES])
def test_handworked_tuples(oracle_mod, case):
    t = oracle_mod.placement_tuple(case["k"], case["a"], case["b"])
    pre, post, rn = oracle_mod.placement_eval(case["k"], case["sa"], case["sb"], t)
    assert _same(pre, case["pre"]) and _same(post, case["post"]) and _same(rn, case["rn"]), (pre, post, rn)


@pytest.mark.parametrize("k", [1, 2, 3])
def test_unit_scales_agree_everywhere(oracle_mod, k):
    """sa = sb = 127: every product and partial sum is a small multiple of 1/4,
    exact in binary32, so pre = post = rn for all 16^(2k) tuples."""
    counts, first = oracle_mod.placement_scan(k, [127], [127])
    n = 16 ** (2 * k)
    assert counts.tolist() == [[0, n, n]] and first.tolist() == [-1]


@pytest.mark.parametrize("sa", [0, 60, 127, 200, 248])
@pytest.mark.parametrize("sb", [0, 127, 254])
def test_post_is_exactly_rounded_when_the_first_scaling_cannot_overflow(oracle_mod, sa, sb):
    """k = 2: the sum s is a multiple of 1/4 with |s| <= 72 < 2^7, so s * 2^(sa-127)
    is exact (>= 2^-129 in magnitude, on the subnormal grid) and finite for
    sa <= 248; the second scaling then rounds once: post == rn for every tuple."""
    counts, _ = oracle_mod.placement_scan(2, [sa], [sb])
    assert counts[0, 2] == 16 ** 4


@pytest.mark.parametrize("sa", [0, 1, 126, 127, 252])
@pytest.mark.parametrize("sb", [0, 100, 200, 252])
def test_single_products_pre_scale_exactly_without_element_overflow(oracle_mod, sa, sb):
    """k = 1: a * 2^(sa-127) is exact for sa <= 252 (|a| <= 6 keeps it below 2^128,
    |a| >= 1/2 keeps it on the subnormal grid), so pre rounds once: pre == rn."""
    counts, _ = oracle_mod.placement_scan(1, [sa], [sb])
    assert counts[0, 1] == 256


def test_element_overflow_breaks_pre_scaling(oracle_mod):
    """k = 1, sa = 254: every tuple with |a| >= 2 and b != 0 overflows the scaled
    element (a * 2^127 >= 2^128) while the exact value a*b*2^(sb-127) need not;
    with sb = 0 the exact values are <= 36 and finite, so exactly those
    (4 magnitudes x 2 signs) x (7 x 2 nonzero b) = 112 tuples, plus the 8 x 2 with
    b = +-0 (inf * 0 = NaN), differ from rn."""
    counts, _ = oracle_mod.placement_scan(1, [254], [0])
    assert counts[0, 1] == 256 - 112 - 16


def test_first_counterexample_is_the_smallest(oracle_mod):
    counts, first = oracle_mod.placement_scan(2, [254], [127])
    assert counts[0, 0] > 0
    t = int(first[0])
    pre, post, _ = oracle_mod.placement_eval(2, 254, 127, t)
    assert not _same(pre, post)
    for u in range(t):
        p2, q2, _ = oracle_mod.placement_eval(2, 254, 127, u)
        assert _same(p2, q2)


def test_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.placement_scan(5, [127], [127])
    with pytest.raises(ValueError):
        oracle_mod.placement_scan(1, [255], [127])


def test_vector_values_agree_with_single_evaluations(oracle_mod):
    v = oracle_mod.placement_values(2, 254, 3)
    rng = np.random.default_rng(4)
    for t in rng.integers(0, 1 << 16, size=64):
        pre, post, rn = oracle_mod.placement_eval(2, 254, 3, int(t))
        assert _same(pre, v[t, 0]) and _same(post, v[t, 1]) and _same(rn, v[t, 2])


def _e2m1(code):
    mag = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0][code & 7]
    return -mag if code & 8 else mag


def test_rn_is_the_exact_rational_value_rounded_once(oracle_mod):
    """The exact value sum a_i b_i * 2^(sa+sb-254) is a multiple of 2^(sa+sb-256)
    with at most 10 significant bits, so Python's exact Fraction -> float is exact
    and numpy's binary32 conversion rounds it once (to nearest even, subnormals and
    overflow to infinity included): an independent statement of rn."""
    from fractions import Fraction
    rng = np.random.default_rng(17)
    for _ in range(400):
        k = int(rng.integers(1, 4))
        sa, sb = int(rng.integers(0, 255)), int(rng.integers(0, 255))
        a = [int(x) for x in rng.integers(0, 16, size=k)]
        b = [int(x) for x in rng.integers(0, 16, size=k)]
        exact = sum(Fraction(_e2m1(x)) * Fraction(_e2m1(y)) for x, y in zip(a, b)) * Fraction(2) ** (sa + sb - 254)
        with np.errstate(over="ignore"):
            want = float(np.float32(float(exact)))
        _, _, rn = oracle_mod.placement_eval(k, sa, sb, oracle_mod.placement_tuple(k, a, b))
        assert _same(rn, want), (k, sa, sb, a, b, rn, want)


@pytest.mark.parametrize("sa,sb", [(254, 127), (0, 30), (250, 1), (127, 127)])
def test_counts_are_recounts_of_single_evaluations(oracle_mod, sa, sb):
    """Brute force: the scan's counts and first counterexample equal a recount of
    every tuple's individually evaluated values."""
    v = oracle_mod.placement_values(2, sa, sb)
    pre, post, rn = v[:, 0], v[:, 1], v[:, 2]

    def same(x, y):
        return (np.isnan(x) & np.isnan(y)) | (x == y)
    d = ~same(pre, post)
    counts, first = oracle_mod.placement_scan(2, [sa], [sb])
    assert counts[0].tolist() == [int(d.sum()), int(same(pre, rn).sum()), int(same(post, rn).sum())]
    assert first[0] == (int(np.argmax(d)) if d.any() else -1)


@pytest.mark.parametrize("sa,sb", [(254, 3), (0, 200), (126, 129)])
def test_pre_and_rn_are_symmetric_in_the_operands(oracle_mod, sa, sb):
    """Swapping the operands (codes and scales) leaves every product (a f_a)(b f_b)
    and the exact value unchanged, so pre and rn of tuple (a, b) at (sa, sb) equal
    those of (b, a) at (sb, sa); post is not symmetric (f_a is applied first)."""
    v1 = oracle_mod.placement_values(2, sa, sb)
    v2 = oracle_mod.placement_values(2, sb, sa)
    t = np.arange(1 << 16)
    swapped = (t >> 8) | ((t & 255) << 8)
    for col in (0, 2):
        x, y = v1[:, col], v2[swapped, col]
        assert ((np.isnan(x) & np.isnan(y)) | (x == y)).all()

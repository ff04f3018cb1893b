"""Checks of the synthetic-input generator (no GPU).

The quantiser is the step before the GEMM; these tests check it follows the
stated recipe (E8M0 exponent floor(log2 amax) - e_max, RNE, saturation), using
PyTorch's float8 decoder and the E2M1 magnitude set as independent decoders.
"""
import numpy as np
import pytest
import torch

from mx_block_scaled_gb300.inputs import (FMT_MXFP4, FMT_MXFP8, WORKLOADS, make_operand,
                                          pack_fp4, quantize_mx, unpack_fp4, workload_cases,
                                          with_outlier_blocks)

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def dec_e4m3(c):
    return torch.from_numpy(np.ascontiguousarray(c, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def dec_e2m1(c):
    c = np.asarray(c, np.int64)
    return np.where(c & 8, -E2M1[c & 7], E2M1[c & 7])


def block(values, fill=0.0):
    x = np.full((1, 32), fill, np.float32)
    x[0, :len(values)] = values
    return x


def test_e4m3_rounding_ties_to_even_and_saturation():
    # amax = 256 -> floor(log2) = 8 -> scale 2^0 (code 127); values map 1:1 onto E4M3.
    vals = [256.0, 1.0625, 1.1875, 300.0, 2.0 ** -10, 3 * 2.0 ** -10, -0.0]
    codes, scales = quantize_mx(block(vals), FMT_MXFP8)
    assert scales[0, 0] == 127
    d = dec_e4m3(codes[0, :len(vals)])
    # 1.0625 is a tie between 1.0 and 1.125 -> even mantissa (1.0);
    # 1.1875 ties 1.125 / 1.25 -> 1.25; 300 -> 288 (grid step 32 in [256,512));
    # 2^-10 ties 0 / 2^-9 -> 0; 3*2^-10 ties 2^-9 / 2^-8 -> 2^-8.
    assert d.tolist() == [256.0, 1.0, 1.25, 288.0, 0.0, 2.0 ** -8, -0.0]
    assert np.signbit(d[6])
    # amax 480 -> floor(log2) = 8 -> scale 2^0; 480 saturates to 448.
    codes, scales = quantize_mx(block([480.0, -500.0]), FMT_MXFP8)
    assert scales[0, 0] == 127 and dec_e4m3(codes[0, :2]).tolist() == [448.0, -448.0]


def test_e2m1_rounding_ties_to_even_and_saturation():
    # amax = 7 -> floor(log2) = 2 -> scale exponent 0 -> code 127.
    vals = [7.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, -0.2]
    codes, scales = quantize_mx(block(vals), FMT_MXFP4)
    assert scales[0, 0] == 127
    d = dec_e2m1(unpack_fp4(codes)[0, :len(vals)])
    assert d.tolist() == [6.0, 0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -4.0, -0.0]


@pytest.mark.parametrize("fmt,e_max", [(FMT_MXFP8, 8), (FMT_MXFP4, 2)])
def test_scale_exponent_is_floor_log2_amax_minus_emax(fmt, e_max):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 256), dtype=np.float32)
    x[5, :32] = 0.0                                     # all-zero block -> code 127
    _, scales = quantize_mx(x, fmt)
    amax = np.abs(x.astype(np.float64)).reshape(64, 8, 32).max(axis=2)
    expect = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - e_max, 0) + 127
    assert (scales == expect).all()
    assert scales[5, 0] == 127


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_dequantised_values_within_half_a_grid_step(fmt):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((32, 512), dtype=np.float32).astype(np.float64)
    codes, scales = quantize_mx(x.astype(np.float32), fmt)
    v = dec_e4m3(codes) if fmt == FMT_MXFP8 else dec_e2m1(unpack_fp4(codes))
    s = np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32, axis=1)
    deq = v * s
    # the grid step at |x| is at most 2^(floor(log2|x|) - mbits); half of that bounds the error
    mbits = 3 if fmt == FMT_MXFP8 else 1
    floor_exp = np.floor(np.log2(np.maximum(np.abs(x), 1e-300)))
    step = np.maximum(2.0 ** (floor_exp - mbits), s * (2.0 ** -9 if fmt == FMT_MXFP8 else 0.5))
    sat = np.abs(x) > s * (448.0 if fmt == FMT_MXFP8 else 6.0)
    assert (np.abs(deq - x)[~sat] <= step[~sat] / 2 + 1e-300).all()


def test_fp4_pack_roundtrip_and_nibble_order():
    codes = np.arange(32, dtype=np.uint8).reshape(1, 32) & 15
    p = pack_fp4(codes)
    assert p[0, 0] == (0 | (1 << 4)) and p[0, 1] == (2 | (3 << 4))
    assert (unpack_fp4(p) == codes).all()


def test_outlier_blocks_count_and_factor():
    rng = np.random.default_rng(5)
    x = np.ones((10, 320), np.float32)
    y = with_outlier_blocks(x, rng)
    scaled = (y.reshape(-1, 32) == 256.0).all(axis=1)
    assert scaled.sum() == round(0.01 * 100) and (y.reshape(-1, 32)[~scaled] == 1.0).all()


def test_workload_seeds_are_deterministic_and_weights_shared_across_m():
    A1, SA1 = make_operand("llama31_8b", "A", 0, 16, 4096, FMT_MXFP4)
    A2, SA2 = make_operand("llama31_8b", "A", 0, 16, 4096, FMT_MXFP4)
    assert (A1 == A2).all() and (SA1 == SA2).all()
    cases = list(workload_cases("llama33_70b"))
    assert len(cases) == 2 * 4 * 4
    assert {c[0] for c in cases} == {"mxfp8", "mxfp4"}
    assert all(set(w) >= {"cfg", "fmts", "out", "values", "nks", "ms"} for w in WORKLOADS.values())

"""Pins for the oracle's MX quantiser (no GPU).

The quantiser is the step before the GEMM; the FlyDSL page (English digest,
"Performance numbers need their baselines") leaves it outside the timed region
and prints no formula, so its recipe is a reading (stated in ``oracle/mxref.c``).
Each test below checks the oracle against something other than itself:
hand-worked blocks (``tests/golden/quantize_handworked.txt``), a brute-force
nearest-value search over the element grid decoded by PyTorch's independent
float8 decoders, the exact binade bound on the scale, and PyTorch's BF16
widening.
"""
import numpy as np
import pytest
import torch

from golden_io import load_quantize_handworked
from mx_block_scaled_gb300.inputs import FMT_MXFP4, FMT_MXFP8, unpack_fp4
from test_oracle import e2m1_from_set, torch_e4m3

HANDWORKED = load_quantize_handworked()
E_MAX = {FMT_MXFP8: 8, FMT_MXFP4: 2}


def element_codes(fmt, codes):
    """One code per element: bytes for MXFP8, unpacked nibbles for MXFP4."""
    return codes if fmt == FMT_MXFP8 else unpack_fp4(codes)


def decode(fmt, codes):
    return torch_e4m3(codes) if fmt == FMT_MXFP8 else e2m1_from_set(codes)


def to_bf16_bits(x32):
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", HANDWORKED, ids=[c["name"] for c in HANDWORKED])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_handworked_blocks(oracle_mod, case, src):
    if src == "bf16":
        if not case["bf16"]:
            pytest.skip("inputs not exact in BF16")
        x, dt = to_bf16_bits(case["x"]), oracle_mod.IN_BF16
    else:
        x, dt = case["x"], oracle_mod.IN_F32
    codes, scales = oracle_mod.quantize(case["fmt"], x, dt)
    assert scales.tolist() == [[case["scale"]]]
    assert element_codes(case["fmt"], codes)[0].tolist() == case["codes"].tolist()


def _grid(fmt):
    """Every finite, non-negative grid value with its code (from the independent decoders)."""
    if fmt == FMT_MXFP8:
        c = np.arange(0x7F, dtype=np.uint8)          # 0x00..0x7E: +0 .. 448
    else:
        c = np.arange(8, dtype=np.uint8)             # 0..7: +0 .. 6
    return decode(fmt, c), c


def _brute_nearest(fmt, v):
    """Nearest grid value to |v| by exhaustive search, ties to the even code,
    sign copied from v; returns element codes."""
    g, gc = _grid(fmt)
    d = np.abs(np.abs(v)[..., None] - g)             # exact in float64 (dyadic values)
    best = d.min(axis=-1, keepdims=True)
    cand = (d == best)
    even = cand & (gc % 2 == 0)
    pick = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    code = gc[pick].astype(np.uint8)
    sign = np.signbit(v)
    return code | (sign.astype(np.uint8) << (7 if fmt == FMT_MXFP8 else 3))


def _wide_range_input(seed, rows, K):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    # per-block magnitudes from 2^-140 (FP32 subnormal) to 2^120, some exact
    # ties, some exact zeros and negative zeros
    mag = np.ldexp(1.0, rng.integers(-140, 121, size=(rows, K // 32)))
    x = (x * np.repeat(mag, 32, axis=1)).astype(np.float32)
    ties = rng.random((rows, K)) < 0.1
    x[ties] = np.ldexp(rng.integers(-20, 20, size=ties.sum()) + 0.5, -3).astype(np.float32)
    x[rng.random((rows, K)) < 0.02] = 0.0
    x[rng.random((rows, K)) < 0.02] = -0.0
    return x


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_codes_are_brute_force_nearest_grid_values(oracle_mod, fmt):
    x = _wide_range_input(11 + fmt, 48, 1024)
    codes, scales = oracle_mod.quantize(fmt, x)
    s = scales.astype(np.int64) - 127
    v = np.ldexp(x.astype(np.float64), -np.repeat(s, 32, axis=1))
    expect = _brute_nearest(fmt, v)
    assert (element_codes(fmt, codes) == expect).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_scale_puts_amax_in_the_top_binade(oracle_mod, fmt):
    x = _wide_range_input(21 + fmt, 48, 1024)
    _, scales = oracle_mod.quantize(fmt, x)
    amax = np.abs(x.astype(np.float64)).reshape(48, 32, 32).max(axis=2)
    s = scales.astype(np.int64) - 127
    scaled = np.ldexp(amax, -s)
    free = (amax > 0) & (s > -127)
    # 2^e_max <= amax / 2^s < 2^(e_max + 1) unless clamped at s = -127
    assert (scaled[free] >= 2.0 ** E_MAX[fmt]).all()
    assert (scaled[free] < 2.0 ** (E_MAX[fmt] + 1)).all()
    clamped = (amax > 0) & (s == -127)
    assert (scaled[clamped] < 2.0 ** (E_MAX[fmt] + 1)).all()
    assert (scales[amax == 0] == 127).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_dequantised_error_is_at_most_half_a_grid_step(oracle_mod, fmt):
    rng = np.random.default_rng(31)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    codes, scales = oracle_mod.quantize(fmt, x)
    deq = decode(fmt, element_codes(fmt, codes)) * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    mbits = 3 if fmt == FMT_MXFP8 else 1
    emin = -6 if fmt == FMT_MXFP8 else 0
    s = np.repeat(scales.astype(np.int64) - 127, 32, axis=1)
    _, e = np.frexp(np.abs(x.astype(np.float64)) * np.ldexp(1.0, -s))
    step = np.ldexp(1.0, np.maximum(e - 1, emin) - mbits + s)
    vmax = 448.0 if fmt == FMT_MXFP8 else 6.0
    over = np.abs(x) > vmax * np.ldexp(1.0, s)
    err = np.abs(deq - x)
    assert (err[~over] <= step[~over] / 2).all()
    assert (np.abs(deq[over]) == (vmax * np.ldexp(1.0, s))[over]).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_bf16_input_equals_its_fp32_widening(oracle_mod, fmt):
    rng = np.random.default_rng(41)
    bits = rng.integers(0, 1 << 16, size=(32, 256), dtype=np.uint16)
    wide = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    c16, s16 = oracle_mod.quantize(fmt, bits, oracle_mod.IN_BF16)
    c32, s32 = oracle_mod.quantize(fmt, wide, oracle_mod.IN_F32)
    assert (c16 == c32).all() and (s16 == s32).all()
    # uniform bit patterns include NaN and infinity: those blocks carry the NaN scale
    bad = ~np.isfinite(wide).reshape(32, 8, 32).all(axis=2)
    assert bad.any() and (s16[bad] == 255).all() and (s16[~bad] != 255).all()


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_MXFP4])
def test_nonfinite_block_leaves_neighbours_alone(oracle_mod, fmt):
    rng = np.random.default_rng(51)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    ref_c, ref_s = oracle_mod.quantize(fmt, x)
    y = x.copy()
    y[2, 64 + 5] = np.nan
    y[3, 31] = -np.inf
    c, s = oracle_mod.quantize(fmt, y)
    assert s[2, 2] == 255 and s[3, 0] == 255
    mask = np.ones_like(s, dtype=bool)
    mask[2, 2] = mask[3, 0] = False
    assert (s[mask] == ref_s[mask]).all()
    ec, rc = element_codes(fmt, c), element_codes(fmt, ref_c)
    assert (ec[2, 64:96] == 0).all() and (ec[3, 0:32] == 0).all()
    keep = np.ones_like(ec, dtype=bool)
    keep[2, 64:96] = keep[3, 0:32] = False
    assert (ec[keep] == rc[keep]).all()


def test_quantize_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.quantize(FMT_MXFP8, np.zeros((2, 48), np.float32))   # K % 32
    with pytest.raises(ValueError):
        oracle_mod.quantize(3, np.zeros((2, 64), np.float32))

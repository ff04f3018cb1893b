"""GPU parity of the MX quantiser (mxgemm_quantize) against the oracle's.

Codes and scales are bytes, so the bar is bit-exact equality with
``oracle.quantize`` on the same inputs.  The tile-layout output is checked
against the documented index formula applied to the oracle's row-major
scales, and the quantise -> GEMM chain against the GEMM fed with the same
codes and row-major scales.
"""
import numpy as np
import pytest

from gpu_util import OUT_BF16, OUT_F32, assert_within, lib, tile_sample_indices, to_dev
from mx_block_scaled_gb300.inputs import FMT_MXFP4, FMT_MXFP8, with_outlier_blocks
from test_gemm_gpu import relayout_reference
from test_oracle_quantize import _wide_range_input

pytestmark = pytest.mark.gpu

FMTS = [FMT_MXFP8, FMT_MXFP4]
SRCS = ["f32", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3)
    lib()


def _bf16_bits(x32):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _device_input(x32, src):
    """The device tensor for `src` and the host array the oracle reads."""
    import torch
    if src == "bf16":
        bits = _bf16_bits(x32)
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16), bits
    return to_dev(x32), x32


def _oracle(oracle_mod, fmt, host, src):
    return oracle_mod.quantize(fmt, host, oracle_mod.IN_BF16 if src == "bf16" else oracle_mod.IN_F32)


def _gpu(fmt, dx, tiled=False):
    import torch
    b = lib()
    codes, scales = b.quantize(dx, fmt, tiled=tiled)
    b.check_device_status()
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def _with_nonfinite_blocks(x, seed):
    rng = np.random.default_rng(seed)
    y = x.copy()
    n = max(1, y.size // 4096)
    pos = rng.integers(0, y.size, size=n)
    y.reshape(-1)[pos] = rng.choice(np.array([np.nan, np.inf, -np.inf], np.float32), size=n)
    return y


# ---- bit-exact parity, ragged shapes --------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("src", SRCS)
@pytest.mark.parametrize("rows,K", [(1, 32), (3, 96), (7, 544), (129, 1056), (300, 4096), (64, 5152)])
def test_quantize_bit_exact(oracle_mod, fmt, src, rows, K):
    x = _with_nonfinite_blocks(_wide_range_input(rows * 31 + K, rows, K), rows + K)
    dx, host = _device_input(x, src)
    c_ref, s_ref = _oracle(oracle_mod, fmt, host, src)
    c, s = _gpu(fmt, dx)
    assert s.shape == s_ref.shape and (s == s_ref).all(), np.argwhere(s != s_ref)[:5].tolist()
    bad = np.argwhere(c != c_ref)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first {bad[:5].tolist()}"


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_bit_pattern(oracle_mod, fmt):
    """All 65536 BF16 patterns shuffled into 32-blocks (NaN/Inf blocks included),
    then the same with the NaN/Inf patterns made finite."""
    rng = np.random.default_rng(7)
    bits = rng.permutation(np.arange(1 << 16, dtype=np.uint32)).astype(np.uint16).reshape(256, 256)
    import torch
    c_ref, s_ref = oracle_mod.quantize(fmt, bits, oracle_mod.IN_BF16)
    c, s = _gpu(fmt, torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16))
    assert (s == 255).any()
    assert (s == s_ref).all() and (c == c_ref).all()
    # finite only: clear the exponent-all-ones patterns, so every block has a real scale
    fin = bits.copy()
    fin[(fin & 0x7F80) == 0x7F80] &= np.uint16(0x807F)
    c_ref, s_ref = oracle_mod.quantize(fmt, fin, oracle_mod.IN_BF16)
    c, s = _gpu(fmt, torch.from_numpy(fin.view(np.int16)).cuda().view(torch.bfloat16))
    assert (s != 255).all()
    assert (s == s_ref).all() and (c == c_ref).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_random_fp32_bit_patterns(oracle_mod, fmt):
    rng = np.random.default_rng(8)
    bits = rng.integers(0, 1 << 32, size=(512, 2048), dtype=np.uint64).astype(np.uint32)
    # keep most blocks finite: clear the top exponent bit on 7 of 8 elements
    bits[:, np.arange(2048) % 8 != 0] &= np.uint32(0xBFFFFFFF)
    x = bits.view(np.float32)
    c_ref, s_ref = oracle_mod.quantize(fmt, x)
    c, s = _gpu(fmt, to_dev(x))
    assert (s == s_ref).all() and (c == c_ref).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_handworked_blocks_on_the_gpu(fmt):
    from golden_io import load_quantize_handworked
    from mx_block_scaled_gb300.inputs import unpack_fp4
    for case in load_quantize_handworked():
        if case["fmt"] != fmt:
            continue
        for src in SRCS:
            dx, _ = _device_input(case["x"], src)
            c, s = _gpu(fmt, dx)
            codes = c if fmt == FMT_MXFP8 else unpack_fp4(c)
            assert s.tolist() == [[case["scale"]]], case["name"]
            assert codes[0].tolist() == case["codes"].tolist(), (case["name"], src)


# ---- tile layout ----------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("src", SRCS)
@pytest.mark.parametrize("rows,K", [(1, 128), (127, 256), (129, 640), (300, 4096), (8, 28672)])
def test_tiled_scales_match_the_index_formula(oracle_mod, fmt, src, rows, K):
    x = _wide_range_input(rows + 3 * K, rows, K)
    dx, host = _device_input(x, src)
    c_ref, s_ref = _oracle(oracle_mod, fmt, host, src)
    c, t = _gpu(fmt, dx, tiled=True)
    assert (c == c_ref).all()
    assert t.size == lib().mxgemm_sf_bytes(rows, K)
    if rows * K <= 300 * 4096:
        assert (t == relayout_reference(s_ref, rows, K)).all()
    else:
        r = np.arange(rows)[:, None]
        j = np.arange(K // 32)[None, :]
        pos = ((r // 128) * (K // 128) + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4
        assert (t[pos] == s_ref).all()
        pad = np.ones(t.size, bool)
        pad[pos.reshape(-1)] = False
        assert (t[pad] == 127).all()


# ---- quantise -> GEMM ------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(8, 1024, 2048), (200, 328, 1024), (1024, 768, 512)])
def test_quantize_then_gemm_with_tiled_scales(oracle_mod, fmt, M, N, K):
    """BF16 activations and weights quantised on the GPU, scales straight in the
    tile layout, the GEMM run with both operands pre-laid-out: same C as the
    GEMM fed the row-major scales, and within the bound of the oracle GEMM on
    the oracle's codes."""
    import torch
    b = lib()
    rng = np.random.default_rng(M + N + K)
    xa = rng.standard_normal((M, K), dtype=np.float32)
    xb = rng.standard_normal((N, K), dtype=np.float32)
    da, ha = _device_input(xa, "bf16")
    db, hb = _device_input(xb, "bf16")
    A, SA = b.quantize(da, fmt)
    B, SB = b.quantize(db, fmt)
    _, tSA = b.quantize(da, fmt, tiled=True)
    _, tSB = b.quantize(db, fmt, tiled=True)
    plan = b.Plan(M, N, K, fmt, OUT_F32)
    C1 = plan.run(A, SA, B, SB)
    C2 = plan.run(A, tSA, B, tSB, run_flags=b.MXGEMM_RUN_SA_PRELAYOUT | b.MXGEMM_RUN_SB_PRELAYOUT)
    b.check_device_status()
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    rA, rSA = oracle_mod.quantize(fmt, ha, oracle_mod.IN_BF16)
    rB, rSB = oracle_mod.quantize(fmt, hb, oracle_mod.IN_BF16)
    C_ref, S = oracle_mod.gemm(fmt, rA, rSA, rB, rSB, K)
    assert_within(C2.double().cpu().numpy(), C_ref, S, OUT_F32, f"quantize+gemm {M}x{N}x{K}")


# ---- the served models' activation shapes at full size ---------------------------

ACT_SHAPES = [  # (workload, M, K): the largest token count of each (N,K) weight family
    ("llama31_8b", 8192, 4096), ("llama31_8b", 8192, 14336),
    ("llama33_70b", 8, 8192), ("llama33_70b", 16384, 8192), ("llama33_70b", 16384, 28672),
    ("qwen3_32b", 4096, 5120), ("qwen3_32b", 4096, 25600),
]


@pytest.mark.parametrize("name,M,K", ACT_SHAPES)
def test_activation_shapes_full_size_sampled(oracle_mod, name, M, K):
    """Full-size BF16 activations (N(0,1); the 32B model's with 1% outlier
    blocks x2^8), quantised to both formats with tiled scales; sampled rows
    against the oracle, bit-exact."""
    import torch
    rng = np.random.default_rng([len(name), M, K])
    x = rng.standard_normal((M, K), dtype=np.float32)
    if name == "qwen3_32b":
        x = with_outlier_blocks(x, rng)
    bits = _bf16_bits(x)
    del x
    dx = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    rows = tile_sample_indices(M, M + K)  # one row in every 128-row scale tile
    r = rows[:, None]
    j = np.arange(K // 32)[None, :]
    pos = ((r // 128) * (K // 128) + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4
    b = lib()
    for fmt in FMTS:
        codes, tiled = b.quantize(dx, fmt, tiled=True)
        b.check_device_status()
        torch.cuda.synchronize()
        c_ref, s_ref = oracle_mod.quantize(fmt, bits[rows], oracle_mod.IN_BF16)
        assert (codes[torch.from_numpy(rows).cuda()].cpu().numpy() == c_ref).all(), fmt
        assert (tiled.cpu().numpy()[pos] == s_ref).all(), fmt
        del codes, tiled

"""GPU parity of the BF16 NT GEMM (the same kernels with kind::f16 MMAs and no
scales) against the oracle's BF16 reference.

Exact where every partial sum is representable in FP32 (small integer and
half-integer operands); elsewhere within |C - C_ref| <= 1e-5 * sum|a*b|
(+ 2^-8 |C_ref| for BF16 output).
"""
import numpy as np
import pytest

from gpu_util import OUT_BF16, OUT_F32, assert_within, lib, tile_sample_indices

pytestmark = pytest.mark.gpu

FMT_BF16 = 3
BN128, BN256, NOSWAP, SWAP, PAIR, SINGLE = 1 << 0, 1 << 1, 1 << 2, 1 << 3, 1 << 4, 1 << 5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3)
    lib()


def _bits(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _gemm(A_bits, B_bits, out, flags=0):
    import torch
    b = lib()
    M, K = A_bits.shape
    N = B_bits.shape[0]
    plan = b.Plan(M, N, K, FMT_BF16, out, flags)
    C = plan.run(_dev(A_bits), None, _dev(B_bits), None)
    b.check_device_status()
    torch.cuda.synchronize()
    return C.float().double().cpu().numpy(), plan.describe()


def _small(rng, rows, K):
    vals = np.array([0.0, 0.5, 1.0, 2.0, -0.5, -1.0, -2.0], np.float32)
    return _bits(vals[rng.integers(0, len(vals), size=(rows, K))])


def _bf16_round(x):
    import torch
    return torch.from_numpy(x.astype(np.float32)).bfloat16().double().numpy()


@pytest.mark.parametrize("flags", [0, SINGLE, PAIR, SWAP, NOSWAP | BN128, SINGLE | BN256, 3 << 8])
@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (8, 129, 192), (127, 255, 256), (129, 8, 64), (255, 300, 1024),
                                   (300, 520, 640), (64, 512, 2048)])
def test_bf16_exact(oracle_mod, flags, M, N, K):
    if (flags & PAIR) and min(M, N) < 128:
        pytest.skip("CTA-pair tiles are for shapes with at least 128 rows on each side")
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A, B = _small(rng, M, K), _small(rng, N, K)
    ref, _ = oracle_mod.bf16_gemm(A, B)
    for out in (OUT_F32, OUT_BF16):
        C, desc = _gemm(A, B, out, flags)
        expect = ref if out == OUT_F32 else _bf16_round(ref)
        assert (C == expect).all(), f"{M}x{N}x{K} {desc}"


@pytest.mark.parametrize("flags", [0, SINGLE, 1 << 7])
def test_bf16_normal_values_within_bound(oracle_mod, flags):
    rng = np.random.default_rng(11)
    M, N, K = 640, 1152, 4096
    A = _bits(rng.standard_normal((M, K), dtype=np.float32))
    B = _bits(rng.standard_normal((N, K), dtype=np.float32))
    ref, S = oracle_mod.bf16_gemm(A, B)
    C, desc = _gemm(A, B, OUT_F32, flags)
    assert_within(C, ref, S, OUT_F32, desc)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (8, 57344, 8192), (16384, 8192, 8192), (4096, 5120, 25600)])
def test_bf16_full_size_sampled(oracle_mod, M, N, K):
    import torch
    rng = np.random.default_rng([M, N, K])
    A = _bits(rng.standard_normal((M, K), dtype=np.float32))
    B = _bits(rng.standard_normal((N, K), dtype=np.float32))
    b = lib()
    plan = b.Plan(M, N, K, FMT_BF16, OUT_BF16)
    C = plan.run(_dev(A), None, _dev(B), None)
    b.check_device_status()
    torch.cuda.synchronize()
    # every 128-row and every 128-column tile of the plan holds a sampled row / column
    rows, cols = tile_sample_indices(M, M + 1), tile_sample_indices(N, N + 2)
    ref_r, S_r = oracle_mod.bf16_gemm(A, B, rows=rows)
    got_r = C[torch.from_numpy(rows).cuda()].float().double().cpu().numpy()
    assert_within(got_r, ref_r, S_r, OUT_BF16, f"rows {plan.describe()}")
    ref_c, S_c = oracle_mod.bf16_gemm(A, B, cols=cols)
    got_c = C[:, torch.from_numpy(cols).cuda()].float().double().cpu().numpy()
    assert_within(got_c, ref_c, S_c, OUT_BF16, f"cols {plan.describe()}")


@pytest.mark.parametrize("M,N,K", [(256, 1000, 512), (300, 2000, 1024)])
def test_bf16_pair_192_wide_tiles_exact(oracle_mod, M, N, K):
    """BF16 on 256 x 192 CTA-pair tiles (MXGEMM_PLAN_FORCE_BN192), exact against the
    oracle in FP32 and BF16 out."""
    rng = np.random.default_rng(M + N + K + 192)
    A, B = _small(rng, M, K), _small(rng, N, K)
    ref, _ = oracle_mod.bf16_gemm(A, B)
    for out in (OUT_F32, OUT_BF16):
        C, desc = _gemm(A, B, out, (1 << 17) | (1 << 8))
        expect = ref if out == OUT_F32 else _bf16_round(ref)
        assert "tile=256x192" in desc, desc
        assert (C == expect).all(), f"{M}x{N}x{K} {desc}"


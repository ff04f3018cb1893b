"""GPU parity of the scale-placement checker (mxgemm_placement_scan) against the
oracle's checker: counts and first counterexamples are integers, so the bar is
exact equality."""
import numpy as np
import pytest

from gpu_util import lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3)
    lib()


def _gpu_scan(k, sa, sb):
    import torch
    b = lib()
    dsa = torch.tensor(np.asarray(sa, np.int32), device="cuda")
    dsb = torch.tensor(np.asarray(sb, np.int32), device="cuda")
    counts, first = b.placement_scan(k, dsa, dsb)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), first.cpu().numpy()


def test_k1_every_scale_pair(oracle_mod):
    sa, sb = np.meshgrid(np.arange(255), np.arange(255), indexing="ij")
    sa, sb = sa.reshape(-1), sb.reshape(-1)
    c_ref, f_ref = oracle_mod.placement_scan(1, sa, sb)
    c, f = _gpu_scan(1, sa, sb)
    assert (c == c_ref).all() and (f == f_ref).all()


@pytest.mark.parametrize("band", ["low", "unit", "high", "mixed"])
def test_k2_scale_bands(oracle_mod, band):
    rng = np.random.default_rng(len(band))
    if band == "low":
        sa, sb = rng.integers(0, 12, 400), rng.integers(0, 12, 400)
    elif band == "unit":
        sa, sb = rng.integers(110, 145, 400), rng.integers(110, 145, 400)
    elif band == "high":
        sa, sb = rng.integers(190, 255, 400), rng.integers(190, 255, 400)
    else:
        sa, sb = rng.integers(0, 255, 400), rng.integers(0, 255, 400)
    c_ref, f_ref = oracle_mod.placement_scan(2, sa, sb)
    c, f = _gpu_scan(2, sa, sb)
    assert (c == c_ref).all() and (f == f_ref).all()


def test_k3_selected_pairs(oracle_mod):
    sa = [127, 254, 0, 200, 60, 250]
    sb = [127, 0, 254, 200, 60, 2]
    c_ref, f_ref = oracle_mod.placement_scan(3, sa, sb)
    c, f = _gpu_scan(3, sa, sb)
    assert (c == c_ref).all() and (f == f_ref).all()


def test_invalid_codes_are_flagged():
    c, f = _gpu_scan(1, [255, 127, -1], [127, 127, 3])
    assert (c[0] == -1).all() and f[0] == -1 and (c[2] == -1).all() and f[2] == -1
    assert c[1].tolist() == [0, 256, 256] and f[1] == -1


def test_mxfp4_mma_is_exact_then_truncated_below_the_normal_range(oracle_mod):
    """HARDWARE CHARACTERISATION, not parity: it records what the MXFP4 tensor
    cores do with results below the FP32 normal range, where the GEMM leaves
    the FP32-accumulation bound (the parity tests never go there).

    Replay of every k = 2 tuple through the MXFP4 tensor-core GEMM: A rows are
    all 256 (a0, a1) code pairs and B rows all 256 (b0, b1) pairs, placed at K
    positions 0 and 1 of block 0 (the rest zero), with block-0 scale codes sa / sb
    across the range.  C[i, j] is the hardware's value of tuple i | j << 8.

    The tensor cores follow neither binary32 placement: they form the block's
    dot product exactly.  Where the exact value is in the normal range (for
    k = 2 it is then representable) or overflows, C equals the oracle's exactly
    rounded value (infinity included); below the normal range (|x| < 2^-126) C
    is the exact value truncated toward zero onto the subnormal grid 2^-149,
    where round-to-nearest-even would round up in some cases (1.5 * 2^-149 ->
    2^-149, not 2^-148)."""
    import torch
    from mx_block_scaled_gb300.inputs import FMT_MXFP4, pack_fp4
    from gpu_util import OUT_F32
    b = lib()
    K = 128
    codes = np.zeros((256, K), np.uint8)
    idx = np.arange(256)
    codes[:, 0], codes[:, 1] = idx & 15, idx >> 4
    dA = torch.from_numpy(pack_fp4(codes)).cuda()
    plan = b.Plan(256, 256, K, FMT_MXFP4, OUT_F32)
    E2M1 = oracle_mod.decode_table("e2m1")  # the oracle's (pinned) element values
    t = np.arange(1 << 16)
    dot = E2M1[t & 15] * E2M1[(t >> 8) & 15] + E2M1[(t >> 4) & 15] * E2M1[t >> 12]  # exact in binary64
    picks = [0, 1, 5, 50, 52, 80, 100, 105, 118, 120, 126, 127, 128, 150, 240, 250, 253, 254]
    n_truncated = 0
    for sa in picks:
        for sb in picks:
            SA = np.full((256, K // 32), 127, np.uint8)
            SB = SA.copy()
            SA[:, 0], SB[:, 0] = sa, sb
            C = plan.run(dA, torch.from_numpy(SA).cuda(), dA, torch.from_numpy(SB).cuda())
            b.check_device_status()
            got = C.cpu().numpy().T.reshape(-1).astype(np.float64)
            exact = dot * 2.0 ** (sa + sb - 254)
            rn = oracle_mod.placement_values(2, sa, sb)[:, 2].astype(np.float64)
            sub = np.abs(exact) < 2.0 ** -126
            expect = np.where(sub, np.trunc(exact * 2.0 ** 149) * 2.0 ** -149, rn)
            same = (np.isnan(got) & np.isnan(expect)) | (got == expect)
            assert same.all(), (sa, sb, int((~same).sum()))
            n_truncated += int((sub & (expect != rn)).sum())
    assert n_truncated > 0  # the replay did reach results where the two roundings differ

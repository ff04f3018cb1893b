"""GPU parity of the grouped (mixture-of-experts) MX GEMM against the oracle's
grouped GEMM (one pinned per-group reference GEMM per group).

Exact equality wherever every partial sum is representable in FP32 (small
integer-valued codes); the full-size workloads within the FP32-accumulation
bound on sampled rows.  Rows outside every group must stay untouched, and
offsets that break the contract (decreasing, negative, past the end) must not
make the kernel touch memory outside its buffers.
"""
import numpy as np
import pytest

from gpu_util import OUT_BF16, OUT_F32, assert_within, lib, to_dev
from mx_block_scaled_gb300.inputs import (FMT_MXFP4, FMT_MXFP8, MOE_WORKLOADS, group_offsets, moe_cases,
                                          normal_f32, quantize_mx)
from test_gemm_gpu import small_int_codes

pytestmark = pytest.mark.gpu

BN128, BN256, NOSWAP, SWAP, PAIR = 1 << 0, 1 << 1, 1 << 2, 1 << 3, 1 << 4
FMTS = [FMT_MXFP8, FMT_MXFP4]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3)
    lib()


def _run(fmt, offsets, A, SA, B, SB, N, K, out, flags=0, sb_pre=False, C=None):
    """Grouped GEMM through the C ABI; returns (C as float64 numpy, plan text)."""
    import torch
    b = lib()
    T, G = A.shape[0], len(offsets) - 1
    plan = b.GroupedPlan(G, T, N, K, fmt, out, flags)
    d_off = torch.tensor(np.asarray(offsets, dtype=np.int64), device="cuda")
    dB, dSB = to_dev(B), to_dev(SB)
    run_flags = 0
    if sb_pre:
        dSB = b.relayout_scales(dSB, B.shape[0], K)
        run_flags = b.MXGEMM_RUN_SB_PRELAYOUT
    if C is None:
        C = torch.full((T, N), float("nan"), dtype=torch.bfloat16 if out == OUT_BF16 else torch.float32,
                       device="cuda")
    plan.run(d_off, to_dev(A), to_dev(SA), dB, dSB, C, run_flags=run_flags)
    b.check_device_status()
    torch.cuda.synchronize()
    return C.float().double().cpu().numpy(), plan.describe()


def _in_groups(offsets, T):
    mask = np.zeros(T, bool)
    for e in range(len(offsets) - 1):
        mask[offsets[e]:offsets[e + 1]] = True
    return mask


def _bf16(x):
    import torch
    return torch.from_numpy(x.astype(np.float32)).bfloat16().double().numpy()


CASES = [
    # (groups sizes, N, K, leading gap rows, trailing gap rows)
    ([64, 64, 64, 64], 256, 256, 0, 0),
    ([0, 1, 127, 128, 129, 300], 384, 512, 0, 0),
    ([5, 0, 33, 0, 200], 128, 1024, 7, 9),
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("flags", [0, SWAP, NOSWAP, NOSWAP | BN128, SWAP | BN128, SWAP | BN256, PAIR])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_grouped_exact(oracle_mod, fmt, flags, case):
    sizes, N, K, lead, trail = CASES[case]
    offsets = list(lead + group_offsets(sizes))
    T = offsets[-1] + trail
    G = len(sizes)
    rng = np.random.default_rng([case, flags, fmt])
    A, SA = small_int_codes(rng, T, K, fmt)
    B, SB = small_int_codes(rng, G * N, K, fmt)
    ref, _ = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K)
    inside = _in_groups(offsets, T)
    for out in (OUT_F32, OUT_BF16):
        C, desc = _run(fmt, offsets, A, SA, B, SB, N, K, out, flags)
        expect = ref if out == OUT_F32 else _bf16(ref)
        assert (C[inside] == expect[inside]).all(), desc
        assert np.isnan(C[~inside]).all(), f"rows outside every group were written: {desc}"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("G", [33, 100])
def test_many_small_groups_exact(oracle_mod, fmt, G):
    """More groups than one warp scans at a time, many of them empty or tiny."""
    rng = np.random.default_rng([G, fmt])
    sizes = rng.integers(0, 12, size=G)
    sizes[rng.integers(0, G, size=G // 4)] = 0
    offsets = list(group_offsets(sizes))
    T = offsets[-1]
    N, K = 256, 256
    A, SA = small_int_codes(rng, T, K, fmt)
    B, SB = small_int_codes(rng, G * N, K, fmt)
    ref, _ = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K)
    for flags in (0, NOSWAP):
        C, desc = _run(fmt, offsets, A, SA, B, SB, N, K, OUT_F32, flags)
        assert (C == ref).all(), desc


@pytest.mark.parametrize("fmt", FMTS)
def test_prelayout_weight_scales_give_the_same_result(fmt):
    rng = np.random.default_rng(5)
    sizes, N, K = [40, 0, 90, 3], 256, 512
    offsets = list(group_offsets(sizes))
    T, G = offsets[-1], len(sizes)
    A, SA = small_int_codes(rng, T, K, fmt)
    B, SB = small_int_codes(rng, G * N, K, fmt)
    C1, _ = _run(fmt, offsets, A, SA, B, SB, N, K, OUT_F32)
    C2, _ = _run(fmt, offsets, A, SA, B, SB, N, K, OUT_F32, sb_pre=True)
    assert (C1 == C2).all()


def _sanitised(offsets, T):
    """The kernel's reading of arbitrary offsets: group e starts at offsets[e]
    clamped to [0, T] and not before any earlier group's end, and ends at
    offsets[e+1] clamped to [start, T]."""
    out, prev_end = [], 0
    for e in range(len(offsets) - 1):
        s = min(max(offsets[e], 0), T)
        end = min(max(offsets[e + 1], s), T)
        s2 = max(s, prev_end)
        end2 = max(end, s2)
        out.append((s2, end2))
        prev_end = max(prev_end, end)
    return out


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("bad", [[0, 50, 20, 90, 60], [-40, 30, 30, 500, 70], [10, 200, 5, 5, 7]])
def test_offsets_outside_the_contract_stay_in_bounds(oracle_mod, fmt, bad):
    """Decreasing, negative or too large offsets: the call succeeds, nothing
    outside C is written (canaries on both sides), and every row follows the
    documented clamping (checked against the oracle on the clamped groups)."""
    import torch
    rng = np.random.default_rng(len(bad) + bad[1])
    T, N, K = 100, 128, 256
    G = len(bad) - 1
    A, SA = small_int_codes(rng, T, K, fmt)
    B, SB = small_int_codes(rng, G * N, K, fmt)
    pad = 4096
    buf = torch.full((pad + T * N + pad,), 12345.0, dtype=torch.float32, device="cuda")
    C = buf[pad:pad + T * N].view(T, N)
    C.fill_(float("nan"))
    got, desc = _run(fmt, bad, A, SA, B, SB, N, K, OUT_F32, C=C)
    host = buf.cpu().numpy()
    assert (host[:pad] == 12345.0).all() and (host[-pad:] == 12345.0).all(), "wrote outside C"
    groups = _sanitised(bad, T)
    for e, (s, end) in enumerate(groups):
        if end > s:
            ref, _ = oracle_mod.gemm(fmt, A[s:end], SA[s:end], B[e * N:(e + 1) * N], SB[e * N:(e + 1) * N], K)
            assert (got[s:end] == ref).all(), (e, s, end, desc)
    covered = np.zeros(T, bool)
    for s, end in groups:
        covered[s:end] = True
    assert np.isnan(got[~covered]).all()


# ---- the grouped workloads at full size, sampled rows -----------------------------

def _moe_all():
    out = []
    for name in MOE_WORKLOADS:
        for fmt_name, nki, G, T, N, K, sizes in moe_cases(name):
            out.append((name, fmt_name, nki, G, T, N, K, sizes))
    return out


_MOE = _moe_all()


@pytest.mark.parametrize("case", _MOE, ids=[f"{c[0]}-{c[1]}-nk{c[2]}" for c in _MOE])
def test_moe_workloads_full_size_sampled(oracle_mod, case):
    name, fmt_name, nki, G, T, N, K, sizes = case
    fmt = FMT_MXFP8 if fmt_name == "mxfp8" else FMT_MXFP4
    rng = np.random.default_rng([len(name), nki, 7])
    A, SA = quantize_mx(normal_f32(rng, T, K), fmt)
    B, SB = quantize_mx(normal_f32(rng, G * N, K), fmt)
    offsets = list(group_offsets(sizes))
    C, desc = _run(fmt, offsets, A, SA, B, SB, N, K, OUT_BF16)
    # sample: the first and last row of every non-empty group and one seeded row
    # inside every 128-row token block of each group (all columns), so that every
    # token tile of every group -- 64- or 128-row tiles starting at the group's
    # first row -- has elements compared with the oracle
    rows = set()
    for e in range(G):
        if sizes[e]:
            lo, hi = offsets[e], offsets[e + 1]
            rows.update((lo, hi - 1))
            for t0 in range(lo, hi, 64):
                rows.add(int(t0 + rng.integers(0, min(64, hi - t0))))
    rows = np.array(sorted(rows), dtype=np.int64)
    ref, S = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K, rows=rows)
    assert_within(C[rows], ref, S, OUT_BF16, f"{name} {fmt_name} {desc}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("sizes,N,K,lead,trail", [([700, 1200, 0, 900], 512, 512, 0, 0),
                                                   ([513, 1, 256, 1030], 384, 1024, 5, 3),
                                                   ([2048], 256, 256, 0, 0)])
def test_grouped_pair_tiles_exact(oracle_mod, fmt, sizes, N, K, lead, trail):
    """Prefill-sized groups (>= 512 tokens on average, or forced) run 256 x 256
    CTA-pair tiles: token tiles of 256 rows inside each group (the odd CTA's rows
    may run past the group's end into the next group, and the last weight tile
    of a group of 384 rows into the next group's weights), exact against the
    oracle; rows outside every group untouched."""
    offsets = list(lead + group_offsets(sizes))
    T = offsets[-1] + trail
    G = len(sizes)
    rng = np.random.default_rng([sum(sizes), N, K, fmt])
    A, SA = small_int_codes(rng, T, K, fmt)
    B, SB = small_int_codes(rng, G * N, K, fmt)
    ref, _ = oracle_mod.grouped_gemm(fmt, offsets, A, SA, B, SB, N, K)
    inside = _in_groups(offsets, T)
    for out, flags in ((OUT_F32, PAIR), (OUT_BF16, 0)):
        C, desc = _run(fmt, offsets, A, SA, B, SB, N, K, out, flags)
        if flags == PAIR or sum(sizes) // G >= 512:
            assert "mode=pair" in desc, desc
        expect = ref if out == OUT_F32 else _bf16(ref)
        assert (C[inside] == expect[inside]).all(), desc
        assert np.isnan(C[~inside]).all(), f"rows outside every group were written: {desc}"


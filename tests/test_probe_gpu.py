"""The tensor-pipe rate probe (mxgemm_probe_tensor_rate) on the GPU: every unit
finishes without a wait expiring, and the cycles one MMA takes match the tile
arithmetic -- an M = 128 (or 256 on a CTA pair) x N MMA of K = 32 bytes per row
occupies the pipe N / 2 cycles for every kind measured on this part, so that the
FP4 kind does twice the FP8 work per cycle."""
import pytest

from gpu_util import lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3)
    lib()


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "bf16"])
@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("n", [128, 256])
def test_mma_cycles_match_the_tile(fmt, cg, n):
    b = lib()
    code = {"mxfp8": b.MXGEMM_FMT_MXFP8_E4M3, "mxfp4": b.MXGEMM_FMT_MXFP4_E2M1, "bf16": b.MXGEMM_FMT_BF16}[fmt]
    r = b.mxgemm_probe_tensor_rate(code, cg, n, 0, 2048)
    b.check_device_status()
    assert r["units"] >= (100 if cg == 1 else 50)
    assert 0.5 < r["sm_ghz"] < 2.5
    # the pipe's own rate, with a little slack for the issue loop and the clock read
    assert n / 2 * 0.97 <= r["cycles_per_mma"] <= n / 2 * 1.15, r


def test_scale_copies_do_not_slow_the_wide_pair_tile():
    """The scale copies a GEMM k-stage issues ride along on the N = 256 pair tile."""
    b = lib()
    base = b.mxgemm_probe_tensor_rate(b.MXGEMM_FMT_MXFP8_E4M3, 2, 256, 0, 2048)
    with_cp = b.mxgemm_probe_tensor_rate(b.MXGEMM_FMT_MXFP8_E4M3, 2, 256, 1, 2048)
    assert with_cp["cycles_per_mma"] <= base["cycles_per_mma"] * 1.10, (base, with_cp)

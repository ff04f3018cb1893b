"""mxgemm_run_noalloc: the entry point for callers that cannot allocate device memory.

Such callers (a serving loop whose memory was planned at start-up, a plain C
program without its own allocator) hand over only inputs and outputs; the
library then uses its one static device scratch array instead of a workspace.
These tests call it through the C ABI twice in a row and check each result
against mxgemm_run's, within the parity tolerance the other tests use.
This file is collected last on purpose.
"""
import numpy as np
import pytest

from gpu_util import OUT_BF16, OUT_F32, lib, to_dev, tolerance
from mx_block_scaled_gb300.inputs import FMT_MXFP4, FMT_MXFP8, make_operand

pytestmark = pytest.mark.gpu

# (workload, fmt, M, N, K, A shape index, B (N,K) index, out): a decode shape whose
# plan splits K (the scratch then holds the tile-layout scales and the FP32
# partial sums of the splits) and a whole-tile prefill shape (scales only).
CASES = [
    ("llama33_70b", FMT_MXFP8, 8, 8192, 8192, 1, 1, OUT_BF16),
    ("llama31_8b", FMT_MXFP4, 8192, 4096, 4096, 9, 1, OUT_F32),
]


def _run_both(b, oracle_mod, case):
    import torch
    name, fmt, M, N, K, si, nki, out = case
    A, SA = make_operand(name, "A", si, M, K, fmt)
    B, SB = make_operand(name, "B", nki, N, K, fmt)
    plan = b.Plan(M, N, K, fmt, out)
    assert plan.ws_bytes <= b.MXGEMM_NOALLOC_SCRATCH_BYTES, plan.describe()
    desc = plan.describe()
    split_k = int(desc.split("split_k=")[1].split()[0])
    sk_units = int(desc.split("streamk=")[1].split()[0].split("/")[1])
    if M <= 64:  # the decode case must keep covering the partial-sum region of the scratch
        assert split_k > 1 or sk_units > 0, desc
    dA, dSA, dB, dSB = to_dev(A), to_dev(SA), to_dev(B), to_dev(SB)
    ref = plan.run(dA, dSA, dB, dSB)
    C = torch.full((M, N), float("nan"), dtype=plan.out_dtype(), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = b.mxgemm_run_noalloc(plan.handle, dA.data_ptr(), dSA.data_ptr(), dB.data_ptr(), dSB.data_ptr(),
                              C.data_ptr(), 0, stream)
    assert st == b.MXGEMM_OK, b.mxgemm_status_str(st)
    assert b.mxgemm_device_status(stream, True) == b.MXGEMM_OK
    got = C.double().cpu().numpy()
    want = ref.double().cpu().numpy()
    rows = np.arange(min(M, 16))
    _, S = oracle_mod.gemm(fmt, A, SA, B, SB, K, rows=rows)
    tol_rows = tolerance(want[rows], S, out)
    assert (np.abs(got[rows] - want[rows]) <= tol_rows).all()
    # beyond the sampled rows: the same kernels in the same order give the same bits
    assert np.array_equal(got, want)
    return plan


def test_noalloc_matches_mxgemm_run_twice_in_a_row(oracle_mod):
    import torch
    assert torch.cuda.is_available()
    b = lib()
    keep = []
    for case in CASES:          # two calls in a row, sharing the static scratch
        keep.append(_run_both(b, oracle_mod, case))
    keep.append(_run_both(b, oracle_mod, CASES[0]))  # and back to the first shape


def test_noalloc_rejects_plans_beyond_its_scratch():
    import torch
    b = lib()
    # M=16384, N=57344, K=8192 MXFP8 needs ~18.9 MB of tile-layout scales alone
    st, h = b.mxgemm_plan_create(16384, 57344, 8192, FMT_MXFP8, OUT_BF16, 0)
    assert st == b.MXGEMM_OK
    try:
        assert b.mxgemm_workspace_bytes(h) > b.MXGEMM_NOALLOC_SCRATCH_BYTES
        dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
        p = dummy.data_ptr()
        st = b.mxgemm_run_noalloc(h, p, p, p, p, p, 0, torch.cuda.current_stream().cuda_stream)
        assert st == b.MXGEMM_ERR_WORKSPACE
    finally:
        b.mxgemm_plan_destroy(h)


def test_noalloc_rejects_a_prepared_run():
    """mxgemm_run_noalloc's scratch is internal, so MXGEMM_RUN_PREPARED cannot apply."""
    import torch
    b = lib()
    plan = b.Plan(256, 256, 256, FMT_MXFP8, OUT_F32)
    p = plan.workspace.data_ptr()
    st = b.mxgemm_run_noalloc(plan.handle, p, p, p, p, p, b.MXGEMM_RUN_PREPARED,
                              torch.cuda.current_stream().cuda_stream)
    assert st == b.MXGEMM_ERR_ARG

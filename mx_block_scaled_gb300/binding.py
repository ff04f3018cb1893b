"""Thin ctypes binding of libmxgemm.so (include/mxgemm.h), same names as the C ABI.

Argument marshalling only: every step of the GEMM (scale relayout, the tcgen05
GEMM, the split-K reduce) runs in the library's CUDA kernels.  PyTorch is used
for device memory and streams.  If the library is missing this module raises
at import time; there is no fallback implementation.  With the environment
variable MXGEMM_DEBUG=1 the module loads the debug build (libmxgemm_debug.so:
bounds-checked kernels, NaN-filled C, synchronous status) instead.
"""
from __future__ import annotations

import ctypes
import os

from .build import DEBUG_LIB_PATH, LIB_PATH

MXGEMM_FMT_MXFP8_E4M3 = 1
MXGEMM_FMT_MXFP4_E2M1 = 2
MXGEMM_FMT_BF16 = 3
MXGEMM_OUT_F32 = 1
MXGEMM_OUT_BF16 = 2

MXGEMM_OK = 0
MXGEMM_ERR_ARG = -1
MXGEMM_ERR_SHAPE = -2
MXGEMM_ERR_ALIGN = -3
MXGEMM_ERR_WORKSPACE = -4
MXGEMM_ERR_ARCH = -5
MXGEMM_ERR_CUDA = -6
MXGEMM_ERR_DEVICE_TIMEOUT = -7
MXGEMM_ERR_UNSUPPORTED = -8
MXGEMM_ERR_DEVICE_BOUNDS = -9

MXGEMM_PLAN_FORCE_BN128 = 1 << 0
MXGEMM_PLAN_FORCE_BN256 = 1 << 1
MXGEMM_PLAN_FORCE_NOSWAP = 1 << 2
MXGEMM_PLAN_FORCE_SWAP = 1 << 3
MXGEMM_PLAN_FORCE_PAIR = 1 << 4
MXGEMM_PLAN_FORCE_SINGLE = 1 << 5
MXGEMM_PLAN_STREAMK = 1 << 7
MXGEMM_PLAN_SPLITK_SHIFT = 8
MXGEMM_PLAN_NO_STREAMK = 1 << 16
MXGEMM_PLAN_FORCE_BN192 = 1 << 17

MXGEMM_RUN_SA_PRELAYOUT = 1 << 0
MXGEMM_RUN_SB_PRELAYOUT = 1 << 1
MXGEMM_RUN_PREPARED = 1 << 2
MXGEMM_RUN_B_STATIC = 1 << 3

MXGEMM_IN_F32 = 1
MXGEMM_IN_BF16 = 2
MXGEMM_QUANT_SF_TILED = 1 << 0

# (name, restype, argtypes) for every entry point declared in include/mxgemm.h
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
SIGNATURES = [
    ("mxgemm_plan_create", ctypes.c_int,
     [ctypes.POINTER(ctypes.c_void_p), _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_uint32]),
    ("mxgemm_plan_destroy", ctypes.c_int, [_P]),
    ("mxgemm_workspace_bytes", ctypes.c_size_t, [_P]),
    ("mxgemm_plan_describe", ctypes.c_int, [_P, ctypes.c_char_p, ctypes.c_size_t]),
    ("mxgemm_sf_bytes", ctypes.c_size_t, [_I64, _I64]),
    ("mxgemm_relayout_scales", ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    ("mxgemm_quantize", ctypes.c_int,
     [ctypes.c_int, ctypes.c_int, _P, _I64, _I64, _P, _P, ctypes.c_uint32, _P]),
    ("mxgemm_run", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    ("mxgemm_prepare", ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    ("mxgemm_run_noalloc", ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_uint32, _P]),
    ("mxgemm_device_status", ctypes.c_int, [_P, ctypes.c_int]),
    ("mxgemm_selftest_stall", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    ("mxgemm_selftest_bounds", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    ("mxgemm_debug_build", ctypes.c_int, []),
    ("mxgemm_grouped_plan_create", ctypes.c_int,
     [ctypes.POINTER(ctypes.c_void_p), _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_uint32]),
    ("mxgemm_grouped_plan_destroy", ctypes.c_int, [_P]),
    ("mxgemm_grouped_workspace_bytes", ctypes.c_size_t, [_P]),
    ("mxgemm_grouped_plan_describe", ctypes.c_int, [_P, ctypes.c_char_p, ctypes.c_size_t]),
    ("mxgemm_grouped_run", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    ("mxgemm_placement_scan", ctypes.c_int, [ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _P]),
    ("mxgemm_probe_tensor_rate", ctypes.c_int,
     [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double), _P]),
    ("mxgemm_status_str", ctypes.c_char_p, [ctypes.c_int]),
    ("mxgemm_version", ctypes.c_int, []),
]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -m mx_block_scaled_gb300.build, or "
            "__graft_entry__.build()); there is no fallback implementation")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load_library(DEBUG_LIB_PATH if os.environ.get("MXGEMM_DEBUG", "0") == "1" else LIB_PATH)


class MxGemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {mxgemm_status_str(status)} (status {status})")
        self.status = status


def _check(status: int, what: str) -> int:
    if status != MXGEMM_OK:
        raise MxGemmError(status, what)
    return status


# ---- the C ABI, one Python function per entry point ---------------------------

def mxgemm_plan_create(M: int, N: int, K: int, fmt: int, out: int, flags: int = 0):
    """Return (status, plan_handle)."""
    h = ctypes.c_void_p()
    st = _lib.mxgemm_plan_create(ctypes.byref(h), M, N, K, fmt, out, flags)
    return st, h


def mxgemm_plan_destroy(plan) -> int:
    return _lib.mxgemm_plan_destroy(plan)


def mxgemm_workspace_bytes(plan) -> int:
    return _lib.mxgemm_workspace_bytes(plan)


def mxgemm_plan_describe(plan) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(_lib.mxgemm_plan_describe(plan, buf, len(buf)), "mxgemm_plan_describe")
    return buf.value.decode()


def mxgemm_sf_bytes(rows: int, K: int) -> int:
    return _lib.mxgemm_sf_bytes(rows, K)


def mxgemm_relayout_scales(src_ptr: int, rows: int, K: int, dst_ptr: int, stream: int) -> int:
    return _lib.mxgemm_relayout_scales(src_ptr, rows, K, dst_ptr, stream)


def mxgemm_quantize(fmt: int, in_dtype: int, x_ptr: int, rows: int, K: int, codes_ptr: int,
                    scales_ptr: int, flags: int, stream: int) -> int:
    return _lib.mxgemm_quantize(fmt, in_dtype, x_ptr, rows, K, codes_ptr, scales_ptr, flags, stream)


def mxgemm_run(plan, A_ptr: int, SA_ptr: int, B_ptr: int, SB_ptr: int, C_ptr: int,
               ws_ptr: int, ws_bytes: int, run_flags: int, stream: int) -> int:
    return _lib.mxgemm_run(plan, A_ptr, SA_ptr, B_ptr, SB_ptr, C_ptr, ws_ptr, ws_bytes, run_flags, stream)


def mxgemm_prepare(plan, SA_ptr: int, SB_ptr: int, ws_ptr: int, ws_bytes: int, run_flags: int, stream: int) -> int:
    return _lib.mxgemm_prepare(plan, SA_ptr, SB_ptr, ws_ptr, ws_bytes, run_flags, stream)


def mxgemm_run_noalloc(plan, A_ptr: int, SA_ptr: int, B_ptr: int, SB_ptr: int, C_ptr: int,
                       run_flags: int, stream: int) -> int:
    return _lib.mxgemm_run_noalloc(plan, A_ptr, SA_ptr, B_ptr, SB_ptr, C_ptr, run_flags, stream)


MXGEMM_NOALLOC_SCRATCH_BYTES = 16 << 20


def mxgemm_grouped_plan_create(groups: int, rows: int, N: int, K: int, fmt: int, out: int, flags: int = 0):
    """Return (status, grouped_plan_handle)."""
    h = ctypes.c_void_p()
    st = _lib.mxgemm_grouped_plan_create(ctypes.byref(h), groups, rows, N, K, fmt, out, flags)
    return st, h


def mxgemm_grouped_plan_destroy(plan) -> int:
    return _lib.mxgemm_grouped_plan_destroy(plan)


def mxgemm_grouped_workspace_bytes(plan) -> int:
    return _lib.mxgemm_grouped_workspace_bytes(plan)


def mxgemm_grouped_plan_describe(plan) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(_lib.mxgemm_grouped_plan_describe(plan, buf, len(buf)), "mxgemm_grouped_plan_describe")
    return buf.value.decode()


def mxgemm_grouped_run(plan, offsets_ptr: int, A_ptr: int, SA_ptr: int, B_ptr: int, SB_ptr: int, C_ptr: int,
                       ws_ptr: int, ws_bytes: int, run_flags: int, stream: int) -> int:
    return _lib.mxgemm_grouped_run(plan, offsets_ptr, A_ptr, SA_ptr, B_ptr, SB_ptr, C_ptr, ws_ptr, ws_bytes,
                                   run_flags, stream)


def mxgemm_device_status(stream: int, reset: bool = True) -> int:
    return _lib.mxgemm_device_status(stream, 1 if reset else 0)


def mxgemm_selftest_stall(plan, A_ptr, SA_ptr, B_ptr, SB_ptr, C_ptr, ws_ptr, ws_bytes, stream) -> int:
    return _lib.mxgemm_selftest_stall(plan, A_ptr, SA_ptr, B_ptr, SB_ptr, C_ptr, ws_ptr, ws_bytes, stream)


def mxgemm_selftest_bounds(plan, A_ptr, SA_ptr, B_ptr, SB_ptr, C_ptr, ws_ptr, ws_bytes, run_flags, stream) -> int:
    return _lib.mxgemm_selftest_bounds(plan, A_ptr, SA_ptr, B_ptr, SB_ptr, C_ptr, ws_ptr, ws_bytes, run_flags, stream)


def mxgemm_debug_build() -> int:
    return _lib.mxgemm_debug_build()


def mxgemm_status_str(status: int) -> str:
    return _lib.mxgemm_status_str(status).decode()


def mxgemm_version() -> int:
    return _lib.mxgemm_version()


# ---- torch conveniences (marshalling only) ------------------------------------

def _stream_handle(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Plan:
    """Owns a plan handle and its device workspace (a torch uint8 tensor)."""

    def __init__(self, M: int, N: int, K: int, fmt: int, out: int, flags: int = 0, device=None):
        import torch
        self.M, self.N, self.K, self.fmt, self.out = M, N, K, fmt, out
        st, h = mxgemm_plan_create(M, N, K, fmt, out, flags)
        _check(st, "mxgemm_plan_create")
        self.handle = h
        self.ws_bytes = mxgemm_workspace_bytes(h)
        self.workspace = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8,
                                     device=device or torch.device("cuda"))

    def describe(self) -> str:
        return mxgemm_plan_describe(self.handle)

    def out_dtype(self):
        import torch
        return torch.bfloat16 if self.out == MXGEMM_OUT_BF16 else torch.float32

    def run(self, A, SA, B, SB, C=None, run_flags: int = 0, stream=None):
        """C = A * B^T on `stream` (default: torch's current stream).  Tensors are CUDA uint8."""
        import torch
        if C is None:
            C = torch.empty((self.M, self.N), dtype=self.out_dtype(), device=A.device)
        sa = SA.data_ptr() if SA is not None else 0
        sb = SB.data_ptr() if SB is not None else 0
        st = mxgemm_run(self.handle, A.data_ptr(), sa, B.data_ptr(), sb, C.data_ptr(),
                        self.workspace.data_ptr(), self.ws_bytes, run_flags, _stream_handle(stream))
        _check(st, "mxgemm_run")
        return C

    def prepare(self, SA, SB, run_flags: int = 0, stream=None):
        """Step (1) alone: lay out the scales not flagged pre-laid-out into this
        plan's workspace and reset its stream-K counters; follow with
        run(..., run_flags=MXGEMM_RUN_PREPARED | <same flags>)."""
        sa = SA.data_ptr() if SA is not None else 0
        sb = SB.data_ptr() if SB is not None else 0
        st = mxgemm_prepare(self.handle, sa, sb, self.workspace.data_ptr(), self.ws_bytes, run_flags,
                            _stream_handle(stream))
        _check(st, "mxgemm_prepare")

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            mxgemm_plan_destroy(h)
            self.handle = None


class GroupedPlan:
    """Owns a grouped-GEMM plan handle and its device workspace (a torch uint8 tensor)."""

    def __init__(self, groups: int, rows: int, N: int, K: int, fmt: int, out: int, flags: int = 0, device=None):
        import torch
        self.groups, self.rows, self.N, self.K, self.fmt, self.out = groups, rows, N, K, fmt, out
        st, h = mxgemm_grouped_plan_create(groups, rows, N, K, fmt, out, flags)
        _check(st, "mxgemm_grouped_plan_create")
        self.handle = h
        self.ws_bytes = mxgemm_grouped_workspace_bytes(h)
        self.workspace = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8,
                                     device=device or torch.device("cuda"))

    def describe(self) -> str:
        return mxgemm_grouped_plan_describe(self.handle)

    def run(self, offsets, A, SA, B, SB, C=None, run_flags: int = 0, stream=None):
        """C = grouped A * B_e^T.  ``offsets``: CUDA int64 tensor of groups + 1 row offsets."""
        import torch
        if C is None:
            C = torch.empty((self.rows, self.N), dtype=torch.bfloat16 if self.out == MXGEMM_OUT_BF16
                            else torch.float32, device=A.device)
        if offsets.dtype != torch.int64 or not offsets.is_cuda or offsets.numel() != self.groups + 1:
            raise ValueError("offsets must be a CUDA int64 tensor of groups + 1 entries")
        st = mxgemm_grouped_run(self.handle, offsets.data_ptr(), A.data_ptr(), SA.data_ptr(), B.data_ptr(),
                                SB.data_ptr(), C.data_ptr(), self.workspace.data_ptr(), self.ws_bytes, run_flags,
                                _stream_handle(stream))
        _check(st, "mxgemm_grouped_run")
        return C

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            mxgemm_grouped_plan_destroy(h)
            self.handle = None


def relayout_scales(S, rows: int, K: int, out=None, stream=None):
    """Row-major [rows, K/32] scales (CUDA uint8) -> tile layout (new CUDA uint8 tensor)."""
    import torch
    if out is None:
        out = torch.empty(mxgemm_sf_bytes(rows, K), dtype=torch.uint8, device=S.device)
    _check(mxgemm_relayout_scales(S.data_ptr(), rows, K, out.data_ptr(), _stream_handle(stream)),
           "mxgemm_relayout_scales")
    return out


def quantize(x, fmt: int, tiled: bool = False, codes=None, scales=None, stream=None):
    """MX-quantise a CUDA tensor x [rows, K] (float32 or bfloat16, contiguous).

    Returns ``(codes, scales)`` as CUDA uint8 tensors: codes [rows, K] (MXFP8)
    or [rows, K/2] (MXFP4); scales [rows, K/32] row-major, or, with
    ``tiled=True``, mxgemm_sf_bytes(rows, K) bytes in the tile layout.
    """
    import torch
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    in_dtype = {torch.float32: MXGEMM_IN_F32, torch.bfloat16: MXGEMM_IN_BF16}.get(x.dtype)
    if in_dtype is None:
        raise ValueError(f"unsupported input dtype {x.dtype}")
    rows, K = x.shape
    if codes is None:
        codes = torch.empty((rows, K if fmt == MXGEMM_FMT_MXFP8_E4M3 else K // 2), dtype=torch.uint8,
                            device=x.device)
    if scales is None:
        n = mxgemm_sf_bytes(rows, K) if tiled else rows * (K // 32)
        scales = torch.empty(max(n, 1), dtype=torch.uint8, device=x.device)
        if not tiled:
            scales = scales[: rows * (K // 32)].view(rows, K // 32) if n else scales
    _check(mxgemm_quantize(fmt, in_dtype, x.data_ptr(), rows, K, codes.data_ptr(), scales.data_ptr(),
                           MXGEMM_QUANT_SF_TILED if tiled else 0, _stream_handle(stream)), "mxgemm_quantize")
    return codes, scales


def mxgemm_placement_scan(k: int, sa_ptr: int, sb_ptr: int, npairs: int, counts_ptr: int, first_ptr: int,
                          stream: int) -> int:
    return _lib.mxgemm_placement_scan(k, sa_ptr, sb_ptr, npairs, counts_ptr, first_ptr, stream)


def placement_scan(k: int, sa, sb, stream=None):
    """Scale-placement checker on the GPU: ``sa``, ``sb`` CUDA int32 tensors of scale
    codes; returns (counts [npairs, 3] int64, first_diff [npairs] int64) CUDA tensors."""
    import torch
    n = sa.numel()
    counts = torch.empty((n, 3), dtype=torch.int64, device=sa.device)
    first = torch.empty(n, dtype=torch.int64, device=sa.device)
    _check(mxgemm_placement_scan(k, sa.data_ptr(), sb.data_ptr(), n, counts.data_ptr(), first.data_ptr(),
                                 _stream_handle(stream)), "mxgemm_placement_scan")
    return counts, first


def mxgemm_probe_tensor_rate(fmt: int, cta_group: int, n: int, scale_copies: int, stages: int,
                             stream=None) -> dict:
    """Tensor-pipe rate probe (tcgen05.mma from shared-memory operands, no loads) on
    the current device.  Synchronous.  Returns cycles per MMA, the SM clock in GHz,
    the whole-GPU dense PFLOP/s and the number of SMs or CTA pairs that ran."""
    out = (ctypes.c_double * 4)()
    _check(_lib.mxgemm_probe_tensor_rate(fmt, cta_group, n, scale_copies, stages, out, _stream_handle(stream)),
           "mxgemm_probe_tensor_rate")
    return {"cycles_per_mma": out[0], "sm_ghz": out[1], "pflops": out[2], "units": int(out[3])}


def check_device_status(stream=None) -> None:
    """Raise if a kernel recorded a device timeout since the last check."""
    _check(mxgemm_device_status(_stream_handle(stream), True), "device status")

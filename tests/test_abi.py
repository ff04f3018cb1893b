"""The C-ABI library without a GPU: it loads, exports every declared entry
point, and validates arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxgemm.h")


@pytest.fixture(scope="module")
def lib():
    from mx_block_scaled_gb300 import build
    build.build()
    from mx_block_scaled_gb300 import binding
    return binding


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MXGEMM_API\s+[\w\s\*]*?\b(mxgemm_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_entry_points()
    for required in ("mxgemm_plan_create", "mxgemm_run", "mxgemm_relayout_scales",
                     "mxgemm_plan_destroy", "mxgemm_workspace_bytes", "mxgemm_sf_bytes",
                     "mxgemm_device_status", "mxgemm_status_str"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_entry_points():
        assert hasattr(so, name), f"{name} declared in mxgemm.h but not exported"
    bound = {n for n, _, _ in lib.SIGNATURES}
    assert set(declared_entry_points()) == bound


def test_debug_library_exports_every_declared_symbol(lib):
    """The debug build (MXGEMM_DEBUG) has the same entry points, and says which
    build it is; the release build's bounds self-test is refused on the host."""
    dbg = lib.load_library(lib.DEBUG_LIB_PATH)
    for name in declared_entry_points():
        assert hasattr(dbg, name), f"{name} declared in mxgemm.h but not exported by the debug build"
    assert dbg.mxgemm_debug_build() == 1
    assert lib._lib.mxgemm_debug_build() == 0
    assert lib._lib.mxgemm_selftest_bounds(None, None, None, None, None, None, None, 0, 0, None) == \
        lib.MXGEMM_ERR_UNSUPPORTED
    assert dbg.mxgemm_selftest_bounds(None, None, None, None, None, None, None, 0, 0, None) == lib.MXGEMM_ERR_ARG
    assert dbg.mxgemm_status_str(lib.MXGEMM_ERR_DEVICE_BOUNDS).decode().startswith("a debug-build kernel")


def test_sf_bytes(lib):
    assert lib.mxgemm_sf_bytes(1, 128) == 128 * 4
    assert lib.mxgemm_sf_bytes(129, 256) == 256 * 8
    assert lib.mxgemm_sf_bytes(57344, 8192) == 57344 * 256
    assert lib.mxgemm_sf_bytes(0, 128) == 0
    assert lib.mxgemm_sf_bytes(8, 96) == 0


def test_status_strings(lib):
    for st in range(-8, 1):
        assert lib.mxgemm_status_str(st) not in ("", "unknown status")
    assert lib.mxgemm_status_str(5) == "unknown status"
    assert lib.mxgemm_version() >= 100


@pytest.mark.parametrize("M,N,K,fmt,out,flags,expect", [
    (16, 16, 100, 1, 2, 0, -2),   # K % 128 != 0 (the FlyDSL page's K constraint)
    (16, 16, 0, 1, 2, 0, -2),
    (0, 16, 128, 1, 2, 0, -2),
    (16, -1, 128, 2, 1, 0, -2),
    (16, 16, 128, 4, 2, 0, -1),   # unknown format
    (16, 16, 128, 1, 9, 0, -1),   # unknown output type
    (16, 16, 128, 1, 2, 1 << 20, -1),  # unknown flag
    (16, 16, 128, 1, 2, (1 << 2) | (1 << 3), -1),  # contradictory flags
    (16, 16, 128, 1, 2, (1 << 7) | (1 << 16), -1),  # stream-K forced on and off
    (16, 16, 128, 1, 2, 1 << 6, -1),  # bit 6 is not a plan flag
    (16, 16, 128, 1, 2, (1 << 4) | (1 << 5), -1),  # pair and single tiles at once
    (16, 16, 128, 1, 2, (1 << 17) | (1 << 1), -1),  # 192- and 256-wide tiles at once
    (16, 16, 128, 1, 2, (1 << 17) | (1 << 7), -1),  # 192-wide tiles with stream-K
])
def test_plan_create_validates_before_touching_the_device(lib, M, N, K, fmt, out, flags, expect):
    st, h = lib.mxgemm_plan_create(M, N, K, fmt, out, flags)
    assert st == expect and not h.value


def test_null_arguments_are_rejected(lib):
    assert lib._lib.mxgemm_plan_create(None, 16, 16, 128, 1, 2, 0) == lib.MXGEMM_ERR_ARG
    assert lib.mxgemm_relayout_scales(0, 16, 128, 0, 0) == lib.MXGEMM_ERR_ARG
    assert lib.mxgemm_relayout_scales(16, 16, 100, 32, 0) == lib.MXGEMM_ERR_SHAPE
    assert lib.mxgemm_relayout_scales(17, 16, 128, 32, 0) == lib.MXGEMM_ERR_ALIGN
    assert lib.mxgemm_run(None, 16, 16, 16, 16, 16, 0, 0, 0, 0) == lib.MXGEMM_ERR_ARG
    assert lib.mxgemm_plan_destroy(None) == lib.MXGEMM_OK
    assert lib.mxgemm_workspace_bytes(None) == 0


def test_valid_plan_needs_an_sm103_device(lib):
    import torch
    st, h = lib.mxgemm_plan_create(256, 256, 256, 1, 2, 0)
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    assert st in (lib.MXGEMM_ERR_CUDA, lib.MXGEMM_ERR_ARCH) and not h.value


def test_oracle_builds_and_is_separate(oracle_mod):
    # The oracle is its own shared object, built from oracle/mxref.c only.
    from oracle import mxref
    assert os.path.exists(mxref.build())
    assert "mx_block_scaled_gb300" not in open(os.path.join(ROOT, "oracle", "mxref.c")).read()


@pytest.mark.parametrize("fmt,in_dtype,x,rows,K,codes,scales,flags,expect", [
    (1, 2, 0, 4, 128, 64, 64, 0, -1),          # NULL x
    (1, 2, 64, 4, 128, 0, 64, 0, -1),          # NULL codes
    (1, 2, 64, 4, 128, 64, 0, 0, -1),          # NULL scales
    (3, 2, 64, 4, 128, 64, 64, 0, -1),         # unknown format
    (1, 7, 64, 4, 128, 64, 64, 0, -1),         # unknown input type
    (1, 2, 64, 4, 128, 64, 64, 1 << 5, -1),    # unknown flag
    (1, 2, 64, 0, 128, 64, 64, 0, -2),         # rows < 1
    (1, 2, 64, 4, 48, 64, 64, 0, -2),          # K % 32 != 0
    (2, 1, 64, 4, 96, 64, 64, 1, -2),          # tile layout needs K % 128 == 0
    (1, 2, 48, 4, 128, 64, 64, 0, -3),         # x only 16-byte aligned (needs 32)
    (1, 2, 64, 4, 128, 72, 64, 0, -3),         # codes misaligned
    (1, 2, 64, 4, 128, 64, 65, 0, -3),         # scales misaligned
])
def test_quantize_validates_before_touching_the_device(lib, fmt, in_dtype, x, rows, K, codes, scales, flags,
                                                        expect):
    assert lib.mxgemm_quantize(fmt, in_dtype, x, rows, K, codes, scales, flags, 0) == expect


@pytest.mark.parametrize("groups,rows,N,K,fmt,out,flags,expect", [
    (0, 64, 128, 128, 1, 2, 0, -2),        # no groups
    (513, 64, 128, 128, 1, 2, 0, -2),      # more groups than a CTA's table holds
    (4, 0, 128, 128, 1, 2, 0, -2),         # no rows
    (4, 64, 100, 128, 1, 2, 0, -2),        # N not a multiple of 128
    (4, 64, 128, 96, 1, 2, 0, -2),         # K not a multiple of 128
    (4, 64, 128, 128, 3, 2, 0, -1),        # unknown format
    (4, 64, 128, 128, 1, 9, 0, -1),        # unknown output type
    (4, 64, 128, 128, 1, 2, (1 << 4) | (1 << 5), -1),  # pair and single tiles at once
    (4, 64, 128, 128, 1, 2, 1 << 7, -1),   # stream-K is not offered for grouped GEMMs
    (4, 64, 128, 128, 1, 2, (1 << 2) | (1 << 3), -1),
])
def test_grouped_plan_validates_before_touching_the_device(lib, groups, rows, N, K, fmt, out, flags, expect):
    st, h = lib.mxgemm_grouped_plan_create(groups, rows, N, K, fmt, out, flags)
    assert st == expect and not h.value


def test_grouped_null_arguments_are_rejected(lib):
    assert lib._lib.mxgemm_grouped_plan_create(None, 4, 64, 128, 128, 1, 2, 0) == lib.MXGEMM_ERR_ARG
    assert lib.mxgemm_grouped_run(None, 8, 16, 16, 16, 16, 16, 16, 0, 0, 0) == lib.MXGEMM_ERR_ARG
    assert lib.mxgemm_grouped_plan_destroy(None) == lib.MXGEMM_OK
    assert lib.mxgemm_grouped_workspace_bytes(None) == 0


@pytest.mark.parametrize("M,N,K,flags,expect", [
    (16, 16, 96, 0, -2),        # BF16 needs K % 64 == 0
    (16, 16, 0, 0, -2),
    (16, 16, 64, 1 << 6, -1),   # bit 6 is not a plan flag
])
def test_bf16_plan_validation(lib, M, N, K, flags, expect):
    st, h = lib.mxgemm_plan_create(M, N, K, 3, 2, flags)
    assert st == expect and not h.value


@pytest.mark.parametrize("k,npairs,sa,sb,counts,first,expect", [
    (2, 4, 0, 16, 32, 64, -1),     # NULL sa
    (0, 4, 16, 16, 32, 64, -2),    # k < 1
    (5, 4, 16, 16, 32, 64, -2),    # k > 4
    (2, 0, 16, 16, 32, 64, -2),    # no pairs
    (2, 4, 18, 16, 32, 64, -3),    # sa not 4-byte aligned
    (2, 4, 16, 16, 36, 64, -3),    # counts not 8-byte aligned
])
def test_placement_scan_validates_before_touching_the_device(lib, k, npairs, sa, sb, counts, first, expect):
    assert lib.mxgemm_placement_scan(k, sa, sb, npairs, counts, first, 0) == expect


def test_prepare_rejects_a_null_plan_on_the_host(lib):
    """mxgemm_prepare checks its arguments before any CUDA call."""
    assert lib.mxgemm_prepare(None, 0, 0, 0, 0, 0, None) == lib.MXGEMM_ERR_ARG
    assert lib.mxgemm_prepare(None, 0, 0, 0, 0, lib.MXGEMM_RUN_PREPARED, None) == lib.MXGEMM_ERR_ARG


def test_binding_constants_match_the_header(lib):
    """Every MXGEMM_* #define and enum value in mxgemm.h that the binding exposes
    has the same value there (flags, status codes, formats)."""
    text = open(HEADER).read()
    values = {}
    for name, expr in re.findall(r"#define\s+(MXGEMM_[A-Z0-9_]+)\s+([^\s/]+(?:\s*<<\s*\d+\))?)", text):
        expr = expr.strip()
        m = re.fullmatch(r"\(?(\d+)u?\s*<<\s*(\d+)\)?", expr)
        if m:
            values[name] = int(m.group(1)) << int(m.group(2))
        elif re.fullmatch(r"-?\d+", expr):
            values[name] = int(expr)
    for name, val in re.findall(r"(MXGEMM_(?:FMT|OUT)_[A-Z0-9_]+)\s*=\s*(\d+)", text):
        values[name] = int(val)
    checked = 0
    for name, val in values.items():
        if hasattr(lib, name):
            assert getattr(lib, name) == val, name
            checked += 1
    assert checked >= 15


@pytest.mark.parametrize("fmt,cg,n,cp,stages", [
    (0, 1, 256, 0, 1024),     # unknown format
    (1, 3, 256, 0, 1024),     # cta_group not 1 or 2
    (1, 1, 192, 0, 1024),     # N not 128 or 256
    (1, 1, 256, 2, 1024),     # scale_copies not 0 or 1
    (1, 1, 256, 0, 8),        # too few k-stages
    (2, 2, 128, 1, 1 << 23),  # too many k-stages
])
def test_tensor_probe_validates_before_touching_the_device(lib, fmt, cg, n, cp, stages):
    import ctypes
    out = (ctypes.c_double * 4)()
    assert lib._lib.mxgemm_probe_tensor_rate(fmt, cg, n, cp, stages, out, None) == lib.MXGEMM_ERR_ARG
    assert lib._lib.mxgemm_probe_tensor_rate(1, 1, 256, 0, 1024, None, None) == lib.MXGEMM_ERR_ARG

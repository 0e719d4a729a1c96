"""CPU checks of the C ABI: the library builds, loads without a GPU, exports
every symbol include/fp4lin.h declares, and rejects bad arguments before it
touches a device (no compute call runs here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fp4lin.h")


def _declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FP4LIN_API\s+[\w\s\*]+?\b(fp4_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from _util import lib

    return lib()


def test_header_declares_the_boundary():
    syms = _declared_symbols()
    for name in ("fp4_requant_nvfp4_to_mxfp4", "fp4_quant_act_mxfp4", "fp4_gemm_mxfp4",
                 "fp4_gemm_mxfp4_grouped", "fp4_quant_act_mxfp4_grouped"):
        assert name in syms


def test_library_exports_every_declared_symbol(L):
    lib = ctypes.CDLL(L.LIB_PATH)
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    assert set(_declared_symbols()) == set(L.SYMBOLS)


def test_sf_sizes(L):
    assert L.fp4_sf_bytes(256, 512, L.FP4_SF_ROWMAJOR) == 256 * 16
    assert L.fp4_sf_bytes(256, 512, L.FP4_SF_SWIZZLED) == 256 * 16
    assert L.fp4_sf_bytes(200, 192, L.FP4_SF_SWIZZLED) == 256 * 8          # rows -> 256, 6 blocks -> 8
    assert L.fp4_sf_bytes(1, 32, L.FP4_SF_SWIZZLED) == 128 * 4
    assert L.fp4_sf_bytes(0, 32, L.FP4_SF_SWIZZLED) == 0
    assert L.fp4_sf_bytes(5, 48, L.FP4_SF_SWIZZLED) == 0                   # K not a multiple of 32
    # grouped bound: sum over groups of ceil(rows/128) <= (total + E*127) / 128
    assert L.fp4_sf_bytes_grouped(32768, 64, 4096) == ((32768 + 64 * 127) // 128) * 128 * 128
    # NVFP4: one E4M3 byte per 16 elements
    assert L.fp4_sf_bytes_nvfp4(256, 512, L.FP4_SF_ROWMAJOR) == 256 * 32
    assert L.fp4_sf_bytes_nvfp4(200, 208, L.FP4_SF_SWIZZLED) == 256 * 16   # 13 blocks -> 16
    assert L.fp4_sf_bytes_nvfp4(1, 16, L.FP4_SF_SWIZZLED) == 128 * 4
    assert L.fp4_sf_bytes_nvfp4(5, 24, L.FP4_SF_SWIZZLED) == 0             # K not a multiple of 16


def test_status_strings(L):
    for s in range(7):
        assert L.status_string(s).startswith("FP4_")
    assert "UNKNOWN" in L.status_string(99)


def test_argument_checks_precede_device_use(L):
    raw = L.load()
    # shapes
    assert raw.fp4_gemm_mxfp4(16, 16, 16, 16, None, 16, 1, 8, 100, None) == 2      # K % 128
    assert raw.fp4_gemm_mxfp4(16, 16, 16, 16, None, 16, 1, 12, 128, None) == 2     # N % 8
    assert raw.fp4_quant_act_mxfp4(16, 16, 16, 4, 48, None, None) == 2             # K % 32
    assert raw.fp4_requant_nvfp4_to_mxfp4(16, 16, 1.0, 16, 16, 0, 32, None) == 2   # N = 0
    assert raw.fp4_requant_nvfp4_to_mxfp4_grouped(32, 32, 32, 32, 32, 2, 4, 96, None, None) == 2   # K % 128
    assert raw.fp4_requant_nvfp4_to_mxfp4_grouped(32, 32, 32, 32, 32, 0, 4, 128, None, None) == 2  # E = 0
    assert raw.fp4_requant_nvfp4_to_mxfp4_grouped(32, 32, 32, 32, 32, 2, 4, 1 << 29, None, None) == 2  # K >= 2^29
    assert raw.fp4_gemm_mxfp4_grouped(16, 16, 16, 16, None, 16, 16, 1025, 4, 8, 128, None) == 2    # E > 1024
    # null pointers
    assert raw.fp4_gemm_mxfp4(None, 16, 16, 16, None, 16, 1, 8, 128, None) == 1
    assert raw.fp4_requant_nvfp4_to_mxfp4(None, 16, 1.0, 16, 16, 4, 32, None) == 1
    assert raw.fp4_requant_nvfp4_to_mxfp4_grouped(32, 32, None, 32, 32, 2, 4, 128, None, None) == 1  # no scales
    # alignment
    assert raw.fp4_gemm_mxfp4(17, 16, 16, 16, None, 16, 1, 8, 128, None) == 3
    assert raw.fp4_quant_act_mxfp4(24, 16, 16, 4, 32, None, None) == 3
    assert raw.fp4_gemm_mxfp4_ws(16, 16, 16, 16, None, 16, 1, 8, 128, 16, 1 << 20, None) == 3   # workspace 256 B
    assert raw.fp4_requant_nvfp4_to_mxfp4_grouped(16, 32, 32, 32, 32, 2, 4, 128, None, None) == 3  # codes 32 B
    # bad option values
    from nvfp4_mxfp4_w4a4_gb300.fp4lin import fp4_quant_opts

    bad = fp4_quant_opts(1, 0)
    assert raw.fp4_quant_act_mxfp4(16, 16, 16, 4, 32, ctypes.byref(bad), None) == 1
    bad_flag = fp4_quant_opts(0, 0, 2)                                  # unknown flag bit
    assert raw.fp4_requant_nvfp4_to_mxfp4_ex(16, 16, 1.0, 16, 16, 4, 32, ctypes.byref(bad_flag), None) == 1
    assert raw.fp4_quant_act_mxfp4(16, 16, 16, 4, 32, ctypes.byref(bad_flag), None) == 1
    # NVFP4 side path
    assert raw.fp4_gemm_nvfp4(16, 16, 16, 16, 1.0, None, 16, 1, 8, 192, None, 0, None) == 2     # K % 128
    assert raw.fp4_gemm_nvfp4(16, None, 16, 16, 1.0, None, 16, 1, 8, 128, None, 0, None) == 1    # no scales
    assert raw.fp4_gemm_nvfp4(16, 16, 16, 24, 1.0, None, 16, 1, 8, 128, None, 0, None) == 3      # sb 16 B
    assert raw.fp4_gemm_nvfp4(16, 16, 16, 16, 1.0, None, 16, 1, 8, 128, 16, 1 << 20, None) == 3  # workspace
    assert raw.fp4_quant_nvfp4_ex(16, 1.0, 16, 16, 4, 24, 0, None) == 2                          # K % 16
    assert raw.fp4_quant_nvfp4_ex(16, 1.0, 16, 16, 4, 32, 5, None) == 1                          # layout
    assert raw.fp4_sf_swizzle(16, 16, 4, 0, None) == 2                                           # kblocks
    assert raw.fp4_sf_swizzle(None, 16, 4, 4, None) == 1
    assert raw.fp4_sf_swizzle(16, 18, 4, 4, None) == 3                                           # out 4 B
    assert raw.fp4_sf_swizzle(None, None, 0, 4, None) == 0
    assert raw.fp4_gemm_mxfp4_ex(16, 16, 16, 16, None, 16, 1, 8, 128, None, 0, 2, None) == 1     # unknown flag
    assert raw.fp4_gemm_mxfp4_ex(16, 16, 16, 16, None, 16, 1, 8, 100, None, 0, 1, None) == 2     # K % 128
    # smooth pre-scale
    assert raw.fp4_smooth_prepare(16, 16, 0, 16, None) == 2                                     # K = 0
    assert raw.fp4_smooth_prepare(None, 16, 8, 16, None) == 1
    assert raw.fp4_smooth_prepare(16, 16, 8, 18, None) == 3                                     # counter 4 B
    assert raw.fp4_quant_act_mxfp4_smooth(16, None, 16, 16, 4, 32, None, None) == 1             # no scale
    assert raw.fp4_quant_act_mxfp8_smooth(16, None, 16, 16, 4, 32, 0, None) == 1
    assert raw.fp4_quant_act_mxfp4_smooth(16, 24, 16, 16, 4, 32, None, None) == 3               # scale 16 B
    # linear layer
    from nvfp4_mxfp4_w4a4_gb300.fp4lin import fp4_linear_opts

    o_bad = fp4_linear_opts(7, 0, None, 0)
    o_a8_uos = fp4_linear_opts(1, 2, None, 0)
    o_flag = fp4_linear_opts(0, 0, None, 4)
    o_ok = fp4_linear_opts(0, 0, None, 0)
    for o, want in ((o_bad, 1), (o_a8_uos, 1), (o_flag, 1)):
        assert raw.fp4_linear(256, 256, 256, None, 256, 4, 8, 128, 256, 1 << 20, ctypes.byref(o), None) == want
    assert raw.fp4_linear(256, 256, 256, None, 256, 4, 8, 192, 256, 1 << 20, ctypes.byref(o_ok), None) == 2  # K
    assert raw.fp4_linear(256, 256, 256, None, 256, 4, 8, 128, 256, 16, ctypes.byref(o_ok), None) == 1     # ws
    assert raw.fp4_linear(256, 256, 256, None, 256, 4, 8, 128, 320, 1 << 20, ctypes.byref(o_ok), None) == 3  # align
    assert raw.fp4_linear(None, None, None, None, None, 0, 8, 128, None, 0, None, None) == 0               # M = 0
    assert raw.fp4_linear_workspace_size(4, 8, 128, ctypes.byref(o_bad)) == 0
    assert raw.fp4_linear_grouped(256, 256, 0, 8, 256, 256, None, 256, 8, 128, 256, 1 << 20, None, None) == 2  # E
    assert raw.fp4_linear_grouped(256, 256, 2, 8, 256, 256, None, 256, 8, 128, 256, 16, None, None) == 1     # ws
    assert raw.fp4_linear_grouped_workspace_size(0, 2, 128) == 0
    # W4A8 fallback
    assert raw.fp4_gemm_w4a8(16, 16, 32, 16, None, 16, 1, 8, 192, None, 0, None) == 2           # K % 128
    assert raw.fp4_gemm_w4a8(16, 16, 48, 16, None, 16, 1, 8, 128, None, 0, None) == 3           # b 32 B
    assert raw.fp4_gemm_w4a8(16, 16, 32, 16, None, 16, 1, 8, 128, 16, 1 << 20, None) == 3       # workspace
    assert raw.fp4_quant_act_mxfp8(16, 16, 16, 4, 48, 0, None) == 2                             # K % 32
    assert raw.fp4_quant_act_mxfp8(16, 16, 16, 4, 32, 3, None) == 1                             # layout
    assert raw.fp4_quant_act_mxfp8(16, 24, 16, 4, 32, 0, None) == 3                             # codes 16 B
    # empty problems are no-ops that need no device
    assert raw.fp4_quant_act_mxfp4(None, None, None, 0, 32, None, None) == 0
    assert raw.fp4_gemm_mxfp4(None, None, None, None, None, None, 0, 8, 128, None) == 0


@pytest.mark.skipif(__import__("_util").gpu_available(), reason="CPU-only check")
def test_valid_call_without_gpu_reports_cuda_error(L):
    raw = L.load()
    st = raw.fp4_quant_act_mxfp4(16, 16, 16, 4, 32, None, None)
    assert st in (4, 5)   # no usable device: UNSUPPORTED or CUDA, never a silent success


def test_no_alloc_argument_checks_match_the_workspace_entry_point(L):
    """The entry point without allocations runs the same host checks as
    fp4_gemm_mxfp4_ws, before it touches a device."""
    raw = L.load()
    cases = [
        ((16, 16, 16, 16, None, 16, 1, 8, 100), 2),      # K % 128
        ((16, 16, 16, 16, None, 16, 1, 12, 128), 2),     # N % 8
        ((16, 16, 16, 16, None, 16, -1, 8, 128), 2),     # M < 0
        ((16, 16, 16, 16, None, 16, 1, 0, 128), 2),      # N = 0
        ((None, 16, 16, 16, None, 16, 1, 8, 128), 1),    # null a
        ((16, 16, 16, None, None, 16, 1, 8, 128), 1),    # null sb
        ((16, 16, 16, 16, None, None, 1, 8, 128), 1),    # null out
        ((17, 16, 16, 16, None, 16, 1, 8, 128), 3),      # a not 16-byte aligned
        ((16, 16, 16, 16, 24, 16, 1, 8, 128), 3),        # bias not 16-byte aligned
        ((None, None, None, None, None, None, 0, 8, 128), 0),   # M = 0: no-op
    ]
    for args, want in cases:
        assert raw.fp4_gemm_mxfp4_noalloc(*args, None) == want, args
        assert raw.fp4_gemm_mxfp4_ws(*args, None, 0, None) == want, args


def test_debug_wait_fault_hook_checks_its_arguments(L):
    raw = L.load()
    assert raw.fp4_debug_set_wait_fault(10, 0) == 1            # below 1 us
    assert raw.fp4_debug_set_wait_fault(2 * 10 ** 10, 0) == 1  # above 10 s
    assert raw.fp4_debug_set_wait_fault(0, 2) == 1
    assert raw.fp4_debug_set_wait_fault(2_000_000, 1) == 0
    assert raw.fp4_debug_set_wait_fault(0, 0) == 0             # back to the defaults


def test_dualscale_argument_checks(L):
    raw = L.load()
    assert raw.fp4_quant_dualscale(16, 16, 16, 16, 4, 1024 + 128, 0, None) == 2     # K % 512
    assert raw.fp4_quant_dualscale(16, 16, 16, 16, 0, 512, 0, None) == 2            # N = 0
    assert raw.fp4_quant_dualscale(16, 16, 16, 16, 4, 512, 7, None) == 1            # layout
    assert raw.fp4_quant_dualscale(None, 16, 16, 16, 4, 512, 0, None) == 1
    assert raw.fp4_quant_dualscale(24, 16, 16, 16, 4, 512, 0, None) == 3            # w 16 B
    assert raw.fp4_quant_dualscale(16, 16, 16, 18, 4, 512, 0, None) == 3            # coarse 4 B
    assert raw.fp4_gemm_mxfp4_dualscale(16, 16, 16, 16, 16, None, 16, 1, 8, 768, None, 0, None) == 2   # K % 512
    assert raw.fp4_gemm_mxfp4_dualscale(16, 16, 16, 16, None, None, 16, 1, 8, 512, None, 0, None) == 1  # coarse
    assert raw.fp4_gemm_mxfp4_dualscale(16, 16, 16, 16, 18, None, 16, 1, 8, 512, None, 0, None) == 3    # coarse 4 B
    assert raw.fp4_gemm_mxfp4_dualscale(16, 16, 16, 16, 16, None, 16, 1, 8, 512, 16, 1 << 20, None) == 3  # ws
    assert raw.fp4_gemm_mxfp4_dualscale(None, None, None, None, None, None, None, 0, 8, 512, None, 0, None) == 0

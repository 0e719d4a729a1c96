"""CPU oracle for the W4A4 MXFP4 linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and its Python binding) never touches it.

This module is a thin numpy/ctypes shim over ``oracle.c``: it builds the C
file with gcc on first use and marshals arrays.  All arithmetic lives in the
C file, which cites the pages it follows; the one piece of logic here is the
grouped GEMM's assignment of rows to experts (each row goes to the expert e
with off[e] <= row < off[e+1]), pinned on its own against a per-expert
matmul.  Work on row ranges can be spread
over host threads (ctypes drops the GIL during a call); the result does not
depend on the thread count because rows are independent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SCALE_OCP = 0
SCALE_UOS = 2

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, no fast math, no FMA contraction)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True, cwd=_HERE)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            for name, res, args in [
                ("orc_e2m1_value", ctypes.c_double, [ctypes.c_uint]),
                ("orc_e4m3_value", ctypes.c_double, [ctypes.c_uint]),
                ("orc_e8m0_value", ctypes.c_double, [ctypes.c_uint]),
                ("orc_bf16_value", ctypes.c_double, [ctypes.c_uint16]),
                ("orc_e2m1_encode", ctypes.c_uint, [ctypes.c_double]),
                ("orc_e4m3_encode", ctypes.c_uint, [ctypes.c_float]),
                ("orc_mx_shared_exp", ctypes.c_int, [ctypes.c_double, ctypes.c_int]),
                ("orc_mx_quantize_block", None, [_p, ctypes.c_int, _p, _p]),
                ("orc_nvfp4_dequant", None, [_p, _p, ctypes.c_float, _i64, _i64, _p]),
                ("orc_requant", None, [_p, _p, ctypes.c_float, _i64, _i64, _i64, ctypes.c_int, _p, _p]),
                ("orc_requant_bf16", None, [_p, _p, ctypes.c_float, _i64, _i64, _i64, ctypes.c_int, _p, _p]),
                ("orc_act_quant", None, [_p, _i64, _i64, _i64, ctypes.c_int, _p, _p]),
                ("orc_gemm", None, [_p, _p, _p, _p, _p, _i64, _p, _i64, _p, _i64, _p, _p]),
                ("orc_bf16_encode", ctypes.c_uint16, [ctypes.c_float]),
                ("orc_smooth_prepare", _i64, [_p, _i64, _p]),
                ("orc_smooth_apply", None, [_p, _p, _i64, _i64, _p]),
                ("orc_mx8_shared_exp", ctypes.c_int, [ctypes.c_double]),
                ("orc_act_quant_mxfp8", None, [_p, _i64, _i64, _i64, _p, _p]),
                ("orc_gemm_w4a8", None, [_p, _p, _p, _p, _p, _i64, _p, _i64, _p, _i64, _p, _p]),
                ("orc_gemm_nvfp4", None,
                 [_p, _p, _p, _p, ctypes.c_double, _p, _i64, _p, _i64, _p, _i64, _p, _p]),
                ("orc_dual_dequant", None, [_p, _p, _p, _i64, _i64, _p]),
                ("orc_dual_quantize", None, [_p, _i64, _i64, _i64, _p, _p, _p]),
                ("orc_gemm_dual", None, [_p, _p, _p, _p, _p, _p, _i64, _p, _i64, _p, _i64, _p, _p]),
                ("orc_nvfp4_global_scale", ctypes.c_float, [_p, _i64]),
                ("orc_nvfp4_quantize", None, [_p, ctypes.c_float, _i64, _i64, _i64, _p, _p]),
                ("orc_sf_swizzled_bytes", _i64, [_i64, _i64]),
                ("orc_sf_swizzled_offset", _i64, [_i64, _i64, _i64]),
                ("orc_sf_swizzle", None, [_p, _i64, _i64, _p]),
            ]:
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _row_chunks(rows: int, threads: int):
    threads = max(1, min(threads, rows))
    step = (rows + threads - 1) // threads
    return [(r, min(rows, r + step)) for r in range(0, rows, step)]


def _parallel(fn, rows: int, threads: int):
    chunks = _row_chunks(rows, threads)
    if len(chunks) == 1:
        fn(*chunks[0])
        return
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(lambda c: fn(*c), chunks))


# ---------------------------------------------------------------- codecs
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e4m3_value(byte: int) -> float:
    return lib().orc_e4m3_value(byte)


def e8m0_value(byte: int) -> float:
    return lib().orc_e8m0_value(byte)


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(bits)


def e2m1_encode(q: float) -> int:
    return lib().orc_e2m1_encode(q)


def e4m3_encode(t: float) -> int:
    return lib().orc_e4m3_encode(t)


def mx_shared_exp(amax: float, alg: int = SCALE_OCP) -> int:
    return lib().orc_mx_shared_exp(amax, alg)


def mx_quantize_block(v: np.ndarray, alg: int = SCALE_OCP):
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.shape == (32,)
    packed = np.zeros(16, np.uint8)
    sf = np.zeros(1, np.uint8)
    lib().orc_mx_quantize_block(_ptr(v), alg, _ptr(packed), _ptr(sf))
    return packed, int(sf[0])


# ---------------------------------------------------------- hot-path math
def nvfp4_dequant(w_packed: np.ndarray, w_scale: np.ndarray, g: float) -> np.ndarray:
    rows, half = w_packed.shape
    K = 2 * half
    out = np.empty((rows, K), np.float32)
    lib().orc_nvfp4_dequant(_ptr(w_packed), _ptr(w_scale), g, rows, K, _ptr(out))
    return out


def requant(w_packed, w_scale, g, alg=SCALE_OCP, threads=1, bf16=False):
    """NVFP4 -> MXFP4; returns (packed [N, K/2] u8, row-major E8M0 [N, K/32] u8).
    bf16: round each decoded value to bf16 before the block rule."""
    w_packed = np.ascontiguousarray(w_packed)
    w_scale = np.ascontiguousarray(w_scale)
    N, half = w_packed.shape
    K = 2 * half
    out_p = np.empty((N, K // 2), np.uint8)
    out_s = np.empty((N, K // 32), np.uint8)
    L = lib()
    fn = L.orc_requant_bf16 if bf16 else L.orc_requant
    _parallel(lambda r0, r1: fn(_ptr(w_packed), _ptr(w_scale), g, r0, r1, K, alg, _ptr(out_p), _ptr(out_s)),
              N, threads)
    return out_p, out_s


def act_quant(x_bf16_bits, alg=SCALE_OCP, threads=1):
    """bf16 (as uint16 bits) [M, K] -> (packed [M, K/2], row-major E8M0 [M, K/32])."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    M, K = x.shape
    out_p = np.empty((M, K // 2), np.uint8)
    out_s = np.empty((M, K // 32), np.uint8)
    L = lib()
    _parallel(lambda r0, r1: L.orc_act_quant(_ptr(x), r0, r1, K, alg, _ptr(out_p), _ptr(out_s)),
              M, threads)
    return out_p, out_s


def gemm(a, sa, b, sb, bias_bf16_bits=None, rows=None, cols=None, threads=1):
    """float64 reference over dequantized MXFP4 operands.

    a [M, K/2], sa row-major [M, K/32]; b [N, K/2], sb row-major [N, K/32].
    Returns (ref, absum) of shape [len(rows), len(cols)].
    """
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    sa = np.ascontiguousarray(sa)
    sb = np.ascontiguousarray(sb)
    M, half = a.shape
    N = b.shape[0]
    K = 2 * half
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    bias = None if bias_bf16_bits is None else np.ascontiguousarray(bias_bf16_bits, np.uint16)
    ref = np.empty((len(rows), len(cols)), np.float64)
    absum = np.empty_like(ref)
    L = lib()

    def run(r0, r1):
        sub_rows = np.ascontiguousarray(rows[r0:r1])
        r = np.empty((r1 - r0, len(cols)), np.float64)
        s = np.empty_like(r)
        L.orc_gemm(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(bias), K, _ptr(sub_rows), r1 - r0,
                   _ptr(cols), len(cols), _ptr(r), _ptr(s))
        ref[r0:r1] = r
        absum[r0:r1] = s

    _parallel(run, len(rows), threads)
    return ref, absum


def bf16_encode(f: float) -> int:
    return lib().orc_bf16_encode(float(f))


def smooth_prepare(mul_scale_f32):
    """float32 [K] -> (bf16 bits [K], count of rejected values)."""
    m = np.ascontiguousarray(mul_scale_f32, np.float32)
    out = np.empty(m.shape, np.uint16)
    bad = lib().orc_smooth_prepare(_ptr(m), m.size, _ptr(out))
    return out, int(bad)


def smooth_apply(x_bf16_bits, m_bf16_bits):
    """bf16(x * m) per element, m per input channel (bf16 bits)."""
    x = np.ascontiguousarray(x_bf16_bits, np.uint16)
    m = np.ascontiguousarray(m_bf16_bits, np.uint16)
    rows, K = x.shape
    out = np.empty_like(x)
    lib().orc_smooth_apply(_ptr(x), _ptr(m), rows, K, _ptr(out))
    return out


def mx8_shared_exp(amax: float) -> int:
    return lib().orc_mx8_shared_exp(float(amax))


def act_quant_mxfp8(x_bf16_bits, threads=1):
    """bf16 (as uint16 bits) [M, K] -> (E4M3 codes [M, K], row-major E8M0 [M, K/32])."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    M, K = x.shape
    out_c = np.empty((M, K), np.uint8)
    out_s = np.empty((M, K // 32), np.uint8)
    L = lib()
    _parallel(lambda r0, r1: L.orc_act_quant_mxfp8(_ptr(x), r0, r1, K, _ptr(out_c), _ptr(out_s)), M, threads)
    return out_c, out_s


def gemm_w4a8(a8, sa, b, sb, bias_bf16_bits=None, rows=None, cols=None, threads=1):
    """float64 reference of MXFP8 activations x MXFP4 weights.

    a8 [M, K] E4M3 bytes, sa row-major [M, K/32]; b [N, K/2], sb row-major [N, K/32].
    Returns (ref, absum) of shape [len(rows), len(cols)].
    """
    a8 = np.ascontiguousarray(a8)
    b = np.ascontiguousarray(b)
    sa = np.ascontiguousarray(sa)
    sb = np.ascontiguousarray(sb)
    M, K = a8.shape
    N = b.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    bias = None if bias_bf16_bits is None else np.ascontiguousarray(bias_bf16_bits, np.uint16)
    ref = np.empty((len(rows), len(cols)), np.float64)
    absum = np.empty_like(ref)
    L = lib()

    def run(r0, r1):
        sub_rows = np.ascontiguousarray(rows[r0:r1])
        r = np.empty((r1 - r0, len(cols)), np.float64)
        s = np.empty_like(r)
        L.orc_gemm_w4a8(_ptr(a8), _ptr(sa), _ptr(b), _ptr(sb), _ptr(bias), K, _ptr(sub_rows), r1 - r0,
                        _ptr(cols), len(cols), _ptr(r), _ptr(s))
        ref[r0:r1] = r
        absum[r0:r1] = s

    _parallel(run, len(rows), threads)
    return ref, absum


def gemm_nvfp4(a, sa, b, sb, alpha, bias_bf16_bits=None, rows=None, cols=None, threads=1):
    """float64 reference of the NVFP4 x NVFP4 GEMM (codes times E4M3 scales, times alpha).

    a [M, K/2], sa row-major E4M3 [M, K/16]; b [N, K/2], sb row-major [N, K/16].
    Returns (ref, absum) of shape [len(rows), len(cols)].
    """
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    sa = np.ascontiguousarray(sa)
    sb = np.ascontiguousarray(sb)
    M, half = a.shape
    N = b.shape[0]
    K = 2 * half
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    bias = None if bias_bf16_bits is None else np.ascontiguousarray(bias_bf16_bits, np.uint16)
    ref = np.empty((len(rows), len(cols)), np.float64)
    absum = np.empty_like(ref)
    L = lib()

    def run(r0, r1):
        sub_rows = np.ascontiguousarray(rows[r0:r1])
        r = np.empty((r1 - r0, len(cols)), np.float64)
        s = np.empty_like(r)
        L.orc_gemm_nvfp4(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), float(alpha), _ptr(bias), K, _ptr(sub_rows),
                         r1 - r0, _ptr(cols), len(cols), _ptr(r), _ptr(s))
        ref[r0:r1] = r
        absum[r0:r1] = s

    _parallel(run, len(rows), threads)
    return ref, absum


def gemm_grouped(a, sa, b, sb, bias_bf16_bits, row_offsets, rows=None, cols=None, threads=1):
    """Per expert e, rows [off[e], off[e+1]) of a against expert e's b[e] / sb[e]."""
    E = len(row_offsets) - 1
    total = int(row_offsets[-1])
    rows = np.arange(total, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    N = b.shape[1]
    cols = np.arange(N, dtype=np.int64) if cols is None else np.asarray(cols, np.int64)
    ref = np.empty((len(rows), len(cols)), np.float64)
    absum = np.empty_like(ref)
    expert_of = np.searchsorted(np.asarray(row_offsets), rows, side="right") - 1
    for e in range(E):
        sel = np.nonzero(expert_of == e)[0]
        if len(sel) == 0:
            continue
        bias = None if bias_bf16_bits is None else bias_bf16_bits[e]
        r, s = gemm(a, sa, b[e], sb[e], bias, rows=rows[sel], cols=cols, threads=threads)
        ref[sel] = r
        absum[sel] = s
    return ref, absum


# ---------------------------------------------------------- DualScale
def dual_dequant(packed, fine, coarse) -> np.ndarray:
    """DualScale weight -> float64 [rows, K] (code x 2^(fine-127) x coarse)."""
    packed = np.ascontiguousarray(packed, np.uint8)
    fine = np.ascontiguousarray(fine, np.uint8)
    coarse = np.ascontiguousarray(coarse, np.float32)
    rows, half = packed.shape
    out = np.empty((rows, 2 * half), np.float64)
    lib().orc_dual_dequant(_ptr(packed), _ptr(fine), _ptr(coarse), rows, 2 * half, _ptr(out))
    return out


def dual_quantize(w_bf16_bits, threads=1):
    """bf16 bits [N, K] (K % 512 == 0) -> (codes [N, K/2] u8, fine E8M0
    [N, K/32] u8, coarse [N, K/512] float32) by the online dual-level rule."""
    w = np.ascontiguousarray(w_bf16_bits, np.uint16)
    N, K = w.shape
    packed = np.empty((N, K // 2), np.uint8)
    fine = np.empty((N, K // 32), np.uint8)
    coarse = np.empty((N, K // 512), np.float32)
    L = lib()
    _parallel(lambda r0, r1: L.orc_dual_quantize(_ptr(w), r0, r1, K, _ptr(packed), _ptr(fine), _ptr(coarse)),
              N, threads)
    return packed, fine, coarse


def gemm_dual(a, sa, b, fine, coarse, bias_bf16_bits=None, rows=None, cols=None, threads=1):
    """float64 reference: MXFP4 activations x DualScale weights (+ bias)."""
    a = np.ascontiguousarray(a)
    sa = np.ascontiguousarray(sa)
    b = np.ascontiguousarray(b)
    fine = np.ascontiguousarray(fine, np.uint8)
    coarse = np.ascontiguousarray(coarse, np.float32)
    M, half = a.shape
    N = b.shape[0]
    K = 2 * half
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    bias = None if bias_bf16_bits is None else np.ascontiguousarray(bias_bf16_bits, np.uint16)
    ref = np.empty((len(rows), len(cols)), np.float64)
    absum = np.empty_like(ref)
    L = lib()

    def run(r0, r1):
        sub_rows = np.ascontiguousarray(rows[r0:r1])
        r = np.empty((r1 - r0, len(cols)), np.float64)
        s_ = np.empty_like(r)
        L.orc_gemm_dual(_ptr(a), _ptr(sa), _ptr(b), _ptr(fine), _ptr(coarse), _ptr(bias), K, _ptr(sub_rows),
                        r1 - r0, _ptr(cols), len(cols), _ptr(r), _ptr(s_))
        ref[r0:r1] = r
        absum[r0:r1] = s_

    _parallel(run, len(rows), threads)
    return ref, absum


# ---------------------------------------------------------- input producer
def nvfp4_global_scale(x_bf16_bits) -> float:
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    return float(lib().orc_nvfp4_global_scale(_ptr(x), x.size))


def nvfp4_quantize(x_bf16_bits, g: float, threads=1):
    """bf16 bits [N, K] -> (packed [N, K/2] u8, E4M3 [N, K/16] u8) for global scale g."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    N, K = x.shape
    out_p = np.empty((N, K // 2), np.uint8)
    out_s = np.empty((N, K // 16), np.uint8)
    L = lib()
    _parallel(lambda r0, r1: L.orc_nvfp4_quantize(_ptr(x), g, r0, r1, K, _ptr(out_p), _ptr(out_s)),
              N, threads)
    return out_p, out_s


# ---------------------------------------------------------- SF layout
def sf_swizzled_bytes(rows: int, kblocks: int) -> int:
    return int(lib().orc_sf_swizzled_bytes(rows, kblocks))


def sf_swizzled_offset(r: int, c: int, kblocks: int) -> int:
    return int(lib().orc_sf_swizzled_offset(r, c, kblocks))


def sf_swizzle(rowmajor: np.ndarray) -> np.ndarray:
    rowmajor = np.ascontiguousarray(rowmajor, np.uint8)
    rows, kb = rowmajor.shape
    out = np.empty(sf_swizzled_bytes(rows, kb), np.uint8)
    lib().orc_sf_swizzle(_ptr(rowmajor), rows, kb, _ptr(out))
    return out

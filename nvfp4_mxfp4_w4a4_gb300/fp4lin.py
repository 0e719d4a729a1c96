"""ctypes binding of libfp4lin (argument marshalling only).

Every function here has the name and argument order of the C entry point
declared in include/fp4lin.h.  Tensor arguments may be torch tensors (their
data pointers are passed), plain integers (raw device pointers) or None
(NULL).  `stream` defaults to torch's current CUDA stream.  A non-OK status
raises Fp4Error.  There is no fallback: if the library is missing or the
GPU is not sm_103, calls fail.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp4lin.so")

FP4_OK = 0
FP4_ERR_INVALID_ARG = 1
FP4_ERR_SHAPE = 2
FP4_ERR_ALIGNMENT = 3
FP4_ERR_UNSUPPORTED = 4
FP4_ERR_CUDA = 5
FP4_ERR_TIMEOUT = 6
FP4_SCALE_OCP = 0
FP4_SCALE_UOS = 2
FP4_SF_SWIZZLED = 0
FP4_SF_ROWMAJOR = 1

# every symbol the header declares
SYMBOLS = (
    "fp4_sf_bytes", "fp4_sf_bytes_grouped", "fp4_status_string", "fp4_get_device_status",
    "fp4_requant_nvfp4_to_mxfp4", "fp4_requant_nvfp4_to_mxfp4_ex", "fp4_requant_nvfp4_to_mxfp4_grouped",
    "fp4_quant_act_mxfp4",
    "fp4_quant_act_mxfp4_grouped", "fp4_quant_nvfp4", "fp4_gemm_mxfp4", "fp4_gemm_workspace_size",
    "fp4_gemm_mxfp4_ws", "fp4_gemm_mxfp4_noalloc", "fp4_gemm_mxfp4_grouped",
    "fp4_quant_nvfp4_ex", "fp4_sf_bytes_nvfp4", "fp4_sf_swizzle", "fp4_gemm_nvfp4",
    "fp4_quant_act_mxfp8", "fp4_gemm_w4a8", "fp4_gemm_w4a8_workspace_size", "fp4_gemm_mxfp4_ex",
    "fp4_smooth_prepare", "fp4_quant_act_mxfp4_smooth", "fp4_quant_act_mxfp8_smooth",
    "fp4_linear_workspace_size", "fp4_linear", "fp4_linear_grouped_workspace_size", "fp4_linear_grouped",
    "fp4_debug_set_wait_fault", "fp4_quant_dualscale", "fp4_gemm_mxfp4_dualscale",
)


class Fp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)}")
        self.status = status


class fp4_quant_opts(ctypes.Structure):
    _fields_ = [("scale_alg", ctypes.c_int32), ("sf_layout", ctypes.c_int32), ("flags", ctypes.c_uint32)]


FP4_QUANT_BF16_INTERMEDIATE = 1


class fp4_linear_opts(ctypes.Structure):
    _fields_ = [("act_format", ctypes.c_int32), ("scale_alg", ctypes.c_int32), ("mul_scale_bf16", ctypes.c_void_p),
                ("gemm_flags", ctypes.c_uint32)]


FP4_ACT_MXFP4 = 0
FP4_ACT_MXFP8 = 1
FP4_LINEAR_FUSED_QUANT = 2


_lib = None
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


def load(path: str = LIB_PATH):
    """Loads the shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise FileNotFoundError(f"{path} is missing: build it with nvfp4_mxfp4_w4a4_gb300.build.build()")
        L = ctypes.CDLL(path)
        sig = {
            "fp4_sf_bytes": (ctypes.c_size_t, [_i64, _i64, _i32]),
            "fp4_sf_bytes_grouped": (ctypes.c_size_t, [_i64, _i32, _i64]),
            "fp4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "fp4_get_device_status": (ctypes.c_int, []),
            "fp4_debug_set_wait_fault": (ctypes.c_int, [ctypes.c_uint64, _i32]),
            "fp4_quant_dualscale": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _i32, _p]),
            "fp4_gemm_mxfp4_dualscale": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p,
                                                        ctypes.c_size_t, _p]),
            "fp4_requant_nvfp4_to_mxfp4": (ctypes.c_int, [_p, _p, ctypes.c_float, _p, _p, _i64, _i64, _p]),
            "fp4_requant_nvfp4_to_mxfp4_ex": (ctypes.c_int, [_p, _p, ctypes.c_float, _p, _p, _i64, _i64,
                                                             ctypes.POINTER(fp4_quant_opts), _p]),
            "fp4_requant_nvfp4_to_mxfp4_grouped": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i64, _i64,
                                                                  ctypes.POINTER(fp4_quant_opts), _p]),
            "fp4_quant_act_mxfp4": (ctypes.c_int, [_p, _p, _p, _i64, _i64, ctypes.POINTER(fp4_quant_opts), _p]),
            "fp4_quant_act_mxfp4_grouped": (ctypes.c_int, [_p, _p, _i32, _i64, _i64, _p, _p,
                                                           ctypes.POINTER(fp4_quant_opts), _p]),
            "fp4_quant_nvfp4": (ctypes.c_int, [_p, ctypes.c_float, _p, _p, _i64, _i64, _p]),
            "fp4_gemm_mxfp4": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p]),
            "fp4_gemm_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64]),
            "fp4_gemm_mxfp4_ws": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p, ctypes.c_size_t, _p]),
            "fp4_gemm_mxfp4_noalloc": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p]),
            "fp4_gemm_mxfp4_grouped": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _p, _i32, _i64, _i64, _i64, _p]),
            "fp4_quant_nvfp4_ex": (ctypes.c_int, [_p, ctypes.c_float, _p, _p, _i64, _i64, _i32, _p]),
            "fp4_sf_bytes_nvfp4": (ctypes.c_size_t, [_i64, _i64, _i32]),
            "fp4_sf_swizzle": (ctypes.c_int, [_p, _p, _i64, _i64, _p]),
            "fp4_gemm_nvfp4": (ctypes.c_int, [_p, _p, _p, _p, ctypes.c_float, _p, _p, _i64, _i64, _i64, _p,
                                              ctypes.c_size_t, _p]),
            "fp4_quant_act_mxfp8": (ctypes.c_int, [_p, _p, _p, _i64, _i64, _i32, _p]),
            "fp4_gemm_w4a8": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p, ctypes.c_size_t, _p]),
            "fp4_gemm_w4a8_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64]),
            "fp4_gemm_mxfp4_ex": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p, ctypes.c_size_t,
                                                 ctypes.c_uint32, _p]),
            "fp4_smooth_prepare": (ctypes.c_int, [_p, _p, _i64, _p, _p]),
            "fp4_quant_act_mxfp4_smooth": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64,
                                                          ctypes.POINTER(fp4_quant_opts), _p]),
            "fp4_quant_act_mxfp8_smooth": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _i32, _p]),
            "fp4_linear_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64, ctypes.POINTER(fp4_linear_opts)]),
            "fp4_linear": (ctypes.c_int, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, ctypes.c_size_t,
                                          ctypes.POINTER(fp4_linear_opts), _p]),
            "fp4_linear_grouped_workspace_size": (ctypes.c_size_t, [_i64, _i32, _i64]),
            "fp4_linear_grouped": (ctypes.c_int, [_p, _p, _i32, _i64, _p, _p, _p, _p, _i64, _i64, _p, ctypes.c_size_t,
                                                  ctypes.POINTER(fp4_quant_opts), _p]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _opts(scale_alg, sf_layout, flags=0):
    if scale_alg is None and sf_layout is None and not flags:
        return None
    o = fp4_quant_opts(FP4_SCALE_OCP if scale_alg is None else scale_alg,
                       FP4_SF_SWIZZLED if sf_layout is None else sf_layout, flags)
    return ctypes.byref(o)


def _check(status: int, where: str):
    if status != FP4_OK:
        raise Fp4Error(status, where)


def status_string(status: int) -> str:
    return load().fp4_status_string(status).decode()


def fp4_sf_bytes(rows: int, K: int, sf_layout: int = FP4_SF_SWIZZLED) -> int:
    return load().fp4_sf_bytes(rows, K, sf_layout)


def fp4_sf_bytes_grouped(total_M: int, E: int, K: int) -> int:
    return load().fp4_sf_bytes_grouped(total_M, E, K)


def fp4_get_device_status() -> int:
    return load().fp4_get_device_status()


def fp4_debug_set_wait_fault(wait_limit_ns: int = 0, withhold_split_signal: int = 0):
    """Test hook: limit of the GEMMs' bounded device waits (0 = the default
    1 s) and whether a split-K partial withholds its ready signal."""
    _check(load().fp4_debug_set_wait_fault(wait_limit_ns, withhold_split_signal), "fp4_debug_set_wait_fault")


def fp4_requant_nvfp4_to_mxfp4(w_packed, w_scale_e4m3, w_global, out_packed, out_scale, N, K, stream=None,
                               scale_alg=None, sf_layout=None, bf16_intermediate=False):
    """bf16_intermediate: round each decoded value to bf16 before the block rule."""
    L = load()
    flags = FP4_QUANT_BF16_INTERMEDIATE if bf16_intermediate else 0
    if scale_alg is None and sf_layout is None and not flags:
        st = L.fp4_requant_nvfp4_to_mxfp4(_ptr(w_packed), _ptr(w_scale_e4m3), float(w_global), _ptr(out_packed),
                                          _ptr(out_scale), N, K, _stream(stream))
    else:
        st = L.fp4_requant_nvfp4_to_mxfp4_ex(_ptr(w_packed), _ptr(w_scale_e4m3), float(w_global),
                                             _ptr(out_packed), _ptr(out_scale), N, K,
                                             _opts(scale_alg, sf_layout, flags), _stream(stream))
    _check(st, "fp4_requant_nvfp4_to_mxfp4")


def fp4_requant_nvfp4_to_mxfp4_grouped(w_packed, w_scale_e4m3, w_global, out_packed, out_scale, E, N, K,
                                       stream=None, scale_alg=None, sf_layout=None, bf16_intermediate=False):
    """w_global: device array of E float32 global scales."""
    flags = FP4_QUANT_BF16_INTERMEDIATE if bf16_intermediate else 0
    st = load().fp4_requant_nvfp4_to_mxfp4_grouped(_ptr(w_packed), _ptr(w_scale_e4m3), _ptr(w_global),
                                                   _ptr(out_packed), _ptr(out_scale), E, N, K,
                                                   _opts(scale_alg, sf_layout, flags), _stream(stream))
    _check(st, "fp4_requant_nvfp4_to_mxfp4_grouped")


def fp4_quant_act_mxfp4(x_bf16, out_packed, out_scale, M, K, stream=None, scale_alg=None, sf_layout=None):
    st = load().fp4_quant_act_mxfp4(_ptr(x_bf16), _ptr(out_packed), _ptr(out_scale), M, K,
                                    _opts(scale_alg, sf_layout), _stream(stream))
    _check(st, "fp4_quant_act_mxfp4")


def fp4_quant_act_mxfp4_grouped(x_bf16, row_offsets, E, total_M, K, out_packed, out_scale, stream=None,
                                scale_alg=None):
    st = load().fp4_quant_act_mxfp4_grouped(_ptr(x_bf16), _ptr(row_offsets), E, total_M, K, _ptr(out_packed),
                                            _ptr(out_scale), _opts(scale_alg, None), _stream(stream))
    _check(st, "fp4_quant_act_mxfp4_grouped")


def fp4_quant_nvfp4(x_bf16, g, out_packed, out_scale_e4m3, M, K, stream=None):
    st = load().fp4_quant_nvfp4(_ptr(x_bf16), float(g), _ptr(out_packed), _ptr(out_scale_e4m3), M, K,
                                _stream(stream))
    _check(st, "fp4_quant_nvfp4")


def fp4_quant_nvfp4_ex(x_bf16, g, out_packed, out_scale_e4m3, M, K, sf_layout=FP4_SF_SWIZZLED, stream=None):
    st = load().fp4_quant_nvfp4_ex(_ptr(x_bf16), float(g), _ptr(out_packed), _ptr(out_scale_e4m3), M, K, sf_layout,
                                   _stream(stream))
    _check(st, "fp4_quant_nvfp4_ex")


def fp4_sf_bytes_nvfp4(rows: int, K: int, sf_layout: int = FP4_SF_SWIZZLED) -> int:
    return load().fp4_sf_bytes_nvfp4(rows, K, sf_layout)


def fp4_sf_swizzle(in_rowmajor, out, rows, kblocks, stream=None):
    st = load().fp4_sf_swizzle(_ptr(in_rowmajor), _ptr(out), rows, kblocks, _stream(stream))
    _check(st, "fp4_sf_swizzle")


def fp4_gemm_nvfp4(a, sa, b, sb, alpha, bias_bf16, out_bf16, M, N, K, workspace=None, workspace_bytes=None,
                   stream=None):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().fp4_gemm_nvfp4(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), float(alpha), _ptr(bias_bf16), _ptr(out_bf16),
                               M, N, K, _ptr(workspace), workspace_bytes, _stream(stream))
    _check(st, "fp4_gemm_nvfp4")


def fp4_quant_act_mxfp8(x_bf16, out_e4m3, out_scale, M, K, sf_layout=FP4_SF_SWIZZLED, stream=None):
    st = load().fp4_quant_act_mxfp8(_ptr(x_bf16), _ptr(out_e4m3), _ptr(out_scale), M, K, sf_layout,
                                    _stream(stream))
    _check(st, "fp4_quant_act_mxfp8")


def fp4_smooth_prepare(mul_scale_f32, out_bf16, K, bad_count, stream=None):
    """Converts the float32 smooth tensor to bf16; bad_count (device int32)
    receives the number of values that loading must reject."""
    st = load().fp4_smooth_prepare(_ptr(mul_scale_f32), _ptr(out_bf16), K, _ptr(bad_count), _stream(stream))
    _check(st, "fp4_smooth_prepare")


def fp4_quant_act_mxfp4_smooth(x_bf16, mul_scale_bf16, out_packed, out_scale, M, K, stream=None, scale_alg=None,
                               sf_layout=None):
    st = load().fp4_quant_act_mxfp4_smooth(_ptr(x_bf16), _ptr(mul_scale_bf16), _ptr(out_packed), _ptr(out_scale),
                                           M, K, _opts(scale_alg, sf_layout), _stream(stream))
    _check(st, "fp4_quant_act_mxfp4_smooth")


def fp4_quant_act_mxfp8_smooth(x_bf16, mul_scale_bf16, out_e4m3, out_scale, M, K, sf_layout=FP4_SF_SWIZZLED,
                               stream=None):
    st = load().fp4_quant_act_mxfp8_smooth(_ptr(x_bf16), _ptr(mul_scale_bf16), _ptr(out_e4m3), _ptr(out_scale), M,
                                           K, sf_layout, _stream(stream))
    _check(st, "fp4_quant_act_mxfp8_smooth")


def _linear_opts(act_format, scale_alg, mul_scale_bf16, gemm_flags):
    return fp4_linear_opts(act_format, scale_alg, _ptr(mul_scale_bf16), gemm_flags)


def fp4_linear_workspace_size(M, N, K, act_format=FP4_ACT_MXFP4, scale_alg=FP4_SCALE_OCP, mul_scale_bf16=None,
                              gemm_flags=0) -> int:
    o = _linear_opts(act_format, scale_alg, mul_scale_bf16, gemm_flags)
    return load().fp4_linear_workspace_size(M, N, K, ctypes.byref(o))


def fp4_linear(x_bf16, w, sw, bias_bf16, out_bf16, M, N, K, workspace, workspace_bytes=None,
               act_format=FP4_ACT_MXFP4, scale_alg=FP4_SCALE_OCP, mul_scale_bf16=None, gemm_flags=0, stream=None):
    """y = quant(x [* mul_scale]) . W^T (+ bias) in one call; workspace from
    fp4_linear_workspace_size, zeroed once before first use."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    o = _linear_opts(act_format, scale_alg, mul_scale_bf16, gemm_flags)
    st = load().fp4_linear(_ptr(x_bf16), _ptr(w), _ptr(sw), _ptr(bias_bf16), _ptr(out_bf16), M, N, K, _ptr(workspace),
                           workspace_bytes, ctypes.byref(o), _stream(stream))
    _check(st, "fp4_linear")


def fp4_linear_grouped_workspace_size(total_M, E, K) -> int:
    return load().fp4_linear_grouped_workspace_size(total_M, E, K)


def fp4_linear_grouped(x_bf16, row_offsets, E, total_M, w, sw, bias_bf16, out_bf16, N, K, workspace,
                       workspace_bytes=None, scale_alg=None, stream=None):
    """MoE form of fp4_linear: grouped act-quant then grouped GEMM."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = load().fp4_linear_grouped(_ptr(x_bf16), _ptr(row_offsets), E, total_M, _ptr(w), _ptr(sw), _ptr(bias_bf16),
                                   _ptr(out_bf16), N, K, _ptr(workspace), workspace_bytes, _opts(scale_alg, None),
                                   _stream(stream))
    _check(st, "fp4_linear_grouped")


def fp4_gemm_w4a8_workspace_size(M, N, K) -> int:
    return load().fp4_gemm_w4a8_workspace_size(M, N, K)


def fp4_gemm_w4a8(a_e4m3, sa, b, sb, bias_bf16, out_bf16, M, N, K, workspace=None, workspace_bytes=None,
                  stream=None):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().fp4_gemm_w4a8(_ptr(a_e4m3), _ptr(sa), _ptr(b), _ptr(sb), _ptr(bias_bf16), _ptr(out_bf16), M, N, K,
                              _ptr(workspace), workspace_bytes, _stream(stream))
    _check(st, "fp4_gemm_w4a8")


def fp4_gemm_mxfp4(a, sa, b, sb, bias_bf16, out_bf16, M, N, K, stream=None):
    st = load().fp4_gemm_mxfp4(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(bias_bf16), _ptr(out_bf16), M, N, K,
                               _stream(stream))
    _check(st, "fp4_gemm_mxfp4")


def fp4_gemm_workspace_size(M, N, K) -> int:
    return load().fp4_gemm_workspace_size(M, N, K)


def fp4_gemm_mxfp4_ws(a, sa, b, sb, bias_bf16, out_bf16, M, N, K, workspace, workspace_bytes=None, stream=None):
    """workspace: device buffer (e.g. a zero-initialised uint8 tensor) or None."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().fp4_gemm_mxfp4_ws(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(bias_bf16), _ptr(out_bf16), M, N, K,
                                  _ptr(workspace), workspace_bytes, _stream(stream))
    _check(st, "fp4_gemm_mxfp4_ws")


FP4_GEMM_WEIGHTS_STATIC = 1


def fp4_gemm_mxfp4_ex(a, sa, b, sb, bias_bf16, out_bf16, M, N, K, workspace=None, workspace_bytes=None, flags=0,
                      stream=None):
    """flags: FP4_GEMM_WEIGHTS_STATIC when b / sb are not written by the kernel
    enqueued just before this call (the GEMM then streams its first weight
    stages while that kernel finishes)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().fp4_gemm_mxfp4_ex(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(bias_bf16), _ptr(out_bf16), M, N, K,
                                  _ptr(workspace), workspace_bytes, flags, _stream(stream))
    _check(st, "fp4_gemm_mxfp4_ex")


def fp4_gemm_mxfp4_noalloc(a, sa, b, sb, bias_bf16, out_bf16, M, N, K, stream=None):
    """The GEMM with the library's fixed device scratch (allocates nothing)."""
    st = load().fp4_gemm_mxfp4_noalloc(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(bias_bf16), _ptr(out_bf16), M, N,
                                       K, _stream(stream))
    _check(st, "fp4_gemm_mxfp4_noalloc")


def fp4_gemm_mxfp4_grouped(a, sa, b, sb, bias_bf16, out_bf16, row_offsets, E, total_M, N, K, stream=None):
    st = load().fp4_gemm_mxfp4_grouped(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(bias_bf16), _ptr(out_bf16),
                                       _ptr(row_offsets), E, total_M, N, K, _stream(stream))
    _check(st, "fp4_gemm_mxfp4_grouped")


def fp4_quant_dualscale(w_bf16, out_packed, out_fine, out_coarse, N, K, sf_layout=FP4_SF_SWIZZLED, stream=None):
    """bf16 weight -> DualScale codes, fine E8M0 scales and coarse float32 scales."""
    st = load().fp4_quant_dualscale(_ptr(w_bf16), _ptr(out_packed), _ptr(out_fine), _ptr(out_coarse), N, K,
                                    sf_layout, _stream(stream))
    _check(st, "fp4_quant_dualscale")


def fp4_gemm_mxfp4_dualscale(a, sa, b, sb, coarse, bias_bf16, out_bf16, M, N, K, workspace=None,
                             workspace_bytes=None, stream=None):
    """MXFP4 activations x DualScale weights (+ bias), bf16 out."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().fp4_gemm_mxfp4_dualscale(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(coarse), _ptr(bias_bf16),
                                         _ptr(out_bf16), M, N, K, _ptr(workspace), workspace_bytes, _stream(stream))
    _check(st, "fp4_gemm_mxfp4_dualscale")

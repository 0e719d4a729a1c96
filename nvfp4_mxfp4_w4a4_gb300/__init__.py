"""libfp4lin: the W4A4 MXFP4 linear layer on one GB300 (sm_103a).

The compute path is the CUDA library libfp4lin.so (C ABI in
include/fp4lin.h); this package only builds it and binds it with ctypes.
"""
from .fp4lin import (  # noqa: F401
    FP4_SCALE_OCP,
    FP4_SCALE_UOS,
    FP4_SF_ROWMAJOR,
    FP4_SF_SWIZZLED,
    SYMBOLS,
    Fp4Error,
    fp4_gemm_mxfp4,
    fp4_gemm_mxfp4_grouped,
    fp4_get_device_status,
    fp4_quant_act_mxfp4,
    fp4_quant_act_mxfp4_grouped,
    fp4_quant_nvfp4,
    fp4_requant_nvfp4_to_mxfp4,
    fp4_sf_bytes,
    fp4_sf_bytes_grouped,
    load,
    status_string,
)

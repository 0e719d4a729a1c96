"""Shared helpers for the tests (no quantization arithmetic here)."""
from __future__ import annotations

import os

import numpy as np

THREADS = max(1, min(16, os.cpu_count() or 1))


def gpu_available() -> bool:
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def lib():
    """Builds (if needed) and loads the CUDA library."""
    from nvfp4_mxfp4_w4a4_gb300 import build as B
    from nvfp4_mxfp4_w4a4_gb300 import fp4lin

    B.build()
    fp4lin.load()
    return fp4lin


def dev(a: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def empty_u8(n: int):
    import torch

    # poison the buffer so unwritten bytes are visible
    return torch.full((max(1, n),), 0xA5, dtype=torch.uint8, device="cuda")


def host(t) -> np.ndarray:
    return t.cpu().numpy()


def bf16_bits_host(t) -> np.ndarray:
    import torch

    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def gemm_check(out_bits: np.ndarray, ref: np.ndarray, absum: np.ndarray):
    """Per-element tolerance |out - ref| <= 2^-8 |ref| + 1e-6 sum|a b|.
    Returns (ok, worst err/bound ratio)."""
    out = bf16_bits_to_f64(out_bits)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-6 * absum
    err = np.abs(out - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    return bool(np.all(err <= bound)), float(np.max(ratio)) if ratio.size else 0.0

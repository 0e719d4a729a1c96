"""Measured dense FP4 tensor-core peak: a tcgen05.mma kind::mxf4 issue-rate
probe (libfp4peak.so) run on every SM at once."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))


def measure(n: int = 256, iters: int = 4000, mmas_per_group: int = 4, with_cp: bool = False, reps: int = 3):
    """Returns dict(tflops, cycles_per_mma, ms) for MMAs of 128 x n x 64 issued
    back to back by one thread per SM on all SMs."""
    import torch

    from . import build as B

    B.build()
    lib = ctypes.CDLL(B.LIB_PEAK)
    f = lib.fp4_mma_peak_probe
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    best = None
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        err = f(n, iters, mmas_per_group, int(with_cp), sms, cycles.data_ptr(), status.data_ptr(), s.cuda_stream)
        b.record()
        torch.cuda.synchronize()
        if err != 0 or int(status.item()) != 0:
            raise RuntimeError(f"probe failed: cuda error {err}, status {int(status.item())}")
        ms = a.elapsed_time(b)
        if best is None or ms < best:
            best = ms
            cyc = float(cycles.float().mean())
    mmas = iters * mmas_per_group
    flops = 2.0 * 128 * n * 64 * mmas * sms
    return {"n": n, "with_cp": with_cp, "tflops": flops / (best * 1e-3) / 1e12, "cycles_per_mma": cyc / mmas,
            "ms": best, "sms": sms}

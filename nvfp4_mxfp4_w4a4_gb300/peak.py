"""Measured dense FP4 tensor-core peak: issue-rate probes of the block-scaled
FP4 MMA forms (libfp4peak.so) run on every SM at once."""
from __future__ import annotations

import ctypes

KINDS = {
    0: "kind::mxf4 scale_vec::2X (UE8M0, block 32)",
    1: "kind::mxf4nvf4 scale_vec::2X (UE8M0, block 32)",
    2: "kind::mxf4nvf4 scale_vec::4X (UE8M0, block 16)",
    3: "kind::mxf4nvf4 scale_vec::4X (UE4M3, block 16)",
    4: "kind::mxf8f6f4 scale_vec::1X (E4M3 x E2M1, UE8M0, block 32; K = 32)",
}

_lib = None


def _probe():
    global _lib
    if _lib is None:
        from . import build as B

        B.build()
        lib = ctypes.CDLL(B.LIB_PEAK)
        f = lib.fp4_mma_peak_probe3
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int] * 10 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        _lib = f
    return _lib


def measure(n: int = 256, iters: int = 4000, mmas_per_group: int = 4, with_cp: bool = False, reps: int = 3,
            kind: int = 0, ctag: int = 1, alt: bool = False, waits: int = 0, random_operands: bool = False):
    """Returns dict(tflops, cycles_per_mma, ms, ...) for MMAs of (128 ctag) x n x 64
    issued back to back by one thread per SM (per SM pair when ctag == 2) on
    all SMs.  waits: completed-barrier waits (and one commit) the issuing
    thread adds after each group of mmas_per_group MMAs."""
    import torch

    f = _probe()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas = sms // ctag * ctag
    cycles = torch.zeros(ctas // ctag, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    best = None
    cyc = 0.0
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        err = f(kind, ctag, n, iters, mmas_per_group, int(with_cp), int(alt), waits, int(random_operands), ctas,
                cycles.data_ptr(), status.data_ptr(), s.cuda_stream)
        b.record()
        torch.cuda.synchronize()
        if err != 0 or int(status.item()) != 0:
            raise RuntimeError(f"probe failed: cuda error {err}, status {int(status.item())}")
        ms = a.elapsed_time(b)
        if best is None or ms < best:
            best = ms
            cyc = float(cycles.float().mean())
    mmas = iters * mmas_per_group
    k = 32 if kind == 4 else 64  # K per instruction
    flops = 2.0 * 128 * ctag * n * k * mmas * (ctas // ctag)
    return {"kind": KINDS[kind], "cta_group": ctag, "n": n, "with_cp": with_cp, "alt_accumulators": alt,
            "mmas_per_group": mmas_per_group, "waits_per_group": waits, "random_operands": random_operands,
            "tflops": flops / (best * 1e-3) / 1e12, "cycles_per_mma": cyc / mmas, "ms": best, "sms": ctas}


def sweep():
    """Every form at N = 256 on both CTA groupings, plus N = 128 with one and
    two accumulators (cta_group::1) and on a pair; the decode tile widths
    N = 16, 32, 64 for kind::mxf4 and for the W4A8 form kind::mxf8f6f4
    (cta_group::1)."""
    rows = []
    for kind in (0, 1, 2, 3):
        for ctag in (1, 2):
            rows.append(measure(n=256, kind=kind, ctag=ctag))
        for alt in (False, True):
            rows.append(measure(n=128, kind=kind, ctag=1, alt=alt))
    rows.append(measure(n=256, kind=0, ctag=1, with_cp=True))
    rows.append(measure(n=256, kind=1, ctag=2, with_cp=True))
    for kind in (0, 4):
        for n in (16, 32, 64) + ((128, 256) if kind == 4 else ()):
            rows.append(measure(n=n, kind=kind, ctag=1))
    rows.append(measure(n=128, kind=0, ctag=2))
    # operand data, and the issuing thread's own per-stage work (a GEMM stage
    # of 8 MMAs: barrier waits that find their phase complete, one commit)
    for ctag in (1, 2):
        for waits in (0, 1, 2, 3, 4):
            rows.append(measure(n=256, kind=0, ctag=ctag, mmas_per_group=8, iters=2000, waits=waits,
                                random_operands=True))
    # narrower MMAs leave a wait exposed
    for n in (16, 128):
        for waits in (0, 1):
            rows.append(measure(n=n, kind=0, ctag=1, mmas_per_group=8, iters=2000, waits=waits, random_operands=True))
    return rows


if __name__ == "__main__":
    import json

    for r in sweep():
        print(json.dumps({k: (round(v, 2) if isinstance(v, float) else v) for k, v in r.items()}))

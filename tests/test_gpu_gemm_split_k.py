"""GPU parity of the workspace GEMM entry point (split-K scheduling for
decode-sized M) against the float64 oracle, through the C ABI.  The shapes
have at most half as many 128-row weight tiles as the GPU has SMs, so the
K stages of every tile are split between 2 to 8 CTAs and the first one adds
the others' fp32 partials.  Tolerance as for the plain GEMM:
|out - ref| <= 2^-8 |ref| + 1e-6 sum_k |a_k b_k|."""
import numpy as np
import pytest

import synth
from _util import THREADS, bf16_bits_host, dev, dev_bf16, gemm_check, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


def _operands(orc, M, N, K, seed):
    X = synth.bf16_normal(seed, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    W = synth.bf16_normal(seed + 1, synth.S_WEIGHT, (N, K), 0.02)
    a, sa = orc.act_quant(X, threads=THREADS)
    g = orc.nvfp4_global_scale(W)
    wp, ws = orc.nvfp4_quantize(W, g, threads=THREADS)
    b, sb = orc.requant(wp, ws, g, threads=THREADS)
    return a, sa, b, sb


def _workspace(L, M, N, K, split=True):
    import torch

    n = L.fp4_gemm_workspace_size(M, N, K)
    assert (n > 0) == split
    return torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")


def _run(L, orc, a, sa, b, sb, bias, M, N, K, ws):
    import torch

    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_mxfp4_ws(dev(a), dev(orc.sf_swizzle(sa)), dev(b), dev(orc.sf_swizzle(sb)),
                        None if bias is None else dev_bf16(bias), out, M, N, K, ws)
    assert L.fp4_get_device_status() == 0
    return bf16_bits_host(out)


def _sm_count():
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("M,N,K", [(1, 2048, 8192), (7, 2000, 8192), (32, 1024, 16384), (64, 4096, 16384),
                                   (64, 392, 30720), (33, 8192, 12288)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_split_k_matches_oracle(orc, L, M, N, K, with_bias):
    tiles, n = -(-N // 128), K // 512
    S = min(8, _sm_count() // tiles, n)
    assert S >= 2 and n * (S - 1) >= 10 * S, "shape must take the split-K path"
    a, sa, b, sb = _operands(orc, M, N, K, M * 7 + N)
    bias = synth.bf16_normal(N, synth.S_BIAS, (N,), 0.01) if with_bias else None
    ws = _workspace(L, M, N, K)
    out = _run(L, orc, a, sa, b, sb, bias, M, N, K, ws)
    ref, absum = orc.gemm(a, sa, b, sb, bias, threads=THREADS)
    ok, ratio = gemm_check(out, ref, absum)
    assert ok, f"max err/bound = {ratio}"
    # every call leaves the counters at zero for the next one
    import torch

    assert int(torch.count_nonzero(ws[: 4 * _sm_count()])) == 0


def test_split_k_is_deterministic_and_reusable(orc, L):
    M, N, K = 64, 2048, 8192
    a, sa, b, sb = _operands(orc, M, N, K, 5)
    ws = _workspace(L, M, N, K)
    first = _run(L, orc, a, sa, b, sb, None, M, N, K, ws)
    for _ in range(3):
        assert np.array_equal(_run(L, orc, a, sa, b, sb, None, M, N, K, ws), first)


def test_workspace_entry_without_split_k(orc, L):
    """Shapes that do not split (M > 64, more tiles than half the SMs, no
    workspace) run the plain path through the same entry point."""
    for (M, N, K, use_ws) in ((100, 256, 1024, True), (16, 12288, 512, True), (8, 1024, 4096, False), (64, 4096, 4096, True)):
        a, sa, b, sb = _operands(orc, M, N, K, M + N)
        ws = _workspace(L, M, N, K, split=False) if use_ws else None
        out = _run(L, orc, a, sa, b, sb, None, M, N, K, ws)
        ref, absum = orc.gemm(a, sa, b, sb, threads=THREADS)
        ok, ratio = gemm_check(out, ref, absum)
        assert ok, f"{(M, N, K)}: max err/bound = {ratio}"


def test_withheld_partial_expires_the_bounded_wait(orc, L):
    """Failure path of the split-K hand-over, driven without a GPU fault: with
    a test hook, the last CTA never publishes its partial, so the finishing
    CTA's bounded wait (2 ms here) expires.  The call completes, the status
    word reports FP4_ERR_TIMEOUT (and reading it clears it), the withheld
    counter is left in the workspace, and once the caller zeroes the
    workspace again the next call is correct."""
    import torch

    M, N, K = 32, 1024, 16384
    a, sa, b, sb = _operands(orc, M, N, K, 11)
    ws = _workspace(L, M, N, K)
    good = _run(L, orc, a, sa, b, sb, None, M, N, K, ws)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_debug_set_wait_fault(2_000_000, 1)
    try:
        L.fp4_gemm_mxfp4_ws(dev(a), dev(orc.sf_swizzle(sa)), dev(b), dev(orc.sf_swizzle(sb)), None, out, M, N, K, ws)
        st = L.fp4_get_device_status()
    finally:
        L.fp4_debug_set_wait_fault(0, 0)
    assert st == L.FP4_ERR_TIMEOUT
    assert L.fp4_get_device_status() == 0
    assert int(torch.count_nonzero(ws[: 4 * _sm_count()])) > 0
    ws.zero_()
    assert np.array_equal(_run(L, orc, a, sa, b, sb, None, M, N, K, ws), good)

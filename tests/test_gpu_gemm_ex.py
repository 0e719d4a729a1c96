"""fp4_gemm_mxfp4_ex with FP4_GEMM_WEIGHTS_STATIC: the GEMM streams its first
weight stages while the kernel before it (here the activation quantizer,
writing into buffers filled with garbage just before) is still running.
The result must be bit-identical to the plain workspace entry point on the
finished activations (no early read of the activations), and within the GEMM
bound of the oracle."""
import numpy as np
import pytest

import synth
from _util import THREADS, bf16_bits_host, dev, dev_bf16, gemm_check, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


def _weight(orc, W_bits):
    g = orc.nvfp4_global_scale(W_bits)
    wp, ws = orc.nvfp4_quantize(W_bits, g, threads=THREADS)
    p, s = orc.requant(wp, ws, g, threads=THREADS)
    return p, s, orc.sf_swizzle(s)


@pytest.mark.parametrize("M,N,K", [(1, 14336, 1024), (32, 4096, 4096), (64, 1024, 8192), (8, 512, 16384),
                                   (200, 1024, 512)])
def test_static_weights_chain_matches_plain_entry(orc, L, M, N, K):
    import torch

    X = synth.bf16_normal(M + N, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    W = synth.bf16_normal(N + K, synth.S_WEIGHT, (N, K), 0.02)
    b, sb, sb_sw = _weight(orc, W)
    bd, sbd = dev(b), dev(sb_sw)
    xd = dev_bf16(X)
    need = L.fp4_gemm_workspace_size(M, N, K)
    ws = torch.zeros(max(need, 1), dtype=torch.uint8, device="cuda") if need else None
    a_p = torch.full((M, K // 2), 0x77, dtype=torch.uint8, device="cuda")
    a_s = torch.full((L.fp4_sf_bytes(M, K),), 0xFE, dtype=torch.uint8, device="cuda")
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    # quantize, then the GEMM with the flag, back to back on one stream
    L.fp4_quant_act_mxfp4(xd, a_p, a_s, M, K)
    L.fp4_gemm_mxfp4_ex(a_p, a_s, bd, sbd, None, out, M, N, K, ws, flags=L.FP4_GEMM_WEIGHTS_STATIC)
    assert L.fp4_get_device_status() == 0
    ref_out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_mxfp4_ws(a_p, a_s, bd, sbd, None, ref_out, M, N, K, ws)
    assert L.fp4_get_device_status() == 0
    got = bf16_bits_host(out)
    assert np.array_equal(got, bf16_bits_host(ref_out))
    a, sa = orc.act_quant(X, threads=THREADS)
    rows = np.unique(np.linspace(0, M - 1, min(M, 16)).astype(np.int64))
    ref, absum = orc.gemm(a, sa, b, sb, rows=rows, threads=THREADS)
    ok, ratio = gemm_check(got[rows], ref, absum)
    assert ok, f"max err/bound = {ratio}"

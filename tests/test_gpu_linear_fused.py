"""fp4_linear with FP4_LINEAR_FUSED_QUANT: for M <= 64 the GEMM quantizes
the bf16 activations itself ("Efficiently Serving NVFP4 Models ...", last
section, "Fusing activation quantization + GEMM").  The output must be the
same bits as the unfused call (the same quantizer arithmetic feeds the same
MMAs), for every token-tile width (M <= 16, <= 32, <= 64), K with an odd
number of 256-element slabs (one-slab stages), the OCP and UOS rules, the
smooth pre-scale, bias, the split-K path, and ragged token counts; one case
per tile width is also held to the oracle's bound directly."""
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
    return orc.requant(wp, ws, g, threads=THREADS)


def _run(L, X, b, sw, bias, M, N, K, ws, flags, alg, md):
    import torch

    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_linear(dev_bf16(X), b, sw, bias, out, M, N, K, ws, scale_alg=alg, mul_scale_bf16=md, gemm_flags=flags)
    assert L.fp4_get_device_status() == 0
    return bf16_bits_host(out)


# (M, N, K): tile widths 16 / 32 / 64; K = 1152 has 4.5 slabs of 256 (one-slab
# stages); N = 2048, K = 8192 takes the split-K path
CASES = [(1, 1024, 4096), (5, 640, 1152), (16, 2048, 8192), (17, 384, 2048), (32, 14336, 4096),
         (33, 512, 7168), (64, 896, 1152), (64, 2048, 8192)]


@pytest.mark.parametrize("M,N,K", CASES)
@pytest.mark.parametrize("mode", ["ocp", "uos", "smooth_bias"])
def test_fused_quant_linear_is_bit_identical(orc, L, M, N, K, mode):
    import torch

    X = synth.bf16_normal(M * 3 + N, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    b, sb = _weight(orc, synth.bf16_normal(N + 7 * K, synth.S_WEIGHT, (N, K), 0.02))
    alg = 2 if mode == "uos" else 0
    md, bias = None, None
    if mode == "smooth_bias":
        m = np.exp((synth.uniform(K + 1, synth.S_SCALES, K) - 0.5) * 4.0).astype(np.float32)
        mb, bad = orc.smooth_prepare(m)
        assert bad == 0
        md = dev_bf16(mb)
        bias = dev_bf16(synth.bf16_normal(N, synth.S_BIAS, (N,), 0.01))
    need = L.fp4_linear_workspace_size(M, N, K, scale_alg=alg, mul_scale_bf16=md)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    bd, swd = dev(b), dev(orc.sf_swizzle(sb))
    plain = _run(L, X, bd, swd, bias, M, N, K, ws, 0, alg, md)
    for _ in range(2):  # twice: the split-K counters are back at zero
        fused = _run(L, X, bd, swd, bias, M, N, K, ws, L.FP4_LINEAR_FUSED_QUANT, alg, md)
        assert np.array_equal(fused, plain)


@pytest.mark.parametrize("M,N,K", [(1, 1024, 4096), (20, 768, 1152), (64, 2048, 8192)])
def test_fused_quant_linear_matches_oracle(orc, L, M, N, K):
    import torch

    X = synth.bf16_normal(M + 2 * N, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    b, sb = _weight(orc, synth.bf16_normal(3 * N + K, synth.S_WEIGHT, (N, K), 0.02))
    bias = synth.bf16_normal(N + 3, synth.S_BIAS, (N,), 0.01)
    ws = torch.zeros(L.fp4_linear_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    got = _run(L, X, dev(b), dev(orc.sf_swizzle(sb)), dev_bf16(bias), M, N, K, ws, L.FP4_LINEAR_FUSED_QUANT, 0,
               None)
    aq, asf = orc.act_quant(X, threads=THREADS)
    ref, absum = orc.gemm(aq, asf, b, sb, bias, threads=THREADS)
    ok, ratio = gemm_check(got, ref, absum)
    assert ok, f"max err/bound = {ratio}"

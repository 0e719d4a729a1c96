"""fp4_linear, the serve-time linear layer in one call, against the oracle's
quantizer (optionally of bf16(x * mul_scale)) followed by its GEMM:
MXFP4 activations with the OCP and UOS rules, the smooth pre-scale, and the
W4A8 fallback; decode sizes that take the split-K path; within the GEMM
bound |out - ref| <= 2^-8 |ref| + 1e-6 sum_k |a_k b_k|."""
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


CASES = [(1, 256, 512), (33, 1024, 8192), (64, 14336, 1024), (200, 384, 640)]


@pytest.mark.parametrize("M,N,K", CASES)
@pytest.mark.parametrize("mode", ["a4_ocp", "a4_uos", "a4_smooth", "a8", "a8_smooth"])
def test_linear_matches_oracle(orc, L, M, N, K, mode):
    import torch

    X = synth.bf16_normal(M + N, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    W = synth.bf16_normal(N + K, synth.S_WEIGHT, (N, K), 0.02)
    bias = synth.bf16_normal(N, synth.S_BIAS, (N,), 0.01)
    b, sb = _weight(orc, W)
    a8 = mode.startswith("a8")
    alg = 2 if mode == "a4_uos" else 0
    mb = None
    Xq = X
    if mode.endswith("smooth"):
        m = np.exp((synth.uniform(K, synth.S_SCALES, K) - 0.5) * 4.0).astype(np.float32)
        mb, bad = orc.smooth_prepare(m)
        assert bad == 0
        Xq = orc.smooth_apply(X, mb)
    act = L.FP4_ACT_MXFP8 if a8 else L.FP4_ACT_MXFP4
    md = None if mb is None else dev_bf16(mb)
    need = L.fp4_linear_workspace_size(M, N, K, act_format=act, scale_alg=alg, mul_scale_bf16=md)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bd = dev(b)
    L.fp4_linear(dev_bf16(X), bd, dev(orc.sf_swizzle(sb)), dev_bf16(bias), out, M, N, K, ws, act_format=act,
                 scale_alg=alg, mul_scale_bf16=md)
    assert L.fp4_get_device_status() == 0
    got = bf16_bits_host(out)
    rows = np.unique(np.linspace(0, M - 1, min(M, 12)).astype(np.int64))
    if a8:
        aq, asf = orc.act_quant_mxfp8(Xq, threads=THREADS)
        ref, absum = orc.gemm_w4a8(aq, asf, b, sb, bias, rows=rows, threads=THREADS)
    else:
        aq, asf = orc.act_quant(Xq, alg, threads=THREADS)
        ref, absum = orc.gemm(aq, asf, b, sb, bias, rows=rows, threads=THREADS)
    ok, ratio = gemm_check(got[rows], ref, absum)
    assert ok, f"max err/bound = {ratio}"
    # a second call on the same workspace gives the same bits (counters back at zero)
    out2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_linear(dev_bf16(X), bd, dev(orc.sf_swizzle(sb)), dev_bf16(bias), out2, M, N, K, ws, act_format=act,
                 scale_alg=alg, mul_scale_bf16=md)
    assert np.array_equal(bf16_bits_host(out2), got)


def test_linear_rejects_small_workspace(L):
    import torch

    M, N, K = 8, 256, 512
    need = L.fp4_linear_workspace_size(M, N, K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    sw = torch.zeros(L.fp4_sf_bytes(N, K), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.Fp4Error) as err:
        L.fp4_linear(x, w, sw, None, out, M, N, K, ws, workspace_bytes=need - 1)
    assert err.value.status == L.FP4_ERR_INVALID_ARG


@pytest.mark.parametrize("counts,N,K", [([3, 0, 130, 1, 200], 136, 256), ([40] * 8, 512, 384)])
@pytest.mark.parametrize("alg", [0, 2])
def test_linear_grouped_matches_oracle(orc, L, counts, N, K, alg):
    import torch

    E = len(counts)
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    total = int(offsets[-1])
    X = synth.bf16_normal(total + N, synth.S_ACT, (total, K), 1.0, 0.01, 16.0)
    bs, sbs, sws = [], [], []
    for e in range(E):
        b, sb = _weight(orc, synth.bf16_normal(N * 10 + e, synth.S_WEIGHT, (N, K), 0.02))
        bs.append(b)
        sbs.append(sb)
        sws.append(orc.sf_swizzle(sb))
    bias = synth.bf16_normal(E + N, synth.S_BIAS, (E, N), 0.01)
    ws = torch.zeros(L.fp4_linear_grouped_workspace_size(total, E, K), dtype=torch.uint8, device="cuda")
    out = torch.full((total, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_linear_grouped(dev_bf16(X), dev(offsets), E, total, dev(np.stack(bs)), dev(np.concatenate(sws)),
                         dev_bf16(bias), out, N, K, ws, scale_alg=alg)
    assert L.fp4_get_device_status() == 0
    aq, asf = orc.act_quant(X, alg, threads=THREADS)
    ref, absum = orc.gemm_grouped(aq, asf, np.stack(bs), np.stack(sbs), bias, offsets, threads=THREADS)
    ok, ratio = gemm_check(bf16_bits_host(out), ref, absum)
    assert ok, f"max err/bound = {ratio}"

"""GPU parity of the smooth pre-scale ("W4A4 MXFP4 Quantization",
Pre-Quantized Single-Scale Weights: both paths quantize x * mul_scale, the
float32 tensor converted to bf16 at load with NaN/Inf/non-positive/overflow/
underflow values rejected): the conversion and rejection count, and the
MXFP4 and MXFP8 quantizers of bf16(x * m), byte for byte against the
oracle."""
import numpy as np
import pytest

import synth
from _util import THREADS, dev, dev_bf16, empty_u8, host, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


def _smooth_f32(K, seed):
    u = synth.uniform(seed, synth.S_SCALES, K)
    return np.exp((u - 0.5) * 6.0).astype(np.float32)         # positive, e^-3 .. e^3


@pytest.mark.parametrize("K", [1, 96, 4096, 70000])
def test_smooth_prepare_matches_oracle(orc, L, K):
    import torch

    m = _smooth_f32(K, K)
    if K >= 96:
        m[[3, 17, 40, 41, 60, 95]] = [np.nan, np.inf, 0.0, -2.0, 1e-45, 3.4e38]
    ref, bad_ref = orc.smooth_prepare(m)
    out = torch.empty(K, dtype=torch.int16, device="cuda")
    bad = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    L.fp4_smooth_prepare(dev(m), out, K, bad)
    assert L.fp4_get_device_status() == 0
    assert int(bad.item()) == bad_ref
    got = out.cpu().numpy().view(np.uint16)
    # NaN payloads are not part of the contract (the value is rejected anyway)
    nan_ref = (ref & 0x7FFF) > 0x7F80
    nan_got = (got & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_got, nan_ref)
    assert np.array_equal(got[~nan_ref], ref[~nan_ref])


@pytest.mark.parametrize("M,K", [(1, 64), (130, 224), (64, 4096)])
@pytest.mark.parametrize("alg", [0, 2])
@pytest.mark.parametrize("layout", [0, 1])
def test_act_quant_mxfp4_smooth_matches_oracle(orc, L, M, K, alg, layout):
    X = synth.bf16_normal(M * 7 + K, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    mb, bad = orc.smooth_prepare(_smooth_f32(K, K + 1))
    assert bad == 0
    p_ref, s_ref = orc.act_quant(orc.smooth_apply(X, mb), alg, threads=THREADS)
    op = empty_u8(M * K // 2)
    osf = empty_u8(L.fp4_sf_bytes(M, K, layout))
    L.fp4_quant_act_mxfp4_smooth(dev_bf16(X), dev_bf16(mb), op, osf, M, K, scale_alg=alg, sf_layout=layout)
    assert L.fp4_get_device_status() == 0
    assert np.array_equal(host(op)[: M * K // 2].reshape(M, K // 2), p_ref)
    s_expect = orc.sf_swizzle(s_ref) if layout == 0 else s_ref.reshape(-1)
    assert np.array_equal(host(osf)[: len(s_expect)], s_expect)


@pytest.mark.parametrize("M,K", [(3, 128), (130, 224), (64, 4096)])
def test_act_quant_mxfp8_smooth_matches_oracle(orc, L, M, K):
    X = synth.bf16_normal(M * 5 + K, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    mb, _ = orc.smooth_prepare(_smooth_f32(K, K + 2))
    c_ref, s_ref = orc.act_quant_mxfp8(orc.smooth_apply(X, mb), threads=THREADS)
    codes = empty_u8(M * K)
    osf = empty_u8(L.fp4_sf_bytes(M, K, 0))
    L.fp4_quant_act_mxfp8_smooth(dev_bf16(X), dev_bf16(mb), codes, osf, M, K, 0)
    assert L.fp4_get_device_status() == 0
    assert np.array_equal(host(codes)[: M * K].reshape(M, K), c_ref)
    s_expect = orc.sf_swizzle(s_ref)
    assert np.array_equal(host(osf)[: len(s_expect)], s_expect)


def test_act_quant_smooth_overflow_and_ties(orc, L):
    """Products that overflow bf16 (a NaN/Inf block), products that round
    at a bf16 tie, and a unit scale (identical to the plain quantizer)."""
    M, K = 4, 128
    X = synth.bf16_normal(3, synth.S_ACT, (M, K), 1.0)
    X[0, 5] = 0x7F00                                    # 1.7e38
    m = np.ones(K, np.float32)
    m[5] = 4.0                                          # 6.8e38 -> Inf
    m[64:] = 1.0078125                                  # 1 + 2^-7: products land on bf16 ties
    mb, bad = orc.smooth_prepare(m)
    assert bad == 0
    p_ref, s_ref = orc.act_quant(orc.smooth_apply(X, mb))
    op = empty_u8(M * K // 2)
    osf = empty_u8(L.fp4_sf_bytes(M, K, 1))
    L.fp4_quant_act_mxfp4_smooth(dev_bf16(X), dev_bf16(mb), op, osf, M, K, sf_layout=1)
    assert L.fp4_get_device_status() == 0
    assert np.array_equal(host(op)[: M * K // 2].reshape(M, K // 2), p_ref)
    assert np.array_equal(host(osf)[: M * K // 32].reshape(M, K // 32), s_ref)
    assert s_ref[0, 0] == 0xFF
    # unit scale: the plain quantizer's bytes
    ones, _ = orc.smooth_prepare(np.ones(K, np.float32))
    L.fp4_quant_act_mxfp4_smooth(dev_bf16(X), dev_bf16(ones), op, osf, M, K, sf_layout=1)
    p_plain, s_plain = orc.act_quant(X)
    assert np.array_equal(host(op)[: M * K // 2].reshape(M, K // 2), p_plain)
    assert np.array_equal(host(osf)[: M * K // 32].reshape(M, K // 32), s_plain)

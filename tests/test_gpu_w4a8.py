"""GPU parity of the W4A8 fallback ("W4A4 MXFP4 Quantization": MXFP8
activations with the same MXFP4 weights): the MXFP8 activation quantizer
byte for byte and the MXFP8 x MXFP4 GEMM within the GEMM bound
|out - ref| <= 2^-8 |ref| + 1e-6 sum_k |a_k b_k|, through the C ABI against
the oracle.  Operands come from the oracle (or are drawn directly), so no
oracle input comes from the CUDA path."""
import numpy as np
import pytest

import synth
from _util import THREADS, bf16_bits_host, bf16_bits_to_f64, dev, dev_bf16, empty_u8, gemm_check, host, lib

pytestmark = pytest.mark.gpu

FINITE_E4M3 = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)


@pytest.fixture(scope="module")
def L():
    return lib()


def _quant(L, X, M, K, layout):
    codes = empty_u8(M * K)
    sf = empty_u8(L.fp4_sf_bytes(M, K, layout))
    L.fp4_quant_act_mxfp8(dev_bf16(X), codes, sf, M, K, layout)
    assert L.fp4_get_device_status() == 0
    return host(codes)[: M * K].reshape(M, K), host(sf)[: L.fp4_sf_bytes(M, K, layout)]


# ---------------------------------------------------------------- quantizer
@pytest.mark.parametrize("M,K", [(1, 64), (130, 224), (257, 1024), (64, 4096)])
@pytest.mark.parametrize("layout", [0, 1])
def test_act_quant_mxfp8_matches_oracle(orc, L, M, K, layout):
    X = synth.bf16_normal(M + K, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    c_ref, s_ref = orc.act_quant_mxfp8(X, threads=THREADS)
    codes, sf = _quant(L, X, M, K, layout)
    assert np.array_equal(codes, c_ref)
    assert np.array_equal(sf, orc.sf_swizzle(s_ref) if layout == 0 else s_ref.reshape(-1))


def test_act_quant_mxfp8_special_values(orc, L):
    """Zeros and -0, infinities, NaN, bf16 subnormals, the bf16 maximum,
    saturating blocks and ties: byte-exact against the oracle."""
    M, K = 8, 128
    X = synth.bf16_normal(9, synth.S_ACT, (M, K), 1.0)
    X[0, :32] = 0x0000
    X[0, 32:64] = 0x8000
    X[1, 3] = 0x7F80
    X[1, 40] = 0xFF80
    X[2, 70] = 0x7FC0
    X[3, :32] = np.arange(1, 33, dtype=np.uint16)                  # subnormals
    X[3, 32:64] = 0x8000 | np.arange(1, 33, dtype=np.uint16)
    X[4, :32] = 0x7F7F                                              # bf16 max
    X[5, :6] = [0x3FF8, 0x3FE0, 0x3FE8, 0xBFF3, 0x3F80, 0x3F00]     # saturating block
    X[6, :4] = [0x4100, 0x40F8, 0x3800, 0x3840]                     # ties to even, half subnormal
    c_ref, s_ref = orc.act_quant_mxfp8(X)
    for layout in (0, 1):
        codes, sf = _quant(L, X, M, K, layout)
        assert np.array_equal(codes, c_ref)
        assert np.array_equal(sf, orc.sf_swizzle(s_ref) if layout == 0 else s_ref.reshape(-1))


# ---------------------------------------------------------------- GEMM
def _weight(orc, W_bits):
    g = orc.nvfp4_global_scale(W_bits)
    wp, ws = orc.nvfp4_quantize(W_bits, g, threads=THREADS)
    return orc.requant(wp, ws, g, threads=THREADS)


def _run(L, a8, sa_sw, b, sb_sw, bias, M, N, K, workspace=None):
    import torch

    out = torch.full((max(M, 1), N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bd = dev(b)
    assert bd.data_ptr() % 32 == 0
    L.fp4_gemm_w4a8(dev(a8), dev(sa_sw), bd, dev(sb_sw), None if bias is None else dev_bf16(bias), out, M, N, K,
                    workspace)
    assert L.fp4_get_device_status() == 0
    return bf16_bits_host(out)[:M]


def _check(orc, L, a8, sa, b, sb, bias, rows=None, workspace=None):
    M, N, K = a8.shape[0], b.shape[0], a8.shape[1]
    out = _run(L, a8, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), bias, M, N, K, workspace)
    ref, absum = orc.gemm_w4a8(a8, sa, b, sb, bias, rows=rows, threads=THREADS)
    sub = out if rows is None else out[rows]
    ok, ratio = gemm_check(sub, ref, absum)
    assert ok, f"max err/bound = {ratio}"
    return out


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (8, 256, 384), (33, 136, 512), (64, 384, 1024),
                                   (130, 136, 384), (257, 264, 640), (300, 512, 256)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_gemm_w4a8_recipe_operands(orc, L, M, N, K, with_bias):
    X = synth.bf16_normal(M * 3 + K, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    W = synth.bf16_normal(N * 5 + K, synth.S_WEIGHT, (N, K), 0.02)
    a8, sa = orc.act_quant_mxfp8(X, threads=THREADS)
    b, sb = _weight(orc, W)
    bias = synth.bf16_normal(N, synth.S_BIAS, (N,), 0.01) if with_bias else None
    _check(orc, L, a8, sa, b, sb, bias)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (70, 200, 384), (20, 128, 256), (256, 512, 1024)])
def test_gemm_w4a8_random_codes_nonuniform_scales(orc, L, M, N, K):
    """Every finite E4M3 byte, every FP4 code and a different scale per
    32-block on both sides pin the operand and scale layouts."""
    rng = np.random.default_rng(M + N + K + 1)
    a8 = rng.choice(FINITE_E4M3, (M, K))
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(112, 142, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(112, 142, (N, K // 32), dtype=np.uint8)
    _check(orc, L, a8, sa, b, sb, None)


def test_gemm_w4a8_one_hot_is_exact(orc, L):
    """B rows one-hot with FP4 code 1.0 under scale 2^0: out[:, n] is one
    E4M3 value times a power of two, exact in bf16."""
    rng = np.random.default_rng(4)
    M, N, K = 200, 136, 512
    a8 = rng.choice(FINITE_E4M3, (M, K))
    sa = rng.integers(115, 140, (M, K // 32), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    out = _run(L, a8, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K)
    ref, _ = orc.gemm_w4a8(a8, sa, b, sb)
    assert np.array_equal(bf16_bits_to_f64(out), ref)


def test_gemm_w4a8_wide_tiles(orc, L):
    """Enough 128 x 256 tiles to fill the GPU, checked on sampled rows."""
    M, N, K = 1024, 4864, 512
    X = synth.bf16_normal(13, synth.S_ACT, (M, K), 1.0, 0.005, 16.0)
    W = synth.bf16_normal(14, synth.S_WEIGHT, (N, K), 0.015)
    a8, sa = orc.act_quant_mxfp8(X, threads=THREADS)
    b, sb = _weight(orc, W)
    rows = np.sort(np.random.default_rng(6).choice(M, 40, replace=False))
    rows[-1] = M - 1
    _check(orc, L, a8, sa, b, sb, None, rows=rows)


@pytest.mark.parametrize("M,N,K", [(8, 1024, 8192), (64, 256, 16384)])
def test_gemm_w4a8_split_k(orc, L, M, N, K):
    """Decode-sized M with the workspace its split plan asks for; two calls
    give identical bits."""
    import torch

    need = L.fp4_gemm_w4a8_workspace_size(M, N, K)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    X = synth.bf16_normal(M + 9, synth.S_ACT, (M, K), 1.0)
    W = synth.bf16_normal(N + 9, synth.S_WEIGHT, (N, K), 0.02)
    a8, sa = orc.act_quant_mxfp8(X, threads=THREADS)
    b, sb = _weight(orc, W)
    first = _check(orc, L, a8, sa, b, sb, None, workspace=ws)
    again = _run(L, a8, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K, ws)
    assert np.array_equal(first, again)


# ---------------------------------------------------------------- full sizes
@pytest.mark.slow
def test_full_decode_and_prefill_w4a8_gemm(orc, L):
    """The benchmark's decode (14336 x 4096, M = 1 and 64, with bias) and
    prefill (2048 x 18432 x 7168) shapes, on sampled rows (all columns)."""
    rng = np.random.default_rng(8)
    w1 = synth.workload1(Ms=(1, 64))
    w2 = synth.workload2(Ms=(2048,))
    b1, sb1 = _weight(orc, w1["W"])
    for X in (w1["X"][1], w1["X"][64]):
        a8, sa = orc.act_quant_mxfp8(X, threads=THREADS)
        _check(orc, L, a8, sa, b1, sb1, w1["bias"])
    b2, sb2 = _weight(orc, w2["W"])
    a8, sa = orc.act_quant_mxfp8(w2["X"][2048], threads=THREADS)
    rows = np.sort(rng.choice(2048, 24, replace=False))
    rows[-1] = 2047
    _check(orc, L, a8, sa, b2, sb2, None, rows=rows)

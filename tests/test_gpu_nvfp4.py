"""GPU parity of the NVFP4 side path ("[SGLang] FP4 ..." sections 5-6): the
NVFP4 quantizer with swizzled scales, the scale swizzle and the NVFP4 x NVFP4
GEMM, through the C ABI against the oracle.  GEMM operands come from the
oracle's NVFP4 quantizer and swizzle (or are drawn directly), so no oracle
input comes from the CUDA path.  Quantizer outputs are compared byte for
byte; the GEMM is held to the same per-element bound as the MXFP4 GEMM:
|out - ref| <= 2^-8 |ref| + 1e-6 sum_k |a_k b_k|."""
import numpy as np
import pytest

import synth
from _util import THREADS, bf16_bits_host, dev, dev_bf16, empty_u8, gemm_check, host, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


# ---------------------------------------------------------------- scale swizzle
@pytest.mark.parametrize("rows,kb", [(1, 1), (128, 4), (130, 6), (257, 32), (300, 224), (64, 449)])
def test_sf_swizzle_matches_oracle(orc, L, rows, kb):
    rm = synth.random_bytes(rows + kb, synth.S_SCALES, rows * kb).reshape(rows, kb)
    expect = orc.sf_swizzle(rm)
    out = empty_u8(len(expect))
    L.fp4_sf_swizzle(dev(rm), out, rows, kb)
    assert L.fp4_get_device_status() == 0
    assert np.array_equal(host(out)[: len(expect)], expect)


# ---------------------------------------------------------------- quantizer
@pytest.mark.parametrize("M,K", [(1, 64), (130, 208), (257, 1024), (64, 4096)])
@pytest.mark.parametrize("layout", [0, 1])
def test_quant_nvfp4_ex_matches_oracle(orc, L, M, K, layout):
    X = synth.bf16_normal(M + K, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    g = orc.nvfp4_global_scale(X)
    p_ref, s_ref = orc.nvfp4_quantize(X, g, threads=THREADS)
    s_expect = orc.sf_swizzle(s_ref) if layout == 0 else s_ref.reshape(-1)
    assert L.fp4_sf_bytes_nvfp4(M, K, layout) == len(s_expect)
    op = empty_u8(M * K // 2)
    osf = empty_u8(len(s_expect))
    L.fp4_quant_nvfp4_ex(dev_bf16(X), g, op, osf, M, K, layout)
    assert L.fp4_get_device_status() == 0
    assert np.array_equal(host(op)[: M * K // 2].reshape(M, K // 2), p_ref)
    assert np.array_equal(host(osf)[: len(s_expect)], s_expect)


@pytest.mark.parametrize("g", [None, 0.0, 1e-30, 3e30, -0.25])
def test_quant_nvfp4_special_values(orc, L, g):
    """Blocks of zeros and -0, infinities, NaN, bf16 subnormals, values near
    the bf16 maximum and ordinary data, under several global scales
    (including 0 and a negative one): byte-exact against the oracle."""
    M, K = 6, 128
    X = synth.bf16_normal(5, synth.S_ACT, (M, K), 1.0)
    X[0, :16] = 0x0000
    X[0, 16:32] = 0x8000                       # -0
    X[1, 3] = 0x7F80                           # +inf
    X[1, 20] = 0xFF80                          # -inf
    X[2, 40] = 0x7FC0                          # NaN
    X[3, :16] = np.arange(1, 17, dtype=np.uint16)          # positive subnormals
    X[3, 16:32] = 0x8000 | np.arange(1, 17, dtype=np.uint16)
    X[4, :16] = 0x7F7F                         # bf16 max
    X[4, 16:32] = 0xFF00 | np.arange(0x60, 0x70, dtype=np.uint16)
    gv = orc.nvfp4_global_scale(X) if g is None else g
    p_ref, s_ref = orc.nvfp4_quantize(X, gv, threads=1)
    for layout in (0, 1):
        s_expect = orc.sf_swizzle(s_ref) if layout == 0 else s_ref.reshape(-1)
        op = empty_u8(M * K // 2)
        osf = empty_u8(len(s_expect))
        L.fp4_quant_nvfp4_ex(dev_bf16(X), gv, op, osf, M, K, layout)
        assert L.fp4_get_device_status() == 0
        assert np.array_equal(host(op)[: M * K // 2].reshape(M, K // 2), p_ref)
        assert np.array_equal(host(osf)[: len(s_expect)], s_expect)


# ---------------------------------------------------------------- GEMM
def _nv_operand(orc, x_bits):
    """bf16 -> NVFP4 by the oracle: (packed, row-major E4M3, swizzled E4M3, g)."""
    g = orc.nvfp4_global_scale(x_bits)
    p, s = orc.nvfp4_quantize(x_bits, g, threads=THREADS)
    return p, s, orc.sf_swizzle(s), g


def _run(L, a, sa_sw, b, sb_sw, alpha, bias, M, N, K, workspace=None):
    import torch

    out = torch.full((max(M, 1), N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_nvfp4(dev(a), dev(sa_sw), dev(b), dev(sb_sw), alpha, None if bias is None else dev_bf16(bias), out,
                     M, N, K, workspace)
    assert L.fp4_get_device_status() == 0
    return bf16_bits_host(out)[:M]


def _check(orc, L, a, sa, b, sb, alpha, bias, rows=None, workspace=None):
    M, N, K = a.shape[0], b.shape[0], 2 * a.shape[1]
    out = _run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), alpha, bias, M, N, K, workspace)
    ref, absum = orc.gemm_nvfp4(a, sa, b, sb, alpha, bias, rows=rows, threads=THREADS)
    sub = out if rows is None else out[rows]
    ok, ratio = gemm_check(sub, ref, absum)
    assert ok, f"max err/bound = {ratio}"
    return out


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (16, 256, 512), (33, 136, 384), (64, 384, 1024),
                                   (130, 136, 384), (257, 264, 640), (300, 512, 256)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_gemm_nvfp4_recipe_operands(orc, L, M, N, K, with_bias):
    X = synth.bf16_normal(M * 3 + K, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    W = synth.bf16_normal(N * 5 + K, synth.S_WEIGHT, (N, K), 0.02)
    a, sa, _, ga = _nv_operand(orc, X)
    b, sb, _, gb = _nv_operand(orc, W)
    alpha = float(np.float32(ga) * np.float32(gb))
    bias = synth.bf16_normal(N, synth.S_BIAS, (N,), 0.01) if with_bias else None
    _check(orc, L, a, sa, b, sb, alpha, bias)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (70, 200, 384), (20, 128, 256), (256, 512, 1024)])
def test_gemm_nvfp4_random_codes_every_scale(orc, L, M, N, K):
    """Every code and independent scale bytes over the whole finite,
    non-negative E4M3 range (0x00 .. 0x7E) per 16-block pin the 16-element
    scale layout: a misplaced scale changes the result far beyond the bound."""
    rng = np.random.default_rng(M + N + K)
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(0, 0x7F, (M, K // 16), dtype=np.uint8)
    sb = rng.integers(0, 0x7F, (N, K // 16), dtype=np.uint8)
    _check(orc, L, a, sa, b, sb, 0.75, None)


def test_gemm_nvfp4_one_hot_is_exact(orc, L):
    """B rows one-hot with code 1.0 under scale 1.0, alpha 1: out[:, n] is
    one A code times its E4M3 scale, exact in bf16."""
    from _util import bf16_bits_to_f64

    rng = np.random.default_rng(3)
    M, N, K = 200, 136, 512
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(0x10, 0x70, (M, K // 16), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = np.full((N, K // 16), 0x38, np.uint8)
    out = _run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), 1.0, None, M, N, K)
    ref, _ = orc.gemm_nvfp4(a, sa, b, sb, 1.0)
    assert np.array_equal(bf16_bits_to_f64(out), ref)


def test_gemm_nvfp4_wide_tiles(orc, L):
    """Enough 128 x 256 tiles to fill the GPU: the wide-tile configuration,
    checked on a sample of rows (all columns)."""
    M, N, K = 1024, 4864, 512
    X = synth.bf16_normal(11, synth.S_ACT, (M, K), 1.0, 0.005, 16.0)
    W = synth.bf16_normal(12, synth.S_WEIGHT, (N, K), 0.015)
    a, sa, _, ga = _nv_operand(orc, X)
    b, sb, _, gb = _nv_operand(orc, W)
    rows = np.sort(np.random.default_rng(5).choice(M, 40, replace=False))
    rows[-1] = M - 1
    _check(orc, L, a, sa, b, sb, float(np.float32(ga) * np.float32(gb)), None, rows=rows)


@pytest.mark.parametrize("M,N,K", [(8, 1024, 16384), (64, 256, 30720)])
def test_gemm_nvfp4_split_k(orc, L, M, N, K):
    """Decode-sized M with a workspace: the split-K plan of the MXFP4 GEMM
    (same workspace size); two calls give identical bits."""
    import torch

    need = L.fp4_gemm_workspace_size(M, N, K)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    X = synth.bf16_normal(M + 7, synth.S_ACT, (M, K), 1.0)
    W = synth.bf16_normal(N + 7, synth.S_WEIGHT, (N, K), 0.02)
    a, sa, _, ga = _nv_operand(orc, X)
    b, sb, _, gb = _nv_operand(orc, W)
    alpha = float(np.float32(ga) * np.float32(gb))
    first = _check(orc, L, a, sa, b, sb, alpha, None, workspace=ws)
    again = _run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), alpha, None, M, N, K, ws)
    assert np.array_equal(first, again)


def test_gemm_nvfp4_end_to_end_on_device(orc, L):
    """bf16 weight and activations through the library alone (NVFP4 quant
    with swizzled scales, then the GEMM) against the oracle's quantize +
    GEMM of the same bf16 tensors."""
    import torch

    M, N, K = 48, 512, 2048
    X = synth.bf16_normal(21, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    W = synth.bf16_normal(22, synth.S_WEIGHT, (N, K), 0.02)
    a, sa, _, ga = _nv_operand(orc, X)
    b, sb, _, gb = _nv_operand(orc, W)
    ap, asf = empty_u8(M * K // 2), empty_u8(L.fp4_sf_bytes_nvfp4(M, K, 0))
    bp, bsf = empty_u8(N * K // 2), empty_u8(L.fp4_sf_bytes_nvfp4(N, K, 0))
    L.fp4_quant_nvfp4_ex(dev_bf16(X), ga, ap, asf, M, K, 0)
    L.fp4_quant_nvfp4_ex(dev_bf16(W), gb, bp, bsf, N, K, 0)
    alpha = float(np.float32(ga) * np.float32(gb))
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_nvfp4(ap, asf, bp, bsf, alpha, None, out, M, N, K)
    assert L.fp4_get_device_status() == 0
    ref, absum = orc.gemm_nvfp4(a, sa, b, sb, alpha, threads=THREADS)
    ok, ratio = gemm_check(bf16_bits_host(out), ref, absum)
    assert ok, f"max err/bound = {ratio}"


# ---------------------------------------------------------------- full sizes
@pytest.mark.slow
def test_full_decode_and_prefill_nvfp4_gemm(orc, L):
    """The benchmark's decode (14336 x 4096, M = 64, with bias) and prefill
    (2048 x 18432 x 7168) shapes in the launch configurations the benchmark
    times, on sampled rows (all columns)."""
    rng = np.random.default_rng(7)
    w1 = synth.workload1(Ms=(64,))
    w2 = synth.workload2(Ms=(2048,))
    for W, X, bias in ((w1["W"], w1["X"][64], w1["bias"]), (w2["W"], w2["X"][2048], None)):
        M = X.shape[0]
        a, sa, _, ga = _nv_operand(orc, X)
        b, sb, _, gb = _nv_operand(orc, W)
        rows = np.sort(rng.choice(M, min(M, 24), replace=False))
        rows[-1] = M - 1
        _check(orc, L, a, sa, b, sb, float(np.float32(ga) * np.float32(gb)), bias, rows=rows)

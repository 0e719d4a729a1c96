"""GPU parity of the CTA-pair GEMM (256 x 256 output tiles on two SMs with
256-row MMAs) against the float64 oracle, through the C ABI.  The library
takes this path for dense MXFP4 problems with M >= 256 whose 128 x 256 tiles
would fill the GPU; the shapes below do, and include ragged M and N tails
(a pair whose second CTA holds no rows, a last tile with 8 valid columns),
K with an odd number of 256-element slabs (one-slab stages) and K a multiple
of 512 (two-slab stages).  Tolerance as for every GEMM:
|out - ref| <= 2^-8 |ref| + 1e-6 sum_k |a_k b_k|."""
import numpy as np
import pytest

import synth
from _util import THREADS, bf16_bits_host, bf16_bits_to_f64, dev, dev_bf16, gemm_check, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


def _takes_pair_path(M, N):
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return M >= 256 and N >= 256 and (-(-M // 128)) * (-(-N // 256)) >= min(148, sms)


def _run(L, a, sa_sw, b, sb_sw, bias, M, N, K):
    import torch

    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_mxfp4(dev(a), dev(sa_sw), dev(b), dev(sb_sw), None if bias is None else dev_bf16(bias), out, M, N, K)
    assert L.fp4_get_device_status() == 0
    return bf16_bits_host(out)


@pytest.mark.parametrize("M,N,K", [(1280, 3840, 512), (1300, 3848, 640), (2048, 2560, 1536), (520, 9472, 256),
                                   (4096, 2560, 1024)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_pair_gemm_recipe_operands(orc, L, M, N, K, with_bias):
    assert _takes_pair_path(M, N)
    X = synth.bf16_normal(M + 7 * K, synth.S_ACT, (M, K), 1.0, 0.005, 16.0)
    W = synth.bf16_normal(N + 11 * K, synth.S_WEIGHT, (N, K), 0.015)
    a, sa = orc.act_quant(X, threads=THREADS)
    g = orc.nvfp4_global_scale(W)
    wp, ws = orc.nvfp4_quantize(W, g, threads=THREADS)
    b, sb = orc.requant(wp, ws, g, threads=THREADS)
    bias = synth.bf16_normal(N + 1, synth.S_BIAS, (N,), 0.01) if with_bias else None
    out = _run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), bias, M, N, K)
    # every row of the last 256-row tile, rows of each CTA half, and a spread sample
    rng = np.random.default_rng(M + N)
    rows = np.unique(np.concatenate([np.arange(max(0, M - 300), M), rng.choice(M, 64, replace=False),
                                     [0, 127, 128, 255, 256]]))
    rows = rows[rows < M]
    ref, absum = orc.gemm(a, sa, b, sb, bias, rows=rows, threads=THREADS)
    ok, ratio = gemm_check(out[rows], ref, absum)
    assert ok, f"max err/bound = {ratio}"


@pytest.mark.parametrize("M,N,K", [(1024, 4864, 1024), (768, 6400, 384)])
def test_pair_gemm_random_codes_nonuniform_scales(orc, L, M, N, K):
    """Every code and a different scale per 32-block: a scale written to the
    wrong TMEM lane or column changes the result far beyond the tolerance."""
    assert _takes_pair_path(M, N)
    rng = np.random.default_rng(M + N + K)
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(112, 142, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(112, 142, (N, K // 32), dtype=np.uint8)
    out = _run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K)
    rows = np.unique(np.concatenate([np.arange(0, 260), np.arange(M - 260, M), rng.choice(M, 64, replace=False)]))
    ref, absum = orc.gemm(a, sa, b, sb, rows=rows, threads=THREADS)
    ok, ratio = gemm_check(out[rows], ref, absum)
    assert ok, f"max err/bound = {ratio}"


def test_pair_gemm_long_k(orc, L):
    """K = 16384: 32 stages a tile, and the scale tiles prefetched into L2
    for the next tile (128 KB) go out as several requests."""
    M, N, K = 1024, 4864, 16384
    assert _takes_pair_path(M, N)
    rng = np.random.default_rng(7)
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(116, 138, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(116, 138, (N, K // 32), dtype=np.uint8)
    out = _run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1], rng.choice(M, 48, replace=False)]))
    ref, absum = orc.gemm(a, sa, b, sb, rows=rows, threads=THREADS)
    ok, ratio = gemm_check(out[rows], ref, absum)
    assert ok, f"max err/bound = {ratio}"


def test_pair_gemm_one_hot_is_exact(orc, L):
    """B rows one-hot with code 1.0 under scale 2^0: out[:, n] = A[:, sel[n]]
    exactly, for every row of both CTAs of every pair and every column."""
    rng = np.random.default_rng(3)
    M, N, K = 1536, 3584, 768
    assert _takes_pair_path(M, N)
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(100, 150, (M, K // 32), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    out = _run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K)
    # the selected column of dequantized A, from the oracle's (pinned) codecs
    A = np.empty((M, K))
    lo, hi = a & 0xF, a >> 4
    codes_a = np.stack([lo, hi], axis=-1).reshape(M, K)
    val = np.array([orc.e2m1_value(c) for c in range(16)])
    A = val[codes_a] * np.repeat(2.0 ** (sa.astype(np.float64) - 127), 32, axis=1)
    assert np.array_equal(bf16_bits_to_f64(out), A[:, sel])


def test_pair_gemm_nan_scale_poisons_its_row_and_column(orc, L):
    """An E8M0 NaN scale (0xFF) on one A row block and one B row block: only
    that output row and that output column become NaN."""
    rng = np.random.default_rng(4)
    M, N, K = 1280, 3840, 512
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(120, 134, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(120, 134, (N, K // 32), dtype=np.uint8)
    r_bad, c_bad = 777, 2999
    sa[r_bad, 5] = 0xFF
    sb[c_bad, 9] = 0xFF
    out = bf16_bits_to_f64(_run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K))
    nan = np.isnan(out)
    assert nan[r_bad].all() and nan[:, c_bad].all()
    nan[r_bad] = False
    nan[:, c_bad] = False
    assert not nan.any()


def test_pair_gemm_is_deterministic(orc, L):
    rng = np.random.default_rng(5)
    M, N, K = 1024, 4864, 1024
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(118, 136, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(118, 136, (N, K // 32), dtype=np.uint8)
    first = _run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K)
    for _ in range(2):
        assert np.array_equal(_run(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K), first)

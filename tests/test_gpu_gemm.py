"""GPU parity of the W4A4 GEMM (dense and grouped) against the float64
oracle, through the C ABI.  Operands come from the oracle's quantizers, so
no input of the oracle comes from the CUDA path.  Tolerance (per element):
|out - ref| <= 2^-8 |ref| + 1e-6 sum_k |a_k b_k|."""
import numpy as np
import pytest

import synth
from _util import THREADS, bf16_bits_host, bf16_bits_to_f64, dev, dev_bf16, empty_u8, gemm_check, host, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


def _mx_operand(orc, x_bits):
    """bf16 -> MXFP4 by the oracle: (packed, row-major SF, swizzled SF)."""
    p, s = orc.act_quant(x_bits, threads=THREADS)
    return p, s, orc.sf_swizzle(s)


def _weight_operand(orc, W_bits):
    g = orc.nvfp4_global_scale(W_bits)
    wp, ws = orc.nvfp4_quantize(W_bits, g, threads=THREADS)
    p, s = orc.requant(wp, ws, g, threads=THREADS)
    return p, s, orc.sf_swizzle(s)


def _run_gemm(L, a, sa_sw, b, sb_sw, bias, M, N, K):
    import torch

    out = torch.full((max(M, 1), N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_mxfp4(dev(a), dev(sa_sw), dev(b), dev(sb_sw), None if bias is None else dev_bf16(bias), out,
                     M, N, K)
    assert L.fp4_get_device_status() == 0
    return bf16_bits_host(out)[:M]


def _check(orc, L, a, sa, sa_sw, b, sb, sb_sw, bias, rows=None, cols=None):
    M, N, K = a.shape[0], b.shape[0], 2 * a.shape[1]
    out = _run_gemm(L, a, sa_sw, b, sb_sw, bias, M, N, K)
    ref, absum = orc.gemm(a, sa, b, sb, bias, rows=rows, cols=cols, threads=THREADS)
    sub = out if rows is None and cols is None else out[np.ix_(
        np.arange(M) if rows is None else rows, np.arange(N) if cols is None else cols)]
    ok, ratio = gemm_check(sub, ref, absum)
    assert ok, f"max err/bound = {ratio}"
    return ratio


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (16, 256, 512), (130, 136, 384), (128, 128, 128),
                                   (257, 264, 640), (64, 384, 1024), (300, 512, 256), (5, 1024, 2048)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_gemm_recipe_operands(orc, L, M, N, K, with_bias):
    X = synth.bf16_normal(M * 3 + K, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    W = synth.bf16_normal(N * 5 + K, synth.S_WEIGHT, (N, K), 0.02)
    a, sa, sa_sw = _mx_operand(orc, X)
    b, sb, sb_sw = _weight_operand(orc, W)
    bias = synth.bf16_normal(N, synth.S_BIAS, (N,), 0.01) if with_bias else None
    _check(orc, L, a, sa, sa_sw, b, sb, sb_sw, bias)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (70, 200, 384), (256, 512, 1024)])
def test_gemm_random_codes_nonuniform_scales(orc, L, M, N, K):
    """Every code and a different scale per 32-block pin the scale-factor
    layout: a misplaced scale changes the result far beyond the tolerance."""
    rng = np.random.default_rng(M + N + K)
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(112, 142, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(112, 142, (N, K // 32), dtype=np.uint8)
    _check(orc, L, a, sa, orc.sf_swizzle(sa), b, sb, orc.sf_swizzle(sb), None)


def test_gemm_one_hot_is_exact(orc, L):
    """B rows one-hot with code 1.0 under scale 2^0: out[:, n] = A[:, sel[n]],
    an E2M1 value times a power of two, exact in bf16."""
    rng = np.random.default_rng(1)
    M, N, K = 200, 136, 512
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(100, 150, (M, K // 32), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    out = _run_gemm(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K)
    ref, _ = orc.gemm(a, sa, b, sb)
    from _util import bf16_bits_to_f64

    assert np.array_equal(bf16_bits_to_f64(out), ref)


def test_gemm_cancellation(orc, L):
    """Rows that cancel to (nearly) zero: the absolute term of the bound is
    what the result is held to."""
    rng = np.random.default_rng(2)
    M, N, K = 128, 128, 1024
    half = rng.integers(0, 256, (M, K // 4), dtype=np.uint8)
    a = np.concatenate([half, half ^ 0x88], axis=1)              # second half = negated first half
    sa = np.full((M, K // 32), 127, np.uint8)
    b = rng.integers(0, 256, (N, K // 4), dtype=np.uint8)
    b = np.concatenate([b, b], axis=1)
    sb = rng.integers(120, 134, (N, K // 64), dtype=np.uint8)
    sb = np.concatenate([sb, sb], axis=1)
    _check(orc, L, a, sa, orc.sf_swizzle(sa), b, sb, orc.sf_swizzle(sb), None)


# ---------------------------------------------------------------- grouped
def _run_grouped(L, a, sa_grouped, b_all, sb_all, bias_all, offsets, N, K):
    import torch

    total = a.shape[0]
    E = len(offsets) - 1
    out = torch.full((max(total, 1), N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_mxfp4_grouped(dev(a), dev(sa_grouped), dev(b_all), dev(sb_all),
                             None if bias_all is None else dev_bf16(bias_all), out, dev(offsets), E, total, N, K)
    assert L.fp4_get_device_status() == 0
    return bf16_bits_host(out)[:total]


def _grouped_sf(orc, s_rowmajor, offsets, K, total):
    from nvfp4_mxfp4_w4a4_gb300 import fp4lin

    buf = np.zeros(fp4lin.fp4_sf_bytes_grouped(total, len(offsets) - 1, K), np.uint8)
    pos = 0
    for e in range(len(offsets) - 1):
        rows = s_rowmajor[offsets[e]:offsets[e + 1]]
        if len(rows):
            sw = orc.sf_swizzle(rows)
            buf[pos:pos + len(sw)] = sw
            pos += len(sw)
    return buf


def _grouped_case(orc, L, counts, N, K, with_bias, seed):
    E = len(counts)
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    total = int(offsets[-1])
    X = synth.bf16_normal(seed, synth.S_ACT, (total, K), 1.0, 0.01, 16.0)
    a, sa = orc.act_quant(X, threads=THREADS)
    bs, sbs, sbs_sw = [], [], []
    for e in range(E):
        W = synth.bf16_normal(seed * 100 + e, synth.S_WEIGHT, (N, K), 0.02)
        p, s, sw = _weight_operand(orc, W)
        bs.append(p)
        sbs.append(s)
        sbs_sw.append(sw)
    bias = synth.bf16_normal(seed, synth.S_BIAS, (E, N), 0.01) if with_bias else None
    out = _run_grouped(L, a, _grouped_sf(orc, sa, offsets, K, total), np.stack(bs), np.concatenate(sbs_sw),
                       bias, offsets, N, K)
    ref, absum = orc.gemm_grouped(a, sa, np.stack(bs), np.stack(sbs), bias, offsets, threads=THREADS)
    ok, ratio = gemm_check(out, ref, absum)
    assert ok, f"max err/bound = {ratio}"


@pytest.mark.parametrize("counts,N,K", [([3, 0, 130, 1, 200], 136, 256), ([128, 128], 256, 512),
                                        ([0, 5, 0], 64, 128), ([40] * 8, 512, 384)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_grouped_gemm(orc, L, counts, N, K, with_bias):
    _grouped_case(orc, L, counts, N, K, with_bias, seed=len(counts) + N)


@pytest.mark.parametrize("counts,N,K,with_bias", [
    ([300, 0, 1, 257, 1000, 129, 640, 0, 77, 512], 2048, 512, True),
    ([256, 130, 513, 0, 700, 1200, 300], 1544, 384, False),
    # K = 1024: two stages a tile with two store boxes in flight per epilogue warp
    ([513, 0, 255, 384, 1, 900, 256], 2304, 1024, True),
    # K = 1280: three-stage ring, the tile's last stage half full
    ([640, 300, 0, 129, 1000], 2048, 1280, False),
])
def test_grouped_gemm_on_cta_pairs(orc, L, counts, N, K, with_bias):
    """Grouped problems large enough for the CTA-pair path (256 x 256 tiles
    of one expert on two SMs): experts with an odd number of 128-row tiles
    (the second CTA of the last pair tile lies past the expert), a one-row
    expert, empty experts, row counts that end inside a 32-row store box
    (stored row by row), a ragged last column tile, one- and two-slab
    stages, the short-K configuration and a partial last stage; every row
    compared."""
    E = len(counts)
    m_tiles = (sum(counts) + E * 127) // 128
    assert N >= 256 and m_tiles * (-(-N // 256)) >= 148, "shape must take the pair path"
    _grouped_case(orc, L, counts, N, K, with_bias, seed=E * 1000 + K)


# ---------------------------------------------------------------- full sizes
@pytest.mark.slow
def test_full_decode_workload_gemm(orc, L):
    w = synth.workload1()
    b, sb, sb_sw = _weight_operand(orc, w["W"])
    for M, X in w["X"].items():
        a, sa, sa_sw = _mx_operand(orc, X)
        _check(orc, L, a, sa, sa_sw, b, sb, sb_sw, w["bias"])


@pytest.mark.slow
def test_full_prefill_workload_gemm(orc, L):
    w = synth.workload2()
    b, sb, sb_sw = _weight_operand(orc, w["W"])
    rng = np.random.default_rng(0)
    for M, X in w["X"].items():
        a, sa, sa_sw = _mx_operand(orc, X)
        rows = np.sort(rng.choice(M, 48, replace=False))
        rows[-1] = M - 1
        _check(orc, L, a, sa, sa_sw, b, sb, sb_sw, None, rows=rows)


@pytest.mark.slow
def test_full_moe_workload_gemm(orc, L):
    w = synth.workload3()
    offsets = w["row_offsets"]
    E = len(offsets) - 1
    rng = np.random.default_rng(1)
    for A, Ws, N, K in ((w["A_gu"], w["W_gu"], 2048, 4096), (w["A_down"], w["W_down"], 4096, 1024)):
        a, sa = orc.act_quant(A, threads=THREADS)
        bs, sbs, sws = [], [], []
        for e in range(E):
            p, s, sw = _weight_operand(orc, Ws[e])
            bs.append(p)
            sbs.append(s)
            sws.append(sw)
        b_all = np.stack(bs)
        total = A.shape[0]
        out = _run_grouped(L, a, _grouped_sf(orc, sa, offsets, K, total), b_all, np.concatenate(sws), None,
                           offsets, N, K)
        rows = np.sort(rng.choice(total, 64, replace=False))
        ref, absum = orc.gemm_grouped(a, sa, b_all, np.stack(sbs), None, offsets, rows=rows, threads=THREADS)
        ok, ratio = gemm_check(out[rows], ref, absum)
        assert ok, f"max err/bound = {ratio}"


# ---------------------------------------------------------------- end to end
def test_end_to_end_tiny_workload(orc, L):
    """CUDA requant + CUDA act-quant + CUDA GEMM on the tiny workload against
    the oracle chain on the same NVFP4 / bf16 inputs."""
    import torch

    w = synth.workload0()
    g = orc.nvfp4_global_scale(w["W"])
    wp, ws = orc.nvfp4_quantize(w["W"], g)
    N, K = w["W"].shape
    M = w["X"].shape[0]
    bq = empty_u8(N * K // 2)
    bs = empty_u8(L.fp4_sf_bytes(N, K))
    L.fp4_requant_nvfp4_to_mxfp4(dev(wp), dev(ws), g, bq, bs, N, K)
    aq = empty_u8(M * K // 2)
    as_ = empty_u8(L.fp4_sf_bytes(M, K))
    L.fp4_quant_act_mxfp4(dev_bf16(w["X"]), aq, as_, M, K)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_mxfp4(aq, as_, bq, bs, None, out, M, N, K)
    rb, rbs = orc.requant(wp, ws, g)
    ra, ras = orc.act_quant(w["X"])
    ref, absum = orc.gemm(ra, ras, rb, rbs)
    ok, ratio = gemm_check(bf16_bits_host(out), ref, absum)
    assert ok, ratio


def test_gemm_nan_and_tiny_scales(orc, L):
    """E8M0 0xFF is NaN: a NaN scale in one block of A row 3 makes output row
    3 NaN, one in B row 5 makes column 5 NaN.  Scales near the bottom of the
    range (2^-111 for a whole A row, 2^-112 for one B block) give tiny
    products that stay normal in float32.  Elsewhere the usual bound holds."""
    rng = np.random.default_rng(11)
    M, N, K = 16, 136, 256
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(120, 134, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(120, 134, (N, K // 32), dtype=np.uint8)
    sa[3, 2] = 0xFF
    sb[5, 7] = 0xFF
    sa[7, :] = 0x10
    sb[9, 1] = 0x0F
    out = _run_gemm(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, M, N, K)
    ref, absum = orc.gemm(a, sa, b, sb)
    from _util import bf16_bits_to_f64

    got = bf16_bits_to_f64(out)
    nan_ref = np.isnan(ref)
    assert nan_ref[3, :].all() and nan_ref[:, 5].all() and nan_ref.sum() == N + M - 1
    assert np.array_equal(np.isnan(got), nan_ref)
    keep = ~nan_ref
    ok, ratio = gemm_check(out[keep], ref[keep], absum[keep])
    assert ok, f"max err/bound = {ratio}"


# ---------------------------------------------------------------- one token (M = 1)
@pytest.mark.parametrize("N,K", [(8, 128), (136, 1152), (1024, 4096), (264, 7168), (64, 32768), (16, 33024)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_one_token_random_codes_nonuniform_scales(orc, L, N, K, with_bias):
    """One token (the split-K swapped path): every FP4 code on both sides and
    a different scale per 32-block, K up to 33024, within the GEMM bound."""
    rng = np.random.default_rng(N + K + with_bias)
    a = rng.integers(0, 256, (1, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(112, 142, (1, K // 32), dtype=np.uint8)
    sb = rng.integers(112, 142, (N, K // 32), dtype=np.uint8)
    bias = synth.bf16_normal(N + K, synth.S_BIAS, (N,), 0.5) if with_bias else None
    out = _run_gemm(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), bias, 1, N, K)
    ref, absum = orc.gemm(a, sa, b, sb, bias, threads=THREADS)
    ok, ratio = gemm_check(out, ref, absum)
    assert ok, f"max err/bound = {ratio}"


def test_one_token_one_hot_is_exact(orc, L):
    """B rows one-hot with code 1.0 under scale 2^0: out[0, n] is one A value
    times its power-of-two scale, exact in bf16."""
    rng = np.random.default_rng(21)
    N, K = 264, 4096
    a = rng.integers(0, 256, (1, K // 2), dtype=np.uint8)
    sa = rng.integers(115, 140, (1, K // 32), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    out = _run_gemm(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, 1, N, K)
    ref, _ = orc.gemm(a, sa, b, sb)
    assert np.array_equal(bf16_bits_to_f64(out), ref)


def test_one_token_nan_and_tiny_scales(orc, L):
    """M = 1 with a NaN scale in one B block (that output is NaN), a NaN
    scale in A (every output NaN) and scales near the bottom of the range."""
    rng = np.random.default_rng(12)
    N, K = 136, 1024
    a = rng.integers(0, 256, (1, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(120, 134, (1, K // 32), dtype=np.uint8)
    sb = rng.integers(120, 134, (N, K // 32), dtype=np.uint8)
    sb[5, 7] = 0xFF
    sb[9, :] = 0x10
    sb[11, 3] = 0x01
    out = _run_gemm(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, 1, N, K)
    ref, absum = orc.gemm(a, sa, b, sb)
    got = bf16_bits_to_f64(out)
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.isnan(ref[0, 5]) and np.isnan(ref).sum() == 1
    keep = ~np.isnan(ref)
    ok, ratio = gemm_check(out[keep], ref[keep], absum[keep])
    assert ok, f"max err/bound = {ratio}"
    sa[0, 2] = 0xFF
    out = _run_gemm(L, a, orc.sf_swizzle(sa), b, orc.sf_swizzle(sb), None, 1, N, K)
    assert np.isnan(bf16_bits_to_f64(out)).all()

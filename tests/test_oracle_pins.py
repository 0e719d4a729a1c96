"""Pins for the CPU oracle: each test checks the oracle against something
other than itself -- hand-derived worked examples (tests/golden), library
codecs (torch's float8 types), closed forms, invariants and brute force.

A plausible slip in the oracle (a swapped nibble order, a k/16 vs k/32 scale
index, a wrong exponent offset, a transposed GEMM operand, a dropped bias)
fails at least one test here.
"""
import math
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN

# ------------------------------------------------------------------ helpers


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _e2m1_table():
    """code -> value from the hand-written fixture (independent of the oracle)."""
    t = {}
    for code, val in _golden_lines("e2m1_values.txt"):
        t[int(code, 16)] = float(val)
    return t


def _hex_bytes(s):
    return np.frombuffer(bytes.fromhex(s), dtype=np.uint8).copy()


def _unpack(packed):
    """packed u8 [..., K/2] -> 4-bit codes [..., K]; element 2j in the low nibble."""
    lo = packed & 0xF
    hi = packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], -1)


def _torch_e4m3(bytes_u8):
    return torch.from_numpy(np.asarray(bytes_u8, np.uint8)).view(torch.float8_e4m3fn).float().numpy()


# ------------------------------------------------------------------ codecs


def test_e2m1_decode_matches_hand_table(orc):
    table = _e2m1_table()
    assert len(table) == 16
    for code, val in table.items():
        got = orc.e2m1_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    assert max(table.values()) == 6.0          # largest finite E2M1 value is 6


def test_e4m3_decode_matches_torch(orc):
    ref = _torch_e4m3(np.arange(256))
    got = np.array([orc.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.nanmax(got) == 448.0


def test_e8m0_decode_matches_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = np.array([orc.e8m0_value(b) for b in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


def test_bf16_decode_matches_torch(orc):
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x0001, 0x0080, 0x7F7F, 0x7F80, 0x4049, 0x3E4D],
                    dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([orc.bf16_value(int(b)) for b in bits])
    assert np.array_equal(got, ref)


def test_e4m3_encode_matches_torch(orc):
    # every E4M3 magnitude, every midpoint between neighbours, and points just off them
    vals = np.array(sorted({abs(v) for v in _torch_e4m3(np.arange(0x7F))}), dtype=np.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                          np.nextafter(mids.astype(np.float32), np.float32(1e9))])
    pts = pts.astype(np.float32)
    rng = np.random.default_rng(7)
    pts = np.concatenate([pts, rng.uniform(0, 448, 5000).astype(np.float32),
                          np.exp(rng.uniform(np.log(1e-4), np.log(448), 5000)).astype(np.float32)])
    ref = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(p)) for p in pts], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # saturation beyond the largest finite value (0x7E = 448)
    for t in (449.0, 464.0, 1000.0, 1e30):
        assert orc.e4m3_encode(t) == 0x7E


def test_e2m1_encode_matches_per_binade_rint(orc):
    """Round to nearest, ties to even code, written as np.rint on each binade:
    the E2M1 grid is uniform with step 0.5 on [0,2], 1 on [2,4], 2 on [4,6];
    the even grid index is the even code."""
    grid = np.unique(np.concatenate([np.arange(0, 8.0001, 1 / 64.0), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]]))
    qs = np.concatenate([grid, -grid])

    def expect(q):
        m = abs(q)
        if m <= 2:
            code = int(np.rint(m * 2))                   # codes 0..4 at step 0.5
        elif m <= 4:
            code = 4 + int(np.rint(m - 2))               # codes 4..6 at step 1
        else:
            code = 6 + int(min(np.rint((m - 4) / 2), 1))  # codes 6..7 at step 2, saturating
        return (8 if math.copysign(1, q) < 0 else 0) | code

    for q in qs:
        assert orc.e2m1_encode(float(q)) == expect(float(q)), q
    assert orc.e2m1_encode(-0.0) == 0x8
    # saturation holds for every magnitude above 6, however large
    for q in (6.0000001, 1e3, 1e17, 1e27, 3.4e38, float("inf")):
        assert orc.e2m1_encode(q) == 0x7 and orc.e2m1_encode(-q) == 0xF, q


# ------------------------------------------------------ shared exponent rule


def _amax_samples():
    rng = np.random.default_rng(11)
    a = list(np.exp(rng.uniform(np.log(1e-38), np.log(1e38), 4000)))
    for k in range(-120, 120, 7):
        for m in (1.0, 1.8125, np.nextafter(1.8125, 2), 1.9999999, 1.5, np.nextafter(2.0, 0)):
            a.append(m * 2.0 ** k)
    return [float(np.float32(x)) for x in a if x > 0]


def test_ocp_exponent_closed_form(orc):
    # OCP MX: amax / 2^e lies in [4, 8) (E2M1's largest exponent is 2)
    for amax in _amax_samples():
        e = orc.mx_shared_exp(amax, orc.SCALE_OCP)
        r = amax / 2.0 ** e
        if e == -127:                                    # clamped at E8M0's smallest scale
            assert r < 8.0 and math.floor(math.log2(amax)) - 2 <= -127, (amax, e)
        else:
            assert 4.0 <= r < 8.0, (amax, e)
    assert orc.mx_shared_exp(0.0, orc.SCALE_OCP) == -127
    assert orc.mx_shared_exp(2.0 ** -140, orc.SCALE_OCP) == -127      # clamped
    assert orc.mx_shared_exp(float(np.finfo(np.float32).max), orc.SCALE_OCP) == 125


def test_uos_exponent_reading(orc):
    # UOS (Qmax = 7.25), reading: smallest e with amax <= 7.25 * 2^e
    for amax in _amax_samples():
        e = orc.mx_shared_exp(amax, orc.SCALE_UOS)
        assert amax <= 7.25 * 2.0 ** e, (amax, e)
        assert e == -127 or amax > 7.25 * 2.0 ** (e - 1), (amax, e)
    assert orc.mx_shared_exp(7.25, orc.SCALE_UOS) == 0       # the boundary itself keeps the smaller e
    assert orc.mx_shared_exp(float(np.nextafter(np.float32(7.25), np.float32(8))), orc.SCALE_UOS) == 1


# ------------------------------------------------------ worked examples


@pytest.mark.parametrize("row", _golden_lines("requant_examples.txt"), ids=lambda r: r[0])
def test_requant_worked_examples(orc, row):
    name, g_hex, codes, scales, ocp_sf, ocp_codes, uos_sf, uos_codes = row
    g = float(np.frombuffer(bytes.fromhex(g_hex)[::-1], dtype=np.float32)[0])
    packed = _hex_bytes(codes).reshape(1, 16)
    sc = _hex_bytes(scales).reshape(1, 2)
    for alg, sf, out in ((orc.SCALE_OCP, ocp_sf, ocp_codes), (orc.SCALE_UOS, uos_sf, uos_codes)):
        p, s = orc.requant(packed, sc, g, alg)
        assert s[0, 0] == int(sf, 16), (name, alg)
        assert p.tobytes().hex() == out, (name, alg)


@pytest.mark.parametrize("row", _golden_lines("act_quant_examples.txt"), ids=lambda r: r[0])
def test_act_quant_worked_examples(orc, row):
    name, xs, ocp_sf, ocp_codes, uos_sf, uos_codes = row
    x = np.array([int(h, 16) for h in xs.split(",")], np.uint16).reshape(1, 32)
    for alg, sf, out in ((orc.SCALE_OCP, ocp_sf, ocp_codes), (orc.SCALE_UOS, uos_sf, uos_codes)):
        p, s = orc.act_quant(x, alg)
        assert s[0, 0] == int(sf, 16), (name, alg)
        assert p.tobytes().hex() == out, (name, alg)


# ------------------------------------------------------ NVFP4 decode


def test_nvfp4_dequant_matches_float32_products(orc):
    """v = fp32((E2M1(c) * E4M3(s)) * g): checked with numpy float32 products
    over the hand E2M1 table and torch's E4M3 decode, per-16 scale index."""
    rng = np.random.default_rng(3)
    N, K = 5, 96
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = rng.integers(0, 0x7F, (N, K // 16), dtype=np.uint8)       # finite, positive
    scale[0, 1] |= 0x80                                                  # one negative scale
    table = _e2m1_table()
    codes = _unpack(packed)
    cval = np.vectorize(lambda c: table[int(c)])(codes).astype(np.float32)
    sval = _torch_e4m3(scale).astype(np.float32)
    for g in (1.0, 0.0001234, 3.7e-3, 2.0 ** -20):
        g32 = np.float32(g)
        expect = (cval * np.repeat(sval, 16, axis=1)) * g32
        got = orc.nvfp4_dequant(packed, scale, float(g32))
        assert np.array_equal(got.view(np.uint32), expect.astype(np.float32).view(np.uint32))



def _decode_f32_indep(packed, scale, g32):
    """NVFP4 decode with numpy float32 products over the hand E2M1 table and
    torch's E4M3 decode (one float32 rounding of the product with g)."""
    table = _e2m1_table()
    cval = np.vectorize(lambda c: table[int(c)])(_unpack(packed)).astype(np.float32)
    sval = _torch_e4m3(scale).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        return (cval * np.repeat(sval, 16, axis=1)) * np.float32(g32)


def test_requant_subnormal_products_worked_example(orc):
    """A block whose decoded values are float32 subnormals (the products
    S * g lie below 2^-126): code 4 (2.0) under scale 0.5625 and
    g = 2796202 * 2^-149 decodes to RN(3145727.25 * 2^-149) = 3145727 * 2^-149;
    its amax is below 2^-125, so e = -127 (byte 0x00) and q = 3145727 * 2^-22
    is just below 0.75: code 1 (0.5), not the tie 0.75 that doubling the
    rounded value of code 2 would give."""
    g = float(np.float32(np.ldexp(2796202.0, -149)))
    packed = np.zeros((1, 16), np.uint8)
    packed[0, 0] = 0x04
    scale = np.full((1, 2), 0x31, np.uint8)
    p, s = orc.requant(packed, scale, g)
    assert p[0, 0] == 0x01 and not p[0, 1:].any() and s[0, 0] == 0x00


def test_requant_subnormal_products_decode_then_quantize(orc):
    """Tiny global scales: requant equals the (brute-force pinned) block
    quantizer applied to an independent float32 decode, subnormals included."""
    rng = np.random.default_rng(31)
    N, K = 8, 128
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = rng.integers(0, 0x7F, (N, K // 16), dtype=np.uint8)
    for G in (2796202, 1234567, 7777777, 3, 99991):
        g32 = np.float32(np.ldexp(float(G), -149))
        v = _decode_f32_indep(packed, scale, g32)
        for alg in (orc.SCALE_OCP, orc.SCALE_UOS):
            p, s = orc.requant(packed, scale, float(g32), alg)
            for r in range(N):
                for b in range(K // 32):
                    bp, bs = orc.mx_quantize_block(v[r, 32 * b:32 * b + 32], alg)
                    assert np.array_equal(p[r, 16 * b:16 * b + 16], bp.reshape(-1)) and s[r, b] == bs, (G, alg, r, b)


def test_requant_bf16_is_act_quant_of_bf16_decode(orc):
    """The bf16-intermediate requant equals the activation quantizer (pinned
    above) applied to the decoded values rounded to bf16 by torch."""
    rng = np.random.default_rng(21)
    N, K = 6, 256
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = rng.integers(0, 256, (N, K // 16), dtype=np.uint8)         # negative and NaN scales too
    for g in (1.0, 0.0037, -0.25, 2.0 ** -20, 3.0e38, 1.0e-38, 2.0 ** -133):
        g32 = np.float32(g)
        v = _decode_f32_indep(packed, scale, g32)
        xb = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        for alg in (orc.SCALE_OCP, orc.SCALE_UOS):
            want_p, want_s = orc.act_quant(xb, alg)
            got_p, got_s = orc.requant(packed, scale, float(g32), alg, bf16=True)
            assert np.array_equal(got_p, want_p) and np.array_equal(got_s, want_s), (g, alg)


def test_requant_bf16_equals_float32_path_for_power_of_two_g(orc):
    """E2M1 x E4M3 products carry at most 6 significant bits, so with g a
    power of two (and the products normal) every decoded value is a bf16
    value and both intermediates give the same bytes."""
    rng = np.random.default_rng(22)
    N, K = 6, 256
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = rng.integers(0, 0x7F, (N, K // 16), dtype=np.uint8)
    scale[:, ::3] |= 0x80
    for k in (-100, -3, 0, 5, 100):
        for alg in (orc.SCALE_OCP, orc.SCALE_UOS):
            a = orc.requant(packed, scale, 2.0 ** k, alg)
            b = orc.requant(packed, scale, 2.0 ** k, alg, bf16=True)
            assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), (k, alg)


def test_requant_bf16_worked_example(orc):
    """Where bf16 rounding crosses an E2M1 threshold: codes 2 (1.0) and 6
    (4.0) under scale 1.0 with g = 0.875 (1 - 2^-20).  Both paths take
    amax < 3.5, e = -1 (byte 126); element 0 has q = 1.75 (1 - 2^-20) in
    float32, code 3 (1.5), but its bf16 value 0.875 gives the tie q = 1.75,
    which goes to the even code 4 (2.0); element 1 saturates to code 7."""
    g = float(np.float32(0.875 * (1 - 2.0 ** -20)))
    packed = np.zeros((1, 16), np.uint8)
    packed[0, 0] = 0x62
    scale = np.full((1, 2), 0x38, np.uint8)
    p32, s32 = orc.requant(packed, scale, g)
    p16, s16 = orc.requant(packed, scale, g, bf16=True)
    assert (p32[0, 0], s32[0, 0]) == (0x73, 126) and (p16[0, 0], s16[0, 0]) == (0x74, 126)

# ------------------------------------------------------ invariants


def _rand_roundtrip_case(orc, rng, g_log2, k):
    """An NVFP4 block with both half-scales times g equal to 2^k and largest
    magnitude code 6 or 7: requant must return the same codes bit for bit."""
    s_log2 = k - g_log2
    s_byte = (s_log2 + 7) << 3                                          # E4M3 power of two (normal)
    codes = rng.integers(0, 16, 32)
    codes[rng.integers(0, 32)] = rng.choice([6, 7, 14, 15])
    codes = np.where((codes & 7) == 7, codes - 1, codes) if rng.random() < 0.5 else codes
    if not np.any((codes & 7) >= 6):
        codes[0] = 6
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8).reshape(1, 16)
    scale = np.array([[s_byte, s_byte]], np.uint8)
    return packed, scale, float(2.0 ** g_log2)


def test_roundtrip_bit_identical(orc):
    rng = np.random.default_rng(5)
    n = 0
    for g_log2 in (-12, -3, 0, 4):
        for k in range(g_log2 - 6, g_log2 + 8):
            s_log2 = k - g_log2
            if not -6 <= s_log2 <= 8:
                continue
            for _ in range(8):
                packed, scale, g = _rand_roundtrip_case(orc, rng, g_log2, k)
                for alg in (orc.SCALE_OCP, orc.SCALE_UOS):
                    p, s = orc.requant(packed, scale, g, alg)
                    assert np.array_equal(p, packed) and s[0, 0] == k + 127, (g_log2, k, alg)
                n += 1
    assert n > 100


def test_emitted_codes_are_nearest(orc):
    """Brute force over all 16 codes: each emitted element is a nearest
    representable value under its block scale (ties to the even code)."""
    rng = np.random.default_rng(9)
    table = _e2m1_table()
    grid = np.array([table[c] for c in range(16)])
    for trial in range(300):
        v = (rng.standard_normal(32) * 10.0 ** rng.uniform(-6, 6)).astype(np.float32)
        if trial % 3 == 0:
            v[rng.integers(0, 32, 4)] *= 16
        for alg in (orc.SCALE_OCP, orc.SCALE_UOS):
            packed, sf = orc.mx_quantize_block(v, alg)
            scale = 2.0 ** (sf - 127)
            codes = _unpack(packed.reshape(1, 16))[0]
            for x, c in zip(v.astype(np.float64), codes):
                d = np.abs(grid * scale - x)
                best = d.min()
                assert d[c] == best, (x, c)
                ties = np.nonzero(d == best)[0]
                if len({abs(grid[t]) for t in ties}) > 1:     # a real tie between magnitudes
                    assert (c & 7) % 2 == 0


def test_requant_error_bound(orc):
    """|dq_mx - v| is at most half the local E2M1 step times 2^e, or the
    saturation error for |q| > 6."""
    rng = np.random.default_rng(13)
    N, K = 16, 256
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = rng.integers(0x20, 0x7E, (N, K // 16), dtype=np.uint8)
    g = 0.0037
    v = orc.nvfp4_dequant(packed, scale, g).astype(np.float64)
    p, s = orc.requant(packed, scale, g)
    table = _e2m1_table()
    dq = np.vectorize(lambda c: table[int(c)])(_unpack(p)) * np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
    e = np.repeat(s.astype(np.float64) - 127, 32, axis=1)
    q = np.abs(v) / 2.0 ** e
    half_step = np.where(q <= 2, 0.25, np.where(q <= 4, 0.5, 1.0)) * 2.0 ** e
    sat = np.maximum(q - 6.0, 0) * 2.0 ** e
    assert np.all(np.abs(dq - v) <= np.maximum(half_step, sat))


# ------------------------------------------------------ GEMM


def _dequant_indep(packed, sf_rowmajor):
    table = _e2m1_table()
    codes = _unpack(packed)
    vals = np.vectorize(lambda c: table[int(c)])(codes)
    return vals * np.repeat(2.0 ** (sf_rowmajor.astype(np.float64) - 127), 32, axis=1)


def test_gemm_matches_numpy_matmul(orc):
    rng = np.random.default_rng(17)
    M, N, K = 7, 13, 160
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(110, 140, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(110, 140, (N, K // 32), dtype=np.uint8)
    bias = torch.randn(N).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    A = _dequant_indep(a, sa)
    B = _dequant_indep(b, sb)
    bias_f = torch.from_numpy(bias.view(np.int16)).view(torch.bfloat16).double().numpy()
    expect = A @ B.T + bias_f
    ref, absum = orc.gemm(a, sa, b, sb, bias)
    assert np.allclose(ref, expect, rtol=1e-12, atol=1e-12 * np.abs(A) @ np.abs(B).T + 1e-300)
    assert np.allclose(absum, np.abs(A) @ np.abs(B).T, rtol=1e-12)
    # a row/column subset gives the same entries
    rows, cols = np.array([5, 0, 3]), np.array([12, 1])
    r2, _ = orc.gemm(a, sa, b, sb, bias, rows=rows, cols=cols)
    assert np.array_equal(r2, ref[np.ix_(rows, cols)])


def test_gemm_one_hot_selects_columns(orc):
    """B rows one-hot with code 1.0 under scale 2^0: out[:, n] = A[:, sel[n]] exactly."""
    rng = np.random.default_rng(19)
    M, N, K = 6, 10, 128
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(120, 135, (M, K // 32), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    ref, _ = orc.gemm(a, sa, b, sb)
    A = _dequant_indep(a, sa)
    assert np.array_equal(ref, A[:, sel])


# ------------------------------------------------------ grouped (MoE) GEMM

# Experts of a grouped problem ("Efficiently Serving NVFP4 Models ...",
# "Native FP4 matmul": MoE experts on MXFP4): rows [off[e], off[e+1]) of the
# activations run against expert e's weight and bias.  The offsets cover an
# empty first expert, a one-row expert, an empty expert in the middle, an
# expert ending on the 128-row boundary, one of exactly 128 rows ending on the
# next, another one-row expert and a ragged last one.
_GROUPED_OFFSETS = np.array([0, 0, 1, 1, 128, 256, 257, 300], np.int32)


def _grouped_case():
    rng = np.random.default_rng(71)
    off = _GROUPED_OFFSETS
    E, total, N, K = len(off) - 1, int(off[-1]), 8, 64
    a = rng.integers(0, 256, (total, K // 2), dtype=np.uint8)
    sa = rng.integers(118, 136, (total, K // 32), dtype=np.uint8)
    b = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    sb = rng.integers(118, 136, (E, N, K // 32), dtype=np.uint8)
    # a distinct bias per expert (bf16 bits of expert-dependent values)
    bias_f = (np.arange(E)[:, None] * 4.0 + np.arange(N)[None, :] / 8.0 + 1.0).astype(np.float32)
    bias = torch.from_numpy(bias_f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return off, a, sa, b, sb, bias


def _grouped_expected(off, a, sa, b, sb, bias):
    """Per expert, a numpy float64 matmul of operands decoded by the E2M1
    fixture and the E8M0 definition, plus that expert's bias (torch's bf16)."""
    A = _dequant_indep(a, sa)
    out = np.full((A.shape[0], b.shape[1]), np.nan)
    for e in range(len(off) - 1):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        Be = _dequant_indep(b[e], sb[e])
        be = torch.from_numpy(bias[e].view(np.int16)).view(torch.bfloat16).double().numpy()
        out[r0:r1] = A[r0:r1] @ Be.T + be
    return out


def _grouped_matches(fn, case):
    off, a, sa, b, sb, bias = case
    expect = _grouped_expected(*case)
    ref, _ = fn(a, sa, b, sb, bias, off)
    ok = not np.isnan(expect).any() and np.allclose(ref, expect, rtol=1e-12, atol=1e-9)
    # a row subset that starts on expert boundaries gives the same entries
    rows = np.array([0, 127, 128, 255, 256, 299])
    r2, _ = fn(a, sa, b, sb, bias, off, rows=rows)
    return ok and np.allclose(r2, expect[rows], rtol=1e-12, atol=1e-9)


def test_gemm_grouped_matches_per_expert_matmul(orc):
    assert _grouped_matches(orc.gemm_grouped, _grouped_case())


def test_gemm_grouped_pin_catches_planted_mistakes(orc):
    """Two plausible slips in the row-to-expert mapping, planted in copies of
    the oracle's grouped GEMM built on its (separately pinned) dense GEMM:
    rows on an offset assigned with searchsorted side="left", and the bias of
    the previous expert.  The pin above must reject both."""
    case = _grouped_case()

    def planted(side, bias_shift):
        def fn(a, sa, b, sb, bias, off, rows=None):
            total = int(off[-1])
            rows = np.arange(total) if rows is None else np.asarray(rows)
            expert_of = np.searchsorted(off, rows, side=side) - 1
            ref = np.full((len(rows), b.shape[1]), np.nan)
            for e in range(len(off) - 1):
                sel = np.nonzero(expert_of == e)[0]
                if len(sel):
                    ref[sel], _ = orc.gemm(a, sa, b[e], sb[e], bias[e - bias_shift], rows=rows[sel])
            return ref, None
        return fn

    assert _grouped_matches(planted("right", 0), case)   # the planting harness itself is faithful
    assert not _grouped_matches(planted("left", 0), case)
    assert not _grouped_matches(planted("right", 1), case)


# ------------------------------------------------------ DualScale weights

# "W4A4 MXFP4 Quantization", "mxfp4_dualscale -- DualScale Offline Mode",
# "Checkpoint tensor layout": FP4 values, fine E8M0 per 32 K-elements, coarse
# float32 per 512 K-elements; value = E2M1 x 2^(fine - 127) x coarse.


def _dual_dequant_indep(packed, fine, coarse):
    """E2M1 fixture x 2^(fine - 127) x coarse, each factor expanded by numpy."""
    table = _e2m1_table()
    vals = np.vectorize(lambda c: table[int(c)])(_unpack(packed))
    return (vals * np.repeat(2.0 ** (fine.astype(np.float64) - 127), 32, axis=1)
            * np.repeat(coarse.astype(np.float64), 512, axis=1))


def _dual_operands(rng, rows, K):
    packed = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    fine = rng.integers(112, 140, (rows, K // 32), dtype=np.uint8)
    coarse = np.exp(rng.normal(-3.0, 1.5, (rows, K // 512))).astype(np.float32)
    return packed, fine, coarse


def test_dual_dequant_matches_numpy(orc):
    rng = np.random.default_rng(81)
    packed, fine, coarse = _dual_operands(rng, 5, 1536)
    assert np.array_equal(orc.dual_dequant(packed, fine, coarse), _dual_dequant_indep(packed, fine, coarse))


def test_dual_quantize_properties(orc):
    """The online dual-level quantizer (stated reading) against what it must
    satisfy: the group's largest element lands on E2M1's largest value with a
    unit fine scale, 6 x coarse recovers the group's largest magnitude, every
    code is the nearest E2M1 value of w / coarse / 2^e (ties to the even code,
    saturating), the fine exponent obeys the OCP closed form, NaN / Inf poison
    only their own block, an all-zero group gets coarse 1, and the
    reconstruction error stays within half a grid step."""
    import synth

    N, K = 10, 1536
    W = synth.bf16_normal(83, synth.S_WEIGHT, (N, K), 0.02, 0.01, 8.0)
    W[0, 512:1024] = 0                                  # an all-zero group
    W[1, 40] = 0x7FC0                                   # NaN
    W[2, 700] = 0xFF80                                  # -Inf
    packed, fine, coarse = orc.dual_quantize(W)
    w = torch.from_numpy(W.view(np.int16)).view(torch.bfloat16).float().numpy()
    codes = _unpack(packed)
    table = _e2m1_table()
    grid = np.array([table[c] for c in range(16)])
    for r in range(N):
        for g in range(K // 512):
            seg = w[r, 512 * g:512 * (g + 1)]
            fin = np.isfinite(seg)
            amax = np.abs(seg[fin]).max()
            c = coarse[r, g]
            if amax == 0:
                assert c == 1.0
            else:
                assert abs(6.0 * float(c) - amax) <= 2.0 ** -22 * amax
                kmax = 512 * g + int(np.argmax(np.where(fin, np.abs(seg), -1)))
                b0 = kmax // 32 * 32
                if np.all(np.isfinite(w[r, b0:b0 + 32])):       # (a NaN / Inf block is all zero instead)
                    assert fine[r, kmax // 32] == 127 and codes[r, kmax] & 7 == 7
            for b in range(16):
                k0 = 512 * g + 32 * b
                blk = w[r, k0:k0 + 32]
                if not np.all(np.isfinite(blk)):
                    assert fine[r, k0 // 32] == 0xFF and not codes[r, k0:k0 + 32].any()
                    continue
                y = (blk / c).astype(np.float32)                   # float32 division, as the reading states
                e = int(fine[r, k0 // 32]) - 127
                ay = float(np.abs(y).max())
                if ay == 0:
                    assert e == -127
                else:
                    assert 4.0 <= ay / 2.0 ** e < 8.0
                q = y.astype(np.float64) / 2.0 ** e
                for i in range(32):
                    d = np.abs(grid - q[i])
                    d[np.abs(grid) < 0] = np.inf
                    best = np.min(np.abs(np.abs(grid[:8]) - min(abs(q[i]), 6.0)))
                    got = codes[r, k0 + i]
                    assert abs(abs(grid[got]) - min(abs(q[i]), 6.0)) == best
                    if best > 0 and np.sum(np.abs(np.abs(grid[:8]) - min(abs(q[i]), 6.0)) == best) > 1:
                        assert got & 1 == 0                         # a tie goes to the even code
                    if q[i] != 0:
                        assert (got >> 3) == (q[i] < 0)
    # reconstruction error: half a grid step of the scaled grid, or the saturation at 6
    dq = orc.dual_dequant(packed, fine, coarse)
    ok = np.isfinite(w)
    for r in range(N):
        for k in range(K):
            if not ok[r, k] or fine[r, k // 32] == 0xFF:
                continue
            s = 2.0 ** (int(fine[r, k // 32]) - 127) * float(coarse[r, k // 512])
            qa = abs(w[r, k]) / s
            half = (0.25 if qa <= 2 else 0.5 if qa <= 4 else 1.0) * s
            assert abs(dq[r, k] - w[r, k]) <= max(half, (qa - 6.0) * s) + 2.0 ** -20 * abs(w[r, k])


def test_gemm_dual_matches_numpy(orc):
    rng = np.random.default_rng(85)
    M, N, K = 6, 9, 2048
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(112, 140, (M, K // 32), dtype=np.uint8)
    b, fine, coarse = _dual_operands(rng, N, K)
    bias = torch.randn(N).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    A = _dequant_indep(a, sa)
    B = _dual_dequant_indep(b, fine, coarse)
    bias_f = torch.from_numpy(bias.view(np.int16)).view(torch.bfloat16).double().numpy()
    ref, absum = orc.gemm_dual(a, sa, b, fine, coarse, bias)
    prod_abs = np.abs(A) @ np.abs(B).T
    assert np.allclose(ref, A @ B.T + bias_f, rtol=1e-12, atol=1e-12 * prod_abs + 1e-300)
    assert np.allclose(absum, prod_abs, rtol=1e-12)
    rows, cols = np.array([4, 1]), np.array([8, 0, 3])
    r2, _ = orc.gemm_dual(a, sa, b, fine, coarse, bias, rows=rows, cols=cols)
    assert np.array_equal(r2, ref[np.ix_(rows, cols)])
    # two plausible slips, each in a copy of the definition, must fail this pin:
    # the coarse scale indexed per 1024 elements, the fine scale per 64
    table = _e2m1_table()
    vals = np.vectorize(lambda c: table[int(c)])(_unpack(b))
    wrong_coarse = vals * np.repeat(2.0 ** (fine.astype(np.float64) - 127), 32, axis=1) * \
        np.repeat(coarse.astype(np.float64), 1024, axis=1)[:, :K]
    wrong_fine = vals * np.repeat(2.0 ** (fine.astype(np.float64) - 127), 64, axis=1)[:, :K] * \
        np.repeat(coarse.astype(np.float64), 512, axis=1)
    for Bw in (wrong_coarse, wrong_fine):
        assert not np.allclose(A @ Bw.T + bias_f, ref, rtol=1e-6, atol=1e-9)


def test_gemm_dual_unit_coarse_equals_mx_gemm(orc):
    """With every coarse scale 1 a DualScale weight is an MXFP4 weight: the
    two GEMMs agree bit for bit."""
    rng = np.random.default_rng(87)
    M, N, K = 5, 7, 1536
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(112, 140, (M, K // 32), dtype=np.uint8)
    b, fine, _ = _dual_operands(rng, N, K)
    one = np.ones((N, K // 512), np.float32)
    r1, s1 = orc.gemm_dual(a, sa, b, fine, one)
    r2, s2 = orc.gemm(a, sa, b, fine)
    assert np.array_equal(r1, r2) and np.array_equal(s1, s2)


def test_gemm_dual_one_hot_selects_scaled_columns(orc):
    """B rows one-hot with code 1.0 under fine scale 2^0 and a power-of-two
    coarse scale per group: out[:, n] = A[:, sel[n]] x coarse[n, sel[n] / 512]
    exactly."""
    rng = np.random.default_rng(89)
    M, N, K = 6, 10, 1024
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(120, 135, (M, K // 32), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    fine = np.full((N, K // 32), 127, np.uint8)
    coarse = (2.0 ** rng.integers(-6, 6, (N, K // 512))).astype(np.float32)
    ref, _ = orc.gemm_dual(a, sa, b, fine, coarse)
    A = _dequant_indep(a, sa)
    assert np.array_equal(ref, A[:, sel] * coarse[np.arange(N), sel // 512].astype(np.float64))


# ------------------------------------------------------ smooth pre-scale


def test_bf16_encode_matches_torch(orc):
    rng = np.random.default_rng(61)
    vals = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.exp(rng.uniform(-40, 40, 3000)).astype(np.float32),
        # exact ties: bf16 values plus half an ulp
        (torch.randn(500).to(torch.bfloat16).float().numpy().view(np.uint32) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 3.4e38, -3.4e38, 1e-45, np.inf, -np.inf, 3.3895314e38], np.float32),
    ])
    got = np.array([orc.bf16_encode(float(v)) for v in vals], np.uint16)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    assert orc.bf16_encode(float("nan")) & 0x7FC0 == 0x7FC0


def test_smooth_prepare_rejects_what_the_page_rejects(orc):
    """NaN, Inf, non-positive values and values that overflow or underflow to
    zero in bf16 are rejected; the rest convert to bf16 as torch does."""
    good = np.array([1.0, 0.5, 3.0, 1e-30, 2.5e38, 7.1234], np.float32)
    out, bad = orc.smooth_prepare(good)
    assert bad == 0
    assert np.array_equal(out, torch.from_numpy(good).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    for v in (np.nan, np.inf, -np.inf, 0.0, -0.0, -1.0, 1e-45, 3.4e38):
        _, bad = orc.smooth_prepare(np.array([1.0, v, 2.0], np.float32))
        assert bad == 1, v


def test_smooth_apply_matches_torch_bf16_multiply(orc):
    rng = np.random.default_rng(67)
    M, K = 7, 96
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32) * 3).to(torch.bfloat16)
    m = torch.from_numpy(np.exp(rng.uniform(-3, 3, K)).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    mb = m.view(torch.int16).numpy().view(np.uint16)
    got = orc.smooth_apply(xb, mb)
    ref = (x * m).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------ W4A8: MXFP8 activations


@pytest.mark.parametrize("row", _golden_lines("act_quant_mxfp8_examples.txt"), ids=lambda r: r[0])
def test_act_quant_mxfp8_worked_examples(orc, row):
    name, xs, sf, codes = row
    x = np.array([int(h, 16) for h in xs.split(",")], np.uint16).reshape(1, 32)
    c, s = orc.act_quant_mxfp8(x)
    assert s[0, 0] == int(sf, 16), name
    assert c.tobytes().hex() == codes, name


def test_mx8_exponent_closed_form(orc):
    """OCP rule with E4M3 elements: amax / 2^e in [256, 512) for every
    unclamped amax; clamps at 2^-127 and 2^127; zero -> -127."""
    rng = np.random.default_rng(43)
    for amax in np.exp(rng.uniform(-80, 80, 2000)):
        e = orc.mx8_shared_exp(float(amax))
        assert 256.0 <= amax / 2.0 ** e < 512.0
    assert orc.mx8_shared_exp(0.0) == -127
    assert orc.mx8_shared_exp(2.0 ** -200) == -127
    assert orc.mx8_shared_exp(2.0 ** 200) == 127


def test_act_quant_mxfp8_against_torch_and_brute_force(orc):
    """Elements in range match torch's float8_e4m3fn rounding of x / 2^e;
    those beyond 448 saturate; every element is the nearest finite E4M3
    value (ties to the even code) by brute force over all 254 codes."""
    rng = np.random.default_rng(47)
    M, K = 24, 256
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32) * np.exp(rng.uniform(-20, 20, (M, 1)))
                         .astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    c, s = orc.act_quant_mxfp8(bits)
    xv = x.double().numpy().reshape(M, K // 32, 32)
    amax = np.abs(xv).max(-1)
    e = np.floor(np.log2(amax)) - 8
    assert np.array_equal(s.astype(np.int64) - 127, e.astype(np.int64))
    q = (xv / 2.0 ** e[..., None]).reshape(M, K)
    inrange = np.abs(q) <= 448
    t = torch.from_numpy(q.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(c[inrange], t[inrange])
    assert np.all((c[~inrange] & 0x7F) == 0x7E)
    finite = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)
    vals = _torch_e4m3(finite).astype(np.float64)
    got = _torch_e4m3(c).astype(np.float64)
    for i in range(0, M * K, 97):
        qi = float(q.flat[i])
        d = np.abs(vals - qi)
        best = d.min()
        assert abs(got.flat[i] - qi) == best
        ties = finite[d == best]
        if len(ties) > 1:
            assert c.flat[i] & 1 == 0            # the even code


def test_gemm_w4a8_matches_numpy_matmul(orc):
    rng = np.random.default_rng(53)
    M, N, K = 6, 11, 160
    finite = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)
    a8 = rng.choice(finite, (M, K))
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(110, 140, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(110, 140, (N, K // 32), dtype=np.uint8)
    bias = torch.randn(N).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bias_f = torch.from_numpy(bias.view(np.int16)).view(torch.bfloat16).double().numpy()
    A = _torch_e4m3(a8).astype(np.float64) * np.repeat(2.0 ** (sa.astype(np.float64) - 127), 32, axis=1)
    B = _dequant_indep(b, sb)
    ref, absum = orc.gemm_w4a8(a8, sa, b, sb, bias)
    prod_abs = np.abs(A) @ np.abs(B).T
    assert np.allclose(ref, A @ B.T + bias_f, rtol=1e-12, atol=1e-12 * prod_abs + 1e-300)
    assert np.allclose(absum, prod_abs, rtol=1e-12)
    rows, cols = np.array([5, 2]), np.array([0, 9, 3])
    r2, _ = orc.gemm_w4a8(a8, sa, b, sb, bias, rows=rows, cols=cols)
    assert np.array_equal(r2, ref[np.ix_(rows, cols)])


def test_gemm_w4a8_one_hot_selects_columns(orc):
    """B rows one-hot with code 1.0 under scale 2^0: out[:, n] = A[:, sel[n]] exactly."""
    rng = np.random.default_rng(59)
    M, N, K = 5, 9, 128
    finite = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)
    a8 = rng.choice(finite, (M, K))
    sa = rng.integers(120, 135, (M, K // 32), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    ref, _ = orc.gemm_w4a8(a8, sa, b, sb)
    A = _torch_e4m3(a8).astype(np.float64) * np.repeat(2.0 ** (sa.astype(np.float64) - 127), 32, axis=1)
    assert np.array_equal(ref, A[:, sel])


# ------------------------------------------------------ NVFP4 x NVFP4 GEMM


def _nv_scaled_indep(packed, s_rowmajor):
    """codes x E4M3 scales per 16 elements, decoded by the E2M1 fixture and torch."""
    table = _e2m1_table()
    vals = np.vectorize(lambda c: table[int(c)])(_unpack(packed))
    return vals * np.repeat(_torch_e4m3(s_rowmajor).astype(np.float64), 16, axis=1)


def test_gemm_nvfp4_matches_numpy_matmul(orc):
    """Random codes and every finite E4M3 scale byte (both signs): the oracle is
    alpha * (scaled A) @ (scaled B)^T + bias, decoded independently."""
    rng = np.random.default_rng(23)
    M, N, K = 5, 11, 192
    finite = np.array([x for x in range(256) if (x & 0x7F) != 0x7F], np.uint8)
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.choice(finite, (M, K // 16))
    sb = rng.choice(finite, (N, K // 16))
    bias = torch.randn(N).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bias_f = torch.from_numpy(bias.view(np.int16)).view(torch.bfloat16).double().numpy()
    alpha = 0.3711
    A = _nv_scaled_indep(a, sa)
    B = _nv_scaled_indep(b, sb)
    prod_abs = np.abs(A) @ np.abs(B).T
    ref, absum = orc.gemm_nvfp4(a, sa, b, sb, alpha, bias)
    assert np.allclose(ref, alpha * (A @ B.T) + bias_f, rtol=1e-12, atol=1e-12 * alpha * prod_abs + 1e-300)
    assert np.allclose(absum, alpha * prod_abs, rtol=1e-12)
    rows, cols = np.array([4, 1]), np.array([0, 10, 7])
    r2, _ = orc.gemm_nvfp4(a, sa, b, sb, alpha, bias, rows=rows, cols=cols)
    assert np.array_equal(r2, ref[np.ix_(rows, cols)])


def test_gemm_nvfp4_power_of_two_scales_equal_mx_gemm(orc):
    """When both 16-element scales of every 32-block are the same power of two
    2^j, an NVFP4 operand is the MXFP4 operand with E8M0 byte j + 127 and the
    same codes: with alpha = 1 the two GEMMs agree bit for bit."""
    rng = np.random.default_rng(29)
    M, N, K = 6, 9, 256
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    ja = rng.integers(-6, 9, (M, K // 32))
    jb = rng.integers(-6, 9, (N, K // 32))
    # E4M3 of 2^j (normal range): exponent field j + 7, mantissa 0
    nva = np.repeat(((ja + 7) << 3).astype(np.uint8), 2, axis=1)
    nvb = np.repeat(((jb + 7) << 3).astype(np.uint8), 2, axis=1)
    assert np.array_equal(_torch_e4m3(nva[:, ::2]), 2.0 ** ja)
    ref_nv, abs_nv = orc.gemm_nvfp4(a, nva, b, nvb, 1.0)
    ref_mx, abs_mx = orc.gemm(a, (ja + 127).astype(np.uint8), b, (jb + 127).astype(np.uint8))
    assert np.array_equal(ref_nv, ref_mx)
    assert np.array_equal(abs_nv, abs_mx)


def test_gemm_nvfp4_one_hot_selects_columns(orc):
    """B rows one-hot with code 1.0 under scale 1.0: out[:, n] = alpha * scaled A[:, sel[n]] exactly."""
    rng = np.random.default_rng(31)
    M, N, K = 4, 12, 128
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(0x20, 0x60, (M, K // 16), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = np.full((N, K // 16), 0x38, np.uint8)   # E4M3 1.0
    ref, _ = orc.gemm_nvfp4(a, sa, b, sb, 0.5)
    assert np.array_equal(ref, 0.5 * _nv_scaled_indep(a, sa)[:, sel])
    # the same through the (separately pinned) NVFP4 decode with g = 1
    dq = orc.nvfp4_dequant(a, sa, 1.0).astype(np.float64)
    assert np.array_equal(ref, 0.5 * dq[:, sel])


# ------------------------------------------------------ SF layout


def test_sf_swizzle_hand_offsets(orc):
    rows = _golden_lines("sf_swizzle_offsets.txt")
    assert orc.sf_swizzled_bytes(200, 6) == 2048
    for r, c, off in rows:
        assert orc.sf_swizzled_offset(int(r), int(c), 6) == int(off)


def test_sf_swizzle_is_injective_and_pads_zero(orc):
    for rows, kb in ((200, 6), (128, 4), (1, 1), (300, 224)):
        rm = np.arange(rows * kb, dtype=np.int64).reshape(rows, kb)
        offs = {orc.sf_swizzled_offset(r, c, kb) for r in range(rows) for c in range(kb)}
        assert len(offs) == rows * kb
        assert max(offs) < orc.sf_swizzled_bytes(rows, kb)
    rm = (np.arange(200 * 6) % 251 + 1).astype(np.uint8).reshape(200, 6)
    sw = orc.sf_swizzle(rm)
    assert np.count_nonzero(sw) == 200 * 6


# ------------------------------------------------------ NVFP4 producer


def test_nvfp4_quantize_nan_propagates(orc):
    """A NaN element makes its block's scale NaN (0x7F) and the block's codes
    signed zeros (the zero-or-NaN denominator rule); other blocks are
    untouched; the global scale of a tensor holding a NaN is NaN."""
    rng = np.random.default_rng(41)
    x = torch.from_numpy(rng.standard_normal((2, 64)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16).copy()
    g = orc.nvfp4_global_scale(bits)
    p0, s0 = orc.nvfp4_quantize(bits, g)
    bits[1, 37] = 0x7FC0                      # NaN in block 2 of row 1
    assert math.isnan(orc.nvfp4_global_scale(bits))
    p1, s1 = orc.nvfp4_quantize(bits, g)
    assert s1[1, 2] == 0x7F
    codes = _unpack(p1)[1, 32:48]
    signs = (bits[1, 32:48] >> 15).astype(np.uint8) << 3
    assert np.array_equal(codes, signs)
    mask = np.ones_like(s0, bool)
    mask[1, 2] = False
    assert np.array_equal(s1[mask], s0[mask])
    keep = np.ones((2, 64), bool)
    keep[1, 32:48] = False
    assert np.array_equal(_unpack(p1)[keep], _unpack(p0)[keep])


def test_nvfp4_quantize_against_float32_recipe(orc):
    """Block scale = torch's E4M3 rounding of fp32(bamax / fp32(6 g)); codes
    are nearest E2M1 values of fp32(x / fp32(scale * g)); dequantization error
    within half a grid step."""
    rng = np.random.default_rng(23)
    N, K = 9, 128
    x = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32) * 0.02).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    xf = x.float().numpy()
    g = orc.nvfp4_global_scale(bits)
    assert np.float32(g) == np.float32(np.abs(xf).max()) / np.float32(2688.0)
    p, s = orc.nvfp4_quantize(bits, g)
    bamax = np.abs(xf).reshape(N, K // 16, 16).max(-1).astype(np.float32)
    t = bamax / (np.float32(6.0) * np.float32(g))
    s_ref = torch.from_numpy(t.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(s, s_ref)
    den = (_torch_e4m3(s).astype(np.float32) * np.float32(g)).astype(np.float32)
    q = (xf.reshape(N, K // 16, 16) / den[..., None]).astype(np.float32).reshape(N, K)
    table = _e2m1_table()
    grid = np.array([table[c] for c in range(8)])
    codes = _unpack(p)
    dq = np.vectorize(lambda c: table[int(c)])(codes)
    err = np.abs(dq - q)
    nearest = np.min(np.abs(grid[None, None, :] - np.abs(q)[..., None]), axis=-1)
    assert np.all(err <= nearest + 1e-12)

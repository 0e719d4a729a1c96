"""GPU parity of the quantizers against the CPU oracle: bit-exact codes and
scale bytes, through the C ABI, on small ragged shapes, edge values and the
full sizes of the decode / prefill / MoE / layer-stream workloads."""
import numpy as np
import pytest

import synth
from _util import THREADS, bf16_bits_host, dev, dev_bf16, empty_u8, host, lib

pytestmark = pytest.mark.gpu

OCP, UOS = 0, 2
SWZ, ROW = 0, 1


@pytest.fixture(scope="module")
def L():
    return lib()


def _kernel_requant(L, packed, scale, g, alg, layout, bf16=False):
    N, half = packed.shape
    K = 2 * half
    dp, ds = dev(packed), dev(scale)
    op = empty_u8(N * K // 2)
    osf = empty_u8(L.fp4_sf_bytes(N, K, layout))
    L.fp4_requant_nvfp4_to_mxfp4(dp, ds, g, op, osf, N, K, scale_alg=alg, sf_layout=layout, bf16_intermediate=bf16)
    assert L.fp4_get_device_status() == 0
    return host(op)[: N * K // 2].reshape(N, K // 2), host(osf)[: L.fp4_sf_bytes(N, K, layout)]


def _check_requant(orc, L, packed, scale, g, alg=OCP, layout=SWZ, bf16=False):
    kp, ks = _kernel_requant(L, packed, scale, g, alg, layout, bf16)
    rp, rs = orc.requant(packed, scale, g, alg, threads=THREADS, bf16=bf16)
    assert np.array_equal(kp, rp), f"codes differ at {np.argwhere(kp != rp)[:5]}"
    expect_sf = orc.sf_swizzle(rs) if layout == SWZ else rs.reshape(-1)
    assert np.array_equal(ks, expect_sf), f"scales differ at {np.argwhere(ks != expect_sf)[:5]}"


def _random_nvfp4(rng, N, K, scale_lo=0, scale_hi=256):
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = rng.integers(scale_lo, scale_hi, (N, K // 16), dtype=np.uint8)
    return packed, scale


@pytest.mark.parametrize("N,K", [(1, 32), (5, 96), (130, 64), (256, 512), (300, 224), (129, 1056)])
@pytest.mark.parametrize("alg", [OCP, UOS])
@pytest.mark.parametrize("layout", [SWZ, ROW])
def test_requant_random_bytes(orc, L, N, K, alg, layout):
    rng = np.random.default_rng(N * 7919 + K)
    packed, scale = _random_nvfp4(rng, N, K)          # every code and every scale byte incl. NaN / negative
    for g in (1.0, 0.0037, 2.0 ** -20, -0.25):
        _check_requant(orc, L, packed, scale, float(np.float32(g)), alg, layout)


def test_requant_special_global_scales(orc, L):
    rng = np.random.default_rng(3)
    packed, scale = _random_nvfp4(rng, 64, 256, 0, 0x7F)
    for g in (0.0, -0.0, float("inf"), float("nan"), 3.0e38, 1.0e-38, 1.0e-45):
        _check_requant(orc, L, packed, scale, g)


def test_requant_tiny_workload_recipe(orc, L):
    w = synth.workload0()
    g = orc.nvfp4_global_scale(w["W"])
    packed, scale = orc.nvfp4_quantize(w["W"], g)
    for alg in (OCP, UOS):
        for layout in (SWZ, ROW):
            _check_requant(orc, L, packed, scale, g, alg, layout)


@pytest.mark.parametrize("N,K", [(1, 128), (5, 256), (130, 1024), (257, 384), (64, 4096)])
@pytest.mark.parametrize("alg", [OCP, UOS])
@pytest.mark.parametrize("layout", [SWZ, ROW])
def test_requant_flat_shapes(orc, L, N, K, alg, layout):
    # K % 128 == 0 with aligned buffers: the flattened-block kernel
    rng = np.random.default_rng(N * 131 + K)
    packed, scale = _random_nvfp4(rng, N, K)
    for g in (1.0, 0.0037, -0.25):
        _check_requant(orc, L, packed, scale, float(np.float32(g)), alg, layout)


@pytest.mark.parametrize("alg", [OCP, UOS])
def test_requant_flat_several_items_per_warp(orc, L, alg):
    """A tensor with more 128-block warp items than the GPU has resident
    warps, so warps walk two and more items through both register buffers;
    random bytes mix warp items with and without negative scales (the two
    sign paths) and a ragged last item; positive and negative g."""
    N, K = 9000, 4224
    rng = np.random.default_rng(4224)
    packed, scale = _random_nvfp4(rng, N, K)
    # rows 0..2999: positive scale bytes only (no sign changes unless g < 0)
    scale[:3000] &= 0x7F
    for g in (0.0123, -0.5):
        _check_requant(orc, L, packed, scale, float(np.float32(g)), alg, SWZ)
    _check_requant(orc, L, packed, scale, float(np.float32(0.0123)), alg, ROW)


def test_requant_16_byte_aligned_buffers(orc, L):
    # codes only 16-byte aligned: the row kernel takes the K % 128 == 0 shape
    import torch

    N, K = 131, 512
    rng = np.random.default_rng(77)
    packed, scale = _random_nvfp4(rng, N, K)
    src = torch.zeros(N * K // 2 + 16, dtype=torch.uint8, device="cuda")
    src[16:] = dev(packed.reshape(-1))
    dst = torch.full((N * K // 2 + 16,), 0xA5, dtype=torch.uint8, device="cuda")
    osf = empty_u8(L.fp4_sf_bytes(N, K, SWZ))
    g = float(np.float32(0.0123))
    L.fp4_requant_nvfp4_to_mxfp4(src[16:], dev(scale), g, dst[16:], osf, N, K)
    assert L.fp4_get_device_status() == 0
    rp, rs = orc.requant(packed, scale, g, OCP, threads=THREADS)
    assert np.array_equal(host(dst[16:]).reshape(N, K // 2), rp)
    assert np.array_equal(host(osf), orc.sf_swizzle(rs))


def _check_requant_grouped(orc, L, packed, scale, gs, alg, layout, bf16=False):
    import torch

    E, N, half = packed.shape
    K = 2 * half
    per = L.fp4_sf_bytes(N, K, layout)
    op = empty_u8(E * N * K // 2)
    osf = empty_u8(E * per)
    gdev = torch.from_numpy(np.asarray(gs, np.float32)).cuda()
    L.fp4_requant_nvfp4_to_mxfp4_grouped(dev(packed), dev(scale), gdev, op, osf, E, N, K, scale_alg=alg,
                                         sf_layout=layout, bf16_intermediate=bf16)
    assert L.fp4_get_device_status() == 0
    hp = host(op)[: E * N * K // 2].reshape(E, N, K // 2)
    hs = host(osf)[: E * per].reshape(E, per)
    for e in range(E):
        rp, rs = orc.requant(packed[e], scale[e], float(gs[e]), alg, threads=THREADS, bf16=bf16)
        assert np.array_equal(hp[e], rp), f"expert {e}: codes differ at {np.argwhere(hp[e] != rp)[:5]}"
        expect = orc.sf_swizzle(rs) if layout == SWZ else rs.reshape(-1)
        assert np.array_equal(hs[e], expect), f"expert {e}: scales differ at {np.argwhere(hs[e] != expect)[:5]}"


@pytest.mark.parametrize("E,N,K", [(3, 130, 1024), (5, 64, 256), (2, 1, 128), (7, 200, 512)])
@pytest.mark.parametrize("alg", [OCP, UOS])
@pytest.mark.parametrize("layout", [SWZ, ROW])
def test_requant_grouped(orc, L, E, N, K, alg, layout):
    rng = np.random.default_rng(E * 1000 + N + K)
    packed = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    scale = rng.integers(0, 256, (E, N, K // 16), dtype=np.uint8)
    gs = np.float32([1.0, 0.0037, -0.25, 2.0 ** -20, 3.0, 1e-4, 7.5])[:E]
    _check_requant_grouped(orc, L, packed, scale, gs, alg, layout)


def test_requant_grouped_special_scales(orc, L):
    rng = np.random.default_rng(9)
    E, N, K = 6, 40, 256
    packed = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    scale = rng.integers(0, 0x7F, (E, N, K // 16), dtype=np.uint8)
    gs = np.float32([0.0, -0.0, np.inf, np.nan, 3.0e38, 1.0e-45])
    _check_requant_grouped(orc, L, packed, scale, gs, OCP, SWZ)



# global scales that put S |g| among the float32 subnormals
SUBNORMAL_G = [float(np.float32(np.ldexp(float(G), -149))) for G in (2796202, 1234567, 7777777, 3, 99991)]
# a scale where bf16 rounding moves an element onto an E2M1 tie
BF16_TIE_G = float(np.float32(0.875 * (1 - 2.0 ** -20)))


@pytest.mark.parametrize("N,K", [(1, 32), (3, 96), (64, 256), (130, 1024)])
@pytest.mark.parametrize("alg", [OCP, UOS])
def test_requant_subnormal_products(orc, L, N, K, alg):
    """Decoded values among the float32 subnormals, where the codes of
    magnitudes 4..7 are not the doublings of codes 2..3 (row 0 block 0 is
    the worked example: code 4 under scale 0.5625 next to the 0.75 tie)."""
    rng = np.random.default_rng(N * 31 + K + alg)
    packed, scale = _random_nvfp4(rng, N, K, 0, 0x7F)
    packed[0, :16] = 0
    packed[0, 0] = 0x04
    scale[0, 0:2] = 0x31
    for g in SUBNORMAL_G:
        for layout in (SWZ, ROW):
            _check_requant(orc, L, packed, scale, g, alg, layout)


@pytest.mark.parametrize("N,K", [(1, 32), (5, 96), (130, 256), (300, 1024)])
@pytest.mark.parametrize("alg", [OCP, UOS])
@pytest.mark.parametrize("layout", [SWZ, ROW])
def test_requant_bf16_intermediate(orc, L, N, K, alg, layout):
    """FP4_QUANT_BF16_INTERMEDIATE: every scale byte and code, ordinary,
    special and subnormal-product global scales; row 0 block 0 is the worked
    example whose bf16 value lands on the q = 1.75 tie."""
    rng = np.random.default_rng(N * 17 + K + alg + layout)
    packed, scale = _random_nvfp4(rng, N, K)
    packed[0, :16] = 0
    packed[0, 0] = 0x62
    scale[0, 0:2] = 0x38
    for g in (1.0, 0.0037, -0.25, 2.0 ** -20, BF16_TIE_G, 3.0e38, 1.0e-38, float("nan"), SUBNORMAL_G[0]):
        _check_requant(orc, L, packed, scale, float(np.float32(g)), alg, layout, bf16=True)


@pytest.mark.parametrize("bf16", [False, True])
def test_requant_grouped_bf16_and_subnormal_scales(orc, L, bf16):
    rng = np.random.default_rng(41)
    E, N, K = 5, 70, 256
    packed = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    scale = rng.integers(0, 256, (E, N, K // 16), dtype=np.uint8)
    gs = np.float32([0.0037, SUBNORMAL_G[0], BF16_TIE_G, -0.25, SUBNORMAL_G[2]])
    for alg in (OCP, UOS):
        _check_requant_grouped(orc, L, packed, scale, gs, alg, SWZ, bf16=bf16)


def _decode_bf16_bits(packed, scale, g):
    """NVFP4 decode on the host, for the identity below: float32 products of
    the exact E2M1 and E4M3 values (torch's E4M3 decode) times g, rounded to
    bf16 by torch (nearest, ties to even)."""
    import torch

    e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], np.float32)
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(packed.shape[0], -1)
    s = torch.from_numpy(np.ascontiguousarray(scale)).view(torch.float8_e4m3fn).float().numpy()
    v = (e2m1[codes] * np.repeat(s, 16, axis=1)) * np.float32(g)
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("alg", [OCP, UOS])
def test_requant_equals_act_quant_of_its_decode(L, bf16, alg):
    """Cross-kernel identity, no oracle: an E2M1 x E4M3 product has at most
    6 significant bits, so with g a power of two every decoded NVFP4 value is
    a bf16 value and the requant's bytes equal the activation quantizer's on
    the decoded tensor; with the bf16 intermediate that holds for any g."""
    rng = np.random.default_rng(51 + alg)
    N, K = 130, 1024
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scale = rng.integers(0x08, 0x7F, (N, K // 16), dtype=np.uint8)  # normal, finite E4M3
    scale[:, ::5] |= 0x80
    for g in ((0.0037, -0.25, 1.7e-3, 2.0 ** -4) if bf16 else (2.0 ** -4, 1.0, -8.0)):
        g32 = float(np.float32(g))
        rp, rs = _kernel_requant(L, packed, scale, g32, alg, SWZ, bf16)
        ap, as_ = _kernel_act(L, _decode_bf16_bits(packed, scale, g32), alg, SWZ)
        assert np.array_equal(rp, ap), (g, np.argwhere(rp != ap)[:5])
        assert np.array_equal(rs, as_), g

# ---------------------------------------------------------------- activations
def _kernel_act(L, x_bits, alg, layout):
    M, K = x_bits.shape
    op = empty_u8(M * K // 2)
    osf = empty_u8(L.fp4_sf_bytes(M, K, layout))
    L.fp4_quant_act_mxfp4(dev_bf16(x_bits), op, osf, M, K, scale_alg=alg, sf_layout=layout)
    return host(op)[: M * K // 2].reshape(M, K // 2), host(osf)[: L.fp4_sf_bytes(M, K, layout)]


def _check_act(orc, L, x_bits, alg=OCP, layout=SWZ):
    kp, ks = _kernel_act(L, x_bits, alg, layout)
    rp, rs = orc.act_quant(x_bits, alg, threads=THREADS)
    assert np.array_equal(kp, rp), f"codes differ at {np.argwhere(kp != rp)[:5]}"
    expect_sf = orc.sf_swizzle(rs) if layout == SWZ else rs.reshape(-1)
    assert np.array_equal(ks, expect_sf), f"scales differ at {np.argwhere(ks != expect_sf)[:5]}"


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (16, 512), (129, 256), (200, 1056), (64, 4096)])
@pytest.mark.parametrize("alg", [OCP, UOS])
@pytest.mark.parametrize("layout", [SWZ, ROW])
def test_act_quant_random_bits(orc, L, M, K, alg, layout):
    rng = np.random.default_rng(M * 31 + K)
    x = rng.integers(0, 1 << 16, (M, K), dtype=np.uint16)      # every bf16 pattern, incl. Inf/NaN/subnormal
    _check_act(orc, L, x, alg, layout)
    y = synth.bf16_normal(M + K, synth.S_ACT, (M, K), 1.0, 0.01, 20.0)
    _check_act(orc, L, y, alg, layout)


def test_act_quant_edge_blocks(orc, L):
    K = 128
    rows = [np.zeros(K, np.uint16), np.full(K, 0x8000, np.uint16), np.full(K, 0x0001, np.uint16),
            np.full(K, 0x0100, np.uint16), np.full(K, 0x7F7F, np.uint16), np.full(K, 0xFF7F, np.uint16),
            np.full(K, 0x40F0, np.uint16)]
    r = np.zeros(K, np.uint16)
    r[5] = 0x7F80                      # +Inf in block 0
    r[40] = 0xFFC1                     # NaN in block 1
    rows.append(r)
    # blocks of subnormals only: the exponent clamps at -127 and the scaled
    # values reach the codes 1..4 (the kernel must keep subnormal inputs)
    sub = (np.arange(K) * 5 % 0x80).astype(np.uint16)
    sub[1::3] |= 0x8000
    rows.append(sub)
    rows.append(np.full(K, 0x007F, np.uint16))
    rows.append((np.arange(K) % 0x81).astype(np.uint16))   # subnormals and the smallest normal
    x = np.stack(rows)
    for alg in (OCP, UOS):
        _check_act(orc, L, x, alg, SWZ)


def test_act_quant_zero_rows_is_noop(L):
    L.fp4_quant_act_mxfp4(None, None, None, 0, 64)


# ---------------------------------------------------------------- grouped
def _expected_grouped_sf(orc, rowmajor_sf, offsets, K):
    kb4 = (K // 32 + 3) // 4
    parts, tiles = [], 0
    for e in range(len(offsets) - 1):
        rows = rowmajor_sf[offsets[e]:offsets[e + 1]]
        if len(rows):
            parts.append(orc.sf_swizzle(rows))
            tiles += (len(rows) + 127) // 128
    used = tiles * kb4 * 512
    return (np.concatenate(parts) if parts else np.zeros(0, np.uint8)), used


@pytest.mark.parametrize("counts,K", [([3, 0, 130, 1, 200], 256), ([0, 0, 5], 96), ([128, 128], 64),
                                      ([1] * 40, 32)])
def test_act_quant_grouped(orc, L, counts, K):
    rng = np.random.default_rng(len(counts) * 100 + K)
    offsets = np.zeros(len(counts) + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    total = int(offsets[-1])
    x = synth.bf16_normal(11, synth.S_ACT, (total, K), 1.0, 0.02, 16.0)
    x[rng.integers(0, total, 3), rng.integers(0, K, 3)] = 0x0001
    E = len(counts)
    op = empty_u8(total * K // 2)
    osf = empty_u8(L.fp4_sf_bytes_grouped(total, E, K))
    L.fp4_quant_act_mxfp4_grouped(dev_bf16(x), dev(offsets), E, total, K, op, osf)
    rp, rs = orc.act_quant(x, OCP)
    assert np.array_equal(host(op)[: total * K // 2].reshape(total, K // 2), rp)
    expect, used = _expected_grouped_sf(orc, rs, offsets, K)
    assert np.array_equal(host(osf)[:used], expect)


# ---------------------------------------------------------------- NVFP4 producer
@pytest.mark.parametrize("M,K", [(1, 16), (7, 48), (256, 512), (300, 1024)])
def test_nvfp4_producer(orc, L, M, K):
    x = synth.bf16_normal(M, synth.S_WEIGHT, (M, K), 0.02, 0.01, 8.0)
    g = orc.nvfp4_global_scale(x)
    op = empty_u8(M * K // 2)
    osc = empty_u8(M * K // 16)
    L.fp4_quant_nvfp4(dev_bf16(x), g, op, osc, M, K)
    rp, rs = orc.nvfp4_quantize(x, g)
    assert np.array_equal(host(op)[: M * K // 2].reshape(M, K // 2), rp)
    assert np.array_equal(host(osc)[: M * K // 16].reshape(M, K // 16), rs)


def test_nvfp4_producer_special_scales(orc, L):
    x = synth.bf16_normal(5, synth.S_WEIGHT, (32, 64), 1.0)
    x[0, :16] = 0
    for g in (1.0, 0.0, 1e-30, 5.0, -0.5):
        op = empty_u8(32 * 32)
        osc = empty_u8(32 * 4)
        L.fp4_quant_nvfp4(dev_bf16(x), g, op, osc, 32, 64)
        rp, rs = orc.nvfp4_quantize(x, float(np.float32(g)))
        assert np.array_equal(host(op).reshape(32, 32), rp), g
        assert np.array_equal(host(osc).reshape(32, 4), rs), g


# ---------------------------------------------------------------- full sizes
def _nvfp4_from_recipe(orc, W):
    g = orc.nvfp4_global_scale(W)
    packed, scale = orc.nvfp4_quantize(W, g, threads=THREADS)
    return packed, scale, g


@pytest.mark.slow
def test_full_decode_workload_quant(orc, L):
    w = synth.workload1()
    packed, scale, g = _nvfp4_from_recipe(orc, w["W"])
    _check_requant(orc, L, packed, scale, g)
    for M, X in w["X"].items():
        _check_act(orc, L, X)


@pytest.mark.slow
def test_full_prefill_workload_quant(orc, L):
    w = synth.workload2()
    packed, scale, g = _nvfp4_from_recipe(orc, w["W"])
    _check_requant(orc, L, packed, scale, g)
    for M, X in w["X"].items():
        _check_act(orc, L, X)


@pytest.mark.slow
def test_full_moe_workload_quant(orc, L):
    w = synth.workload3(experts=[0, 31, 63])
    for e in (0, 31, 63):
        for W in (w["W_gu"][e], w["W_down"][e]):
            packed, scale, g = _nvfp4_from_recipe(orc, W)
            _check_requant(orc, L, packed, scale, g)
    offsets = w["row_offsets"]
    for A in (w["A_gu"], w["A_down"]):
        total, K = A.shape
        E = len(offsets) - 1
        op = empty_u8(total * K // 2)
        osf = empty_u8(L.fp4_sf_bytes_grouped(total, E, K))
        L.fp4_quant_act_mxfp4_grouped(dev_bf16(A), dev(offsets), E, total, K, op, osf)
        rp, rs = orc.act_quant(A, OCP, threads=THREADS)
        assert np.array_equal(host(op)[: total * K // 2].reshape(total, K // 2), rp)
        expect, used = _expected_grouped_sf(orc, rs, offsets, K)
        assert np.array_equal(host(osf)[:used], expect)

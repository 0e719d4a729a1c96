"""GPU parity of the DualScale path ("W4A4 MXFP4 Quantization",
mxfp4_dualscale: fine E8M0 per 32 and coarse float32 per 512 weight
elements) against the oracle, through the C ABI: the online dual-level
quantizer byte for byte (codes, fine scales in both layouts, coarse scales
bit for bit), and the GEMM of MXFP4 activations with DualScale weights
within |out - ref| <= 2^-8 |ref| + 1e-6 sum_k |a_k b_k| on decode (tokens
on the MMA-N side, split-K included) and prefill tile shapes, with an exact
one-hot case."""
import numpy as np
import pytest

import synth
from _util import THREADS, bf16_bits_host, bf16_bits_to_f64, dev, dev_bf16, empty_u8, gemm_check, host, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return lib()


def _weight_bits(N, K, seed, specials=False):
    W = synth.bf16_normal(seed, synth.S_WEIGHT, (N, K), 0.02, 0.002, 16.0)
    if specials and N >= 3:
        W[0, :512] = 0                       # an all-zero group
        W[1, 77] = 0x7FC0                    # NaN
        W[2, K - 3] = 0xFF80                 # -Inf
        W[2, 5] = 0x8000                     # -0
    return W


def _gpu_quant(L, W, sf_layout):
    import torch

    N, K = W.shape
    codes = empty_u8(N * K // 2)
    fine = empty_u8(L.fp4_sf_bytes(N, K, sf_layout))
    coarse = torch.full((N * (K // 512),), float("nan"), dtype=torch.float32, device="cuda")
    L.fp4_quant_dualscale(dev_bf16(W), codes, fine, coarse, N, K, sf_layout)
    assert L.fp4_get_device_status() == 0
    return host(codes).reshape(N, K // 2), host(fine), host(coarse).reshape(N, K // 512)


@pytest.mark.parametrize("N,K", [(1, 512), (100, 1536), (256, 7168), (300, 2048), (129, 4096)])
def test_dual_quant_matches_oracle(orc, L, N, K):
    W = _weight_bits(N, K, N + K, specials=True)
    rp, rf, rc = orc.dual_quantize(W, threads=THREADS)
    for layout in (L.FP4_SF_SWIZZLED, L.FP4_SF_ROWMAJOR):
        codes, fine, coarse = _gpu_quant(L, W, layout)
        assert np.array_equal(codes, rp)
        assert np.array_equal(coarse.view(np.uint32), rc.view(np.uint32))
        want = orc.sf_swizzle(rf) if layout == L.FP4_SF_SWIZZLED else rf.reshape(-1)
        assert np.array_equal(fine, want)


def _gemm_case(orc, L, M, N, K, with_bias, seed, ws=False):
    import torch

    X = synth.bf16_normal(seed, synth.S_ACT, (M, K), 1.0, 0.01, 16.0)
    a, sa = orc.act_quant(X, threads=THREADS)
    b, fine, coarse = orc.dual_quantize(_weight_bits(N, K, seed + 1), threads=THREADS)
    bias = synth.bf16_normal(seed + 2, synth.S_BIAS, (N,), 0.01) if with_bias else None
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    work = None
    if ws:
        need = L.fp4_gemm_workspace_size(M, N, K)
        assert need > 0, "shape must take the split-K path"
        work = torch.zeros(need, dtype=torch.uint8, device="cuda")
    L.fp4_gemm_mxfp4_dualscale(dev(a), dev(orc.sf_swizzle(sa)), dev(b), dev(orc.sf_swizzle(fine)), dev(coarse),
                               None if bias is None else dev_bf16(bias), out, M, N, K, work)
    assert L.fp4_get_device_status() == 0
    got = bf16_bits_host(out)
    rows = np.unique(np.concatenate([np.arange(min(M, 48)), np.linspace(0, M - 1, min(M, 24)).astype(np.int64)]))
    ref, absum = orc.gemm_dual(a, sa, b, fine, coarse, bias, rows=rows, threads=THREADS)
    ok, ratio = gemm_check(got[rows], ref, absum)
    assert ok, f"max err/bound = {ratio}"
    if work is not None:
        assert int(torch.count_nonzero(work[: 4 * torch.cuda.get_device_properties(0).multi_processor_count])) == 0


@pytest.mark.parametrize("M,N,K", [(1, 128, 512), (7, 264, 2048), (16, 1024, 7168), (33, 384, 1536),
                                   (64, 14336, 4096), (130, 640, 1024), (256, 1024, 7168), (1000, 136, 512)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_dual_gemm_matches_oracle(orc, L, M, N, K, with_bias):
    _gemm_case(orc, L, M, N, K, with_bias, M * 31 + N + K)


@pytest.mark.parametrize("M,N,K", [(16, 1024, 8192), (64, 2048, 16384)])
def test_dual_gemm_split_k_matches_oracle(orc, L, M, N, K):
    _gemm_case(orc, L, M, N, K, True, M + N, ws=True)


@pytest.mark.parametrize("M", [9, 200])
def test_dual_gemm_one_hot_is_exact(orc, L, M):
    """B rows one-hot with code 1.0 under fine scale 2^0 and a power-of-two
    coarse scale per group: out[:, n] = A[:, sel[n]] x coarse[n, sel[n] / 512]."""
    import torch

    rng = np.random.default_rng(M)
    N, K = 136, 2048
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sa = rng.integers(110, 140, (M, K // 32), dtype=np.uint8)
    sel = rng.integers(0, K, N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), sel] = 0x2
    b = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    fine = np.full((N, K // 32), 127, np.uint8)
    coarse = (2.0 ** rng.integers(-5, 5, (N, K // 512))).astype(np.float32)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.fp4_gemm_mxfp4_dualscale(dev(a), dev(orc.sf_swizzle(sa)), dev(b), dev(orc.sf_swizzle(fine)), dev(coarse), None,
                               out, M, N, K)
    assert L.fp4_get_device_status() == 0
    ref, _ = orc.gemm_dual(a, sa, b, fine, coarse)
    assert np.array_equal(bf16_bits_to_f64(bf16_bits_host(out)), ref)

"""The GEMM entry point that allocates nothing (its split-K scratch is a fixed
array in the library's device image) against the entry point that takes a
caller workspace: bit-identical outputs on two calls in a row, so the
counters the first call used are back at zero for the second.  Collected
last on purpose; it must pass alone as well as after every other test."""
import numpy as np
import pytest

from _util import bf16_bits_host, lib

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 2 << 20


@pytest.fixture(scope="module")
def L():
    return lib()


def _operands(M, N, K, seed):
    import torch

    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    a = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device="cuda", generator=g)
    b = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=g)
    return a, b


def _scales(L, rows, K, seed):
    import torch

    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(118, 136, (L.fp4_sf_bytes(rows, K),), dtype=torch.uint8, device="cuda", generator=g)


def _out(M, N):
    import torch

    return torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")


@pytest.mark.parametrize("M,N,K", [(32, 1024, 16384), (7, 896, 8192), (64, 256, 30720)])
def test_no_alloc_matches_workspace_entry_twice(L, M, N, K):
    import torch

    need = L.fp4_gemm_workspace_size(M, N, K)
    assert 0 < need <= SCRATCH_BYTES, "shape must split and fit the fixed scratch"
    a, b = _operands(M, N, K, M + N)
    sa, sb = _scales(L, M, K, 1), _scales(L, N, K, 2)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ref = _out(M, N)
    L.fp4_gemm_mxfp4_ws(a, sa, b, sb, None, ref, M, N, K, ws)
    for _ in range(2):
        out = _out(M, N)
        L.fp4_gemm_mxfp4_noalloc(a, sa, b, sb, None, out, M, N, K)
        assert L.fp4_get_device_status() == 0
        assert np.array_equal(bf16_bits_host(out), bf16_bits_host(ref))


def test_no_alloc_without_split_matches_plain_entry(L):
    M, N, K = 64, 14336, 4096          # more tiles than half the SMs: no scratch used
    assert L.fp4_gemm_workspace_size(M, N, K) == 0
    a, b = _operands(M, N, K, 3)
    sa, sb = _scales(L, M, K, 4), _scales(L, N, K, 5)
    ref = _out(M, N)
    L.fp4_gemm_mxfp4(a, sa, b, sb, None, ref, M, N, K)
    for _ in range(2):
        out = _out(M, N)
        L.fp4_gemm_mxfp4_noalloc(a, sa, b, sb, None, out, M, N, K)
        assert L.fp4_get_device_status() == 0
        assert np.array_equal(bf16_bits_host(out), bf16_bits_host(ref))


def test_no_alloc_rejects_problems_beyond_the_scratch(L):
    M, N, K = 64, 2048, 8192           # split plan needs 4 MiB of partial tiles
    assert L.fp4_gemm_workspace_size(M, N, K) > SCRATCH_BYTES
    a, b = _operands(M, N, K, 6)
    sa, sb = _scales(L, M, K, 7), _scales(L, N, K, 8)
    with pytest.raises(L.Fp4Error) as err:
        L.fp4_gemm_mxfp4_noalloc(a, sa, b, sb, None, _out(M, N), M, N, K)
    assert err.value.status == L.FP4_ERR_SHAPE


def test_no_alloc_recovers_after_a_device_timeout(L):
    """A timeout inside the split-K hand-over (driven by the test hook, no GPU
    fault) can leave counters set in the shared array.  The next call clears
    them before its kernel runs, so it matches the workspace entry point
    again, twice in a row."""
    import torch

    M, N, K = 32, 1024, 16384
    a, b = _operands(M, N, K, 9)
    sa, sb = _scales(L, M, K, 10), _scales(L, N, K, 11)
    ws = torch.zeros(L.fp4_gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    ref = _out(M, N)
    L.fp4_gemm_mxfp4_ws(a, sa, b, sb, None, ref, M, N, K, ws)
    L.fp4_debug_set_wait_fault(2_000_000, 1)
    try:
        L.fp4_gemm_mxfp4_noalloc(a, sa, b, sb, None, _out(M, N), M, N, K)
        st = L.fp4_get_device_status()
    finally:
        L.fp4_debug_set_wait_fault(0, 0)
    assert st == L.FP4_ERR_TIMEOUT
    for _ in range(2):
        out = _out(M, N)
        L.fp4_gemm_mxfp4_noalloc(a, sa, b, sb, None, out, M, N, K)
        assert L.fp4_get_device_status() == 0
        assert np.array_equal(bf16_bits_host(out), bf16_bits_host(ref))

"""Host-side logic of bench.py that needs no GPU: the pieces a weight is
uploaded in, the scale-array offset of a row chunk, and the committed
traffic table lookup."""
import types

import pytest

import bench


@pytest.mark.parametrize("N,n", [(14336, 1), (14336, 8), (18432, 3), (200, 4), (128, 8)])
def test_weight_pieces_cover_the_rows_in_128_row_multiples(N, n):
    w = types.SimpleNamespace(N=N, E=1)
    parts = bench.Weight.parts(w, n)
    assert parts[0][0] == 0 and parts[-1][1] == N
    for (a0, a1), (b0, _) in zip(parts, parts[1:]):
        assert a1 == b0                      # contiguous, no overlap
    for p0, p1 in parts:
        assert p0 % 128 == 0 and p1 > p0     # each piece starts a swizzled scale tile
    assert len(parts) <= max(n, 1)
    assert bench.Weight.rows(w, *parts[-1]) == parts[-1]


@pytest.mark.parametrize("E,n", [(64, 8), (64, 1), (5, 2), (3, 8)])
def test_expert_pieces_cover_the_experts(E, n):
    w = types.SimpleNamespace(N=2048, E=E)
    parts = bench.Weight.parts(w, n)
    assert parts[0][0] == 0 and parts[-1][1] == E
    assert all(a1 == b0 for (_, a1), (b0, _) in zip(parts, parts[1:]))
    p0, p1 = parts[-1]
    assert bench.Weight.rows(w, p0, p1) == (p0 * 2048, p1 * 2048)


@pytest.mark.parametrize("K", [1024, 4096, 7168, 1152])
def test_row_chunk_scale_offset_is_the_swizzled_index(orc, K):
    """Act._sf_off(m0) is where row m0's scale bytes start in the swizzled
    layout, for every row-tile start m0."""
    act = types.SimpleNamespace(K=K)
    for m0 in (0, 128, 2048, 6144):
        assert bench.Act._sf_off(act, m0) == orc.sf_swizzled_offset(m0, 0, K // 32)


def test_committed_traffic_rows_parse():
    """Each row of profiles/traffic.md whose source hash still matches is
    returned as bytes; an unknown kernel gives None."""
    for wl in ("decode", "prefill", "moe"):
        v = bench._committed_traffic(wl, "gemm_fp4_kernel")
        assert v is None or v > 1e7
    assert bench._committed_traffic("decode", "no_such_kernel") is None

"""Host-side logic of bench.py that needs no GPU: the pieces a weight is
uploaded in, the scale-array offset of a row chunk, the committed traffic
lookup and the requant error statistic."""
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


def test_committed_traffic_entries_parse():
    """Each entry of bench_traffic.json whose source hash still matches is
    returned as bytes; an unknown kernel gives None."""
    for wl in ("decode", "prefill", "moe"):
        for k in bench.KERNEL_SOURCES:
            v = bench._committed_traffic(wl, k)
            assert v is None or v > 1e6
    assert bench._committed_traffic("decode", "no_such_kernel") is None


def test_requant_error_matches_the_oracle_decodes(orc):
    """bench.requant_error on CPU tensors (two stacked tensors of a small
    seeded weight): its MSE, max-abs and relative RMS error equal the ones
    computed in float64 from the oracle's NVFP4 decode and an MX decode of
    the oracle's requantized bytes."""
    import numpy as np
    import torch

    import synth

    N, K, E = 200, 256, 2
    packed, scale, b_packed, b_scale, gs, diffs, refs = [], [], [], [], [], [], []
    for e in range(E):
        W = synth.bf16_normal(40 + e, synth.S_WEIGHT, (N, K), 0.02, 0.01, 8.0)
        g = orc.nvfp4_global_scale(W)
        wp, ws = orc.nvfp4_quantize(W, g)
        bp, bs = orc.requant(wp, ws, g)
        v = orc.nvfp4_dequant(wp, ws, g).astype(np.float64)
        codes = np.stack([bp & 15, bp >> 4], axis=-1).reshape(N, K)
        table = np.array([orc.e2m1_value(c) for c in range(16)])
        dq = table[codes] * np.repeat(2.0 ** (bs.astype(np.float64) - 127), 32, axis=1)
        diffs.append(dq - v)
        refs.append(v)
        packed.append(wp)
        scale.append(ws)
        b_packed.append(bp)
        b_scale.append(orc.sf_swizzle(bs))
        gs.append(g)
    w = types.SimpleNamespace(
        N=N, K=K, E=E, g=gs, sf_bytes=len(b_scale[0]),
        packed=torch.from_numpy(np.concatenate(packed)), scale=torch.from_numpy(np.concatenate(scale)),
        b_packed=torch.from_numpy(np.concatenate(b_packed)), b_scale=torch.from_numpy(np.concatenate(b_scale)))
    got = bench.requant_error(torch, w, chunk_rows=64)
    d = np.concatenate(diffs)
    ref = np.concatenate(refs)
    assert got["elements"] == E * N * K
    assert got["mse"] == pytest.approx(float(np.mean(d * d)), rel=1e-12)
    assert got["max_abs"] == float(np.max(np.abs(d)))
    assert got["rel_rmse"] == pytest.approx(float(np.sqrt(np.sum(d * d) / np.sum(ref * ref))), rel=1e-12)
    assert got["max_abs"] > 0

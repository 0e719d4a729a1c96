"""Host-side checks of the layer-streamed loader (no GPU): planning, the
memory ledger (staging never above one layer), FP8 pass-through, and
failure at a layer followed by a resume from that layer.  The executor is a
numpy fake whose requant step is the oracle."""
import numpy as np
import pytest

from nvfp4_mxfp4_w4a4_gb300.loader import ALIGN, LayerSpec, LayerStreamLoader, LoadError, TensorSpec, plan

TENSORS = (TensorSpec("q", 256, 128), TensorSpec("o", 256, 128), TensorSpec("mlp", 512, 128))


def _layers(n=6, excluded=(0, 5)):
    return [LayerSpec(i, TENSORS, i in excluded) for i in range(n)]


class FakeExecutor:
    def __init__(self, orc):
        self.orc = orc
        self.bufs = []

    def allocated_bytes(self):
        return sum(b.size for b in self.bufs)

    def alloc(self, n):
        b = np.zeros(n, np.uint8)
        self.bufs.append(b)
        return b

    def stage(self, staging, off, arr, slot):
        flat = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
        staging[off:off + flat.size] = flat

    def requant(self, t, staging, c_off, s_off, g, dc, ds, slot):
        packed = staging[c_off:c_off + t.N * t.K // 2].reshape(t.N, t.K // 2)
        scale = staging[s_off:s_off + t.N * t.K // 16].reshape(t.N, t.K // 16)
        p, s = self.orc.requant(packed, scale, g)
        dc[:] = p.reshape(-1)
        ds[:] = self.orc.sf_swizzle(s)

    def passthrough(self, dst, arr):
        dst[:] = np.ascontiguousarray(arr).reshape(-1)

    def layer_done(self, layer):
        pass

    def sync(self):
        pass


def _source(fail_at=None):
    def src(layer):
        if layer == fail_at:
            raise IOError(f"shard of layer {layer} unreadable")
        rng = np.random.default_rng(layer)
        out = {}
        for t in TENSORS:
            if layer in (0, 5):
                out[t.name] = {"fp8": rng.integers(0, 0x7F, (t.N, t.K), dtype=np.uint8)}
            else:
                out[t.name] = {"packed": rng.integers(0, 256, (t.N, t.K // 2), dtype=np.uint8),
                               "scale": rng.integers(0x30, 0x7E, (t.N, t.K // 16), dtype=np.uint8),
                               "g": float(np.float32(10.0 ** rng.uniform(-4, -2)))}
        return out
    return src


def _sf_bytes(orc):
    return lambda N, K: orc.sf_swizzled_bytes(N, K // 32)


def test_plan_staging_is_one_layer(orc):
    p = plan(_layers(), _sf_bytes(orc))
    one_layer = sum(t.nvfp4_bytes for t in TENSORS)
    assert p.largest_layer_bytes == one_layer
    assert one_layer <= p.staging_bytes <= one_layer + 2 * len(TENSORS) * ALIGN
    offs = sorted(o for v in p.slots.values() for o in v)
    assert all(o % ALIGN == 0 for o in offs)


def test_stream_matches_oracle_and_passes_fp8_through(orc):
    ex = FakeExecutor(orc)
    ld = LayerStreamLoader(_layers(), ex, _sf_bytes(orc))
    assert ld.ledger["staging_bytes"] <= ld.ledger["largest_layer_nvfp4_bytes"] + 2 * len(TENSORS) * ALIGN
    assert ld.load(_source()) == 6
    src = _source()
    for layer in range(6):
        h = src(layer)
        for t in TENSORS:
            if layer in (0, 5):
                assert np.array_equal(ld.dest[(layer, t.name)], h[t.name]["fp8"].reshape(-1))
            else:
                p, s = orc.requant(h[t.name]["packed"], h[t.name]["scale"], h[t.name]["g"])
                dc, ds = ld.dest[(layer, t.name)]
                assert np.array_equal(dc, p.reshape(-1))
                assert np.array_equal(ds, orc.sf_swizzle(s))


def test_failure_reports_layer_and_resume_completes(orc):
    ex = FakeExecutor(orc)
    ld = LayerStreamLoader(_layers(), ex, _sf_bytes(orc))
    with pytest.raises(LoadError) as ei:
        ld.load(_source(fail_at=3))
    assert ei.value.layer == 3 and ld.loaded == 3
    assert isinstance(ei.value.cause, IOError)
    # resume from the failed layer with a healthy source
    assert ld.load(_source(), start=ei.value.layer) == 6
    ref = LayerStreamLoader(_layers(), FakeExecutor(orc), _sf_bytes(orc))
    ref.load(_source())
    for key, v in ref.dest.items():
        got = ld.dest[key]
        if isinstance(v, tuple):
            assert np.array_equal(got[0], v[0]) and np.array_equal(got[1], v[1])
        else:
            assert np.array_equal(got, v)

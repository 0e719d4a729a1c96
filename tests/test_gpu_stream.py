"""GPU run of the layer-streamed load at full size: 60 layers of q,k,v,o
[7168,7168] + MLP [18432,7168]; layers 0 and 59 are FP8 pass-through.  Every
requantized tensor is checked against the oracle on sampled rows (codes and
their swizzled scale bytes), the FP8 layers byte for byte, and the device
memory beyond the preallocated destination is held to one layer."""
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import synth
from _util import THREADS, lib

pytestmark = pytest.mark.gpu


def _layer_specs():
    from nvfp4_mxfp4_w4a4_gb300.loader import LayerSpec, TensorSpec

    tensors = tuple(TensorSpec(n, N, synth.HIDDEN4) for n, N in synth.TENSORS4)
    return [LayerSpec(i, tensors, i in synth.EXCLUDED4) for i in range(synth.LAYERS4)]


class PrefetchingSource:
    """Generates layer l+1 on host threads while layer l is being loaded."""

    def __init__(self, n_layers):
        self.pool = ThreadPoolExecutor(len(synth.TENSORS4))
        self.n = n_layers
        self.pending = {}
        self.lock = threading.Lock()
        self._submit(0)

    def _gen(self, layer):
        futs = [self.pool.submit(synth.workload4_tensor, layer, i) for i in range(len(synth.TENSORS4))]
        return {name: f.result() for (name, _), f in zip(synth.TENSORS4, futs)}

    def _submit(self, layer):
        if layer < self.n and layer not in self.pending:
            self.pending[layer] = self.pool.submit(self._gen, layer)

    def __call__(self, layer):
        self._submit(layer)
        out = self.pending.pop(layer).result()
        self._submit(layer + 1)
        return out


@pytest.mark.slow
def test_full_layer_stream(orc):
    import torch

    L = lib()
    from nvfp4_mxfp4_w4a4_gb300.loader import CudaExecutor, LayerStreamLoader

    torch.cuda.synchronize()
    base_alloc = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    layers = _layer_specs()
    ex = CudaExecutor()
    ld = LayerStreamLoader(layers, ex, lambda N, K: L.fp4_sf_bytes(N, K))
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    torch.cuda.reset_peak_memory_stats()
    ledger = ld.ledger
    one_layer = ledger["largest_layer_nvfp4_bytes"]
    assert ledger["staging_bytes"] <= one_layer + 10 * 256
    # what the loader holds on the device = destination + one staging buffer
    # (the caching allocator may round each block up to its 2 MiB segment)
    n_allocs = 3 * len(layers) * len(synth.TENSORS4)
    held_after_alloc = torch.cuda.memory_allocated()
    assert held_after_alloc - base_alloc <= ledger["destination_bytes"] + ledger["staging_bytes"] + (2 << 20) * n_allocs

    src = PrefetchingSource(len(layers))
    rng = np.random.default_rng(4)
    checked = []      # only the sampled rows are kept on the host

    def source(layer):
        h = src(layer)
        keep = {}
        for name, N in synth.TENSORS4:
            if layer in synth.EXCLUDED4:
                keep[name] = h[name]
            else:
                rows = np.sort(rng.choice(N, 12, replace=False))
                rows[0], rows[-1] = 0, N - 1
                keep[name] = {"rows": rows, "packed": h[name]["packed"][rows].copy(),
                              "scale": h[name]["scale"][rows].copy(), "g": h[name]["g"]}
        checked.append((layer, keep))
        return h

    t0 = time.perf_counter()
    ld.load(source)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    assert L.fp4_get_device_status() == 0
    # streaming allocates no device memory at all: the peak is the level
    # reached right after the destination and the one staging buffer
    assert torch.cuda.max_memory_allocated() == held_after_alloc, (torch.cuda.max_memory_allocated(), held_after_alloc)

    for layer, h in checked:
        for name, N in synth.TENSORS4:
            K = synth.HIDDEN4
            if layer in synth.EXCLUDED4:
                got = ld.dest[(layer, name)].cpu().numpy()
                assert np.array_equal(got, h[name]["fp8"].reshape(-1)), (layer, name)
                continue
            dc, ds = ld.dest[(layer, name)]
            rows = h[name]["rows"]
            p, s = orc.requant(h[name]["packed"], h[name]["scale"], h[name]["g"])
            codes = dc.view(N, K // 2)[torch.from_numpy(rows).cuda()].cpu().numpy()
            assert np.array_equal(codes, p), (layer, name)
            sf = ds.cpu().numpy()
            for j, r in enumerate(rows):
                offs = [orc.sf_swizzled_offset(int(r), c, K // 32) for c in range(K // 32)]
                assert np.array_equal(sf[offs], s[j]), (layer, name, r)
    print(f"\nlayer stream: {len(layers)} layers in {wall:.1f} s wall (host generation bound); "
          f"destination {ledger['destination_bytes'] / 1e9:.2f} GB, staging {ledger['staging_bytes'] / 1e6:.1f} MB, "
          f"one layer {one_layer / 1e6:.1f} MB, device free before/after alloc {free0 / 1e9:.1f}/{free1 / 1e9:.1f} GB")


def test_page_locked_tensor_source(orc):
    """Page-locked torch tensors as the source are uploaded without a host
    copy and load the same bytes as numpy arrays (three layers of 256-row
    tensors, layer 0 an FP8 pass-through); a pageable tensor is refused."""
    import torch

    L = lib()
    from nvfp4_mxfp4_w4a4_gb300.loader import CudaExecutor, LayerSpec, LayerStreamLoader, LoadError, TensorSpec

    rows, K = 256, synth.HIDDEN4
    tensors = tuple(TensorSpec(n, rows, K) for n, _ in synth.TENSORS4)
    layers = [LayerSpec(i, tensors, i == 0) for i in range(3)]
    gen = {ly: {name: synth.workload4_tensor(ly, i, rows=rows) for i, (name, _) in enumerate(synth.TENSORS4)}
           for ly in range(3)}

    def pinned(ly):
        return {name: {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() if isinstance(v, np.ndarray) else v
                       for k, v in d.items()} for name, d in gen[ly].items()}

    loads = []
    for source in (lambda ly: gen[ly], pinned):
        ld = LayerStreamLoader(layers, CudaExecutor(), lambda n, k: L.fp4_sf_bytes(n, k))
        assert ld.load(source) == 3
        loads.append(ld)
    assert L.fp4_get_device_status() == 0
    for key, d in loads[0].dest.items():
        other = loads[1].dest[key]
        if isinstance(d, tuple):
            assert all(torch.equal(x, y) for x, y in zip(d, other)), key
        else:
            assert torch.equal(d, other), key
    # one requantized tensor against the oracle, all rows
    h = gen[2]["mlp"]
    p, s = orc.requant(h["packed"], h["scale"], h["g"], threads=THREADS)
    dc, ds = loads[1].dest[(2, "mlp")]
    assert np.array_equal(dc.view(rows, K // 2).cpu().numpy(), p)
    assert np.array_equal(ds.cpu().numpy(), orc.sf_swizzle(s))
    # the bf16-intermediate option through the executor
    ld16 = LayerStreamLoader(layers, CudaExecutor(bf16_intermediate=True), lambda n, k: L.fp4_sf_bytes(n, k))
    assert ld16.load(pinned) == 3
    p16, s16 = orc.requant(h["packed"], h["scale"], h["g"], threads=THREADS, bf16=True)
    dc, ds = ld16.dest[(2, "mlp")]
    assert np.array_equal(dc.view(rows, K // 2).cpu().numpy(), p16)
    assert np.array_equal(ds.cpu().numpy(), orc.sf_swizzle(s16))

    bad = LayerStreamLoader(layers, CudaExecutor(), lambda n, k: L.fp4_sf_bytes(n, k))
    with pytest.raises(LoadError) as err:
        bad.load(lambda ly: {name: {"fp8": torch.from_numpy(d["fp8"])} for name, d in gen[0].items()})
    assert err.value.layer == 0 and isinstance(err.value.cause, ValueError)

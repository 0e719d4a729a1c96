"""Layer-streamed load-time requantization.

Follows the online requantization pipeline of "Efficiently Serving NVFP4
Models on AMD Instinct MI350X/MI355X Accelerators via Online NVFP4 to Quark
MXFP4 Requantization" (the pipeline description around Figure 1): weights
are requantized once at load, one layer at a time, each result is written
straight into a destination allocated up front, and the extra memory the
pipeline needs is bounded by a single layer.  Layers the producer kept in
higher precision (here: FP8-E4M3 layers) take their own load-as-is path.

Here the per-layer "dequantized intermediate" never exists: a layer's NVFP4
tensors are copied host -> device into ONE staging buffer (sized for the
largest layer) and the requant kernel decodes and re-encodes in registers,
writing MXFP4 codes and swizzled E8M0 scales into the destination.  Copies
run on a copy stream, requants on a compute stream; a staging byte range is
refilled for the next layer only after every requant that read it finished
(one event per issued requant), so copy and compute overlap without a
second buffer.

The orchestration (planning, memory ledger, resume bookkeeping) is plain
Python over an executor; `CudaExecutor` drives libfp4lin through its C ABI.
A failed layer raises LoadError carrying its index; requantization is
idempotent per layer, so `load(source, start=err.layer)` resumes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

ALIGN = 256  # bytes; every staging slot and destination starts 256-byte aligned


def _align(n: int) -> int:
    return (n + ALIGN - 1) // ALIGN * ALIGN


@dataclass(frozen=True)
class TensorSpec:
    name: str
    N: int
    K: int

    @property
    def nvfp4_bytes(self) -> int:
        return self.N * self.K // 2 + self.N * self.K // 16


@dataclass(frozen=True)
class LayerSpec:
    index: int
    tensors: tuple
    excluded: bool = False      # kept as-is (FP8-E4M3 pass-through)


class LoadError(RuntimeError):
    def __init__(self, layer: int, cause: BaseException):
        super().__init__(f"loading layer {layer} failed: {cause!r}")
        self.layer = layer
        self.cause = cause


@dataclass
class Plan:
    """Byte layout of the staging buffer and the destination sizes."""
    staging_bytes: int
    slots: dict = field(default_factory=dict)        # (layer, name) -> (codes_off, scale_off)
    dest_bytes: dict = field(default_factory=dict)   # (layer, name) -> (codes, scales) or fp8 bytes
    largest_layer_bytes: int = 0


def plan(layers, sf_bytes) -> Plan:
    """Staging slots for every requantized layer (offsets restart at 0 for
    each layer: one layer's tensors are resident at a time) and the
    destination sizes.  `sf_bytes(N, K)` gives the swizzled scale size."""
    p = Plan(staging_bytes=0)
    for L in layers:
        layer_bytes = sum(t.nvfp4_bytes for t in L.tensors)
        p.largest_layer_bytes = max(p.largest_layer_bytes, layer_bytes)
        if L.excluded:
            for t in L.tensors:
                p.dest_bytes[(L.index, t.name)] = t.N * t.K
            continue
        off = 0
        for t in L.tensors:
            c = off
            off = _align(off + t.N * t.K // 2)
            s = off
            off = _align(off + t.N * t.K // 16)
            p.slots[(L.index, t.name)] = (c, s)
            p.dest_bytes[(L.index, t.name)] = (t.N * t.K // 2, sf_bytes(t.N, t.K))
        p.staging_bytes = max(p.staging_bytes, off)
    return p


class LayerStreamLoader:
    """Drives the layer stream over an executor.

    The executor provides: alloc(nbytes) -> handle, stage(handle, offset,
    host_bytes, slot_id), requant(layer, tensor, codes_view, scale_view, g,
    dst_codes, dst_scale, slot_id), passthrough(dst, host_bytes), sync(), and
    allocated_bytes().
    """

    def __init__(self, layers, executor, sf_bytes):
        self.layers = list(layers)
        self.ex = executor
        self.plan = plan(self.layers, sf_bytes)
        self.dest = {}
        self.ledger = {}
        before = executor.allocated_bytes()
        for key, sz in self.plan.dest_bytes.items():
            if isinstance(sz, tuple):
                self.dest[key] = (executor.alloc(sz[0]), executor.alloc(sz[1]))
            else:
                self.dest[key] = executor.alloc(sz)
        after_dest = executor.allocated_bytes()
        self.staging = executor.alloc(max(ALIGN, self.plan.staging_bytes))
        after_staging = executor.allocated_bytes()
        self.ledger = {"destination_bytes": after_dest - before,
                       "staging_bytes": after_staging - after_dest,
                       "largest_layer_nvfp4_bytes": self.plan.largest_layer_bytes}
        self.loaded = 0           # layers [0, loaded) are complete

    def load(self, source, start: int = 0):
        """Streams layers [start, n).  `source(layer)` returns, per tensor
        name, either dict(packed, scale, g) (NVFP4 host arrays) or dict(fp8);
        with `CudaExecutor` the arrays may also be page-locked uint8 torch
        tensors, which are uploaded without a host-side copy."""
        self.loaded = start
        for L in self.layers[start:]:
            try:
                host = source(L.index)
                if L.excluded:
                    for t in L.tensors:
                        self.ex.passthrough(self.dest[(L.index, t.name)], host[t.name]["fp8"])
                else:
                    for i, t in enumerate(L.tensors):
                        h = host[t.name]
                        c_off, s_off = self.plan.slots[(L.index, t.name)]
                        self.ex.stage(self.staging, c_off, h["packed"], slot=(i, 0))
                        self.ex.stage(self.staging, s_off, h["scale"], slot=(i, 1))
                        dc, ds = self.dest[(L.index, t.name)]
                        self.ex.requant(t, self.staging, c_off, s_off, float(h["g"]), dc, ds, slot=i)
                self.ex.layer_done(L.index)
            except LoadError:
                raise
            except Exception as e:  # noqa: BLE001 - reported with the layer index
                raise LoadError(L.index, e) from e
            self.loaded = L.index + 1
        self.ex.sync()
        return self.loaded


class CudaExecutor:
    """Executor over torch device memory and libfp4lin.  scale_alg picks the
    MX block rule; bf16_intermediate rounds the decoded NVFP4 values to bf16
    before it (FP4_QUANT_BF16_INTERMEDIATE)."""

    def __init__(self, scale_alg=0, bf16_intermediate=False):
        import torch

        from . import fp4lin as L

        self.torch, self.L = torch, L
        self.alg = scale_alg
        self.bf16 = bool(bf16_intermediate)
        self.copy_stream = torch.cuda.Stream()
        self.compute_stream = torch.cuda.Stream()
        self._allocs = []
        self._readers = []        # (start, end, event): staging ranges read by issued requants
        self._pinned = {}
        self._copy_done = {}

    def allocated_bytes(self) -> int:
        return sum(t.numel() for t in self._allocs)

    def alloc(self, nbytes: int):
        t = self.torch.empty(nbytes, dtype=self.torch.uint8, device="cuda")
        self._allocs.append(t)
        return t

    def _pinned_copy(self, key, arr):
        """Page-locked bytes of `arr` for an asynchronous upload.  A
        page-locked contiguous uint8 torch tensor is used as it is (its owner
        leaves it unchanged until the loader has synchronised); anything else
        is copied into a page-locked buffer kept per slot."""
        import numpy as np

        torch = self.torch
        if isinstance(arr, torch.Tensor):
            if not (arr.is_pinned() and arr.dtype == torch.uint8 and arr.is_contiguous()):
                raise ValueError("tensor sources must be page-locked, contiguous uint8")
            return arr.reshape(-1)
        flat = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
        buf = self._pinned.get(key)
        if buf is None or buf.numel() < flat.size:
            buf = self.torch.empty(flat.size, dtype=self.torch.uint8).pin_memory()
            self._pinned[key] = buf
        # the previous copy out of this pinned buffer must be finished
        ev = self._copy_done.get(key)
        if ev is not None:
            ev.synchronize()
        buf[: flat.size].numpy()[:] = flat
        return buf[: flat.size]

    def stage(self, staging, offset, arr, slot):
        torch = self.torch
        src = self._pinned_copy(slot, arr)
        end = offset + src.numel()
        with torch.cuda.stream(self.copy_stream):
            # refill a staging range only after every requant reading it finished
            for r0, r1, ev in self._readers:
                if r0 < end and offset < r1:
                    self.copy_stream.wait_event(ev)
            staging[offset:end].copy_(src, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.copy_stream)
            self._copy_done[slot] = ev

    def requant(self, t, staging, c_off, s_off, g, dst_codes, dst_scale, slot):
        torch = self.torch
        with torch.cuda.stream(self.compute_stream):
            for part in (0, 1):
                self.compute_stream.wait_event(self._copy_done[(slot, part)])
            base = staging.data_ptr()
            self.L.fp4_requant_nvfp4_to_mxfp4(base + c_off, base + s_off, g, dst_codes, dst_scale, t.N, t.K,
                                              stream=self.compute_stream, scale_alg=self.alg,
                                              bf16_intermediate=self.bf16)
            ev = torch.cuda.Event()
            ev.record(self.compute_stream)
        self._readers = [r for r in self._readers if not r[2].query()]
        self._readers.append((c_off, c_off + t.N * t.K // 2, ev))
        self._readers.append((s_off, s_off + t.N * t.K // 16, ev))

    def passthrough(self, dst, arr):
        torch = self.torch
        src = self._pinned_copy(("fp8",), arr)
        with torch.cuda.stream(self.copy_stream):
            dst[: src.numel()].copy_(src, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.copy_stream)
            self._copy_done[("fp8",)] = ev

    def layer_done(self, layer):
        pass

    def sync(self):
        self.torch.cuda.synchronize()

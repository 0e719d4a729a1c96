"""Benchmark of the W4A4 MXFP4 linear layer (libfp4lin) on GB300.

One step = one pass of the whole hot path on the decode-shaped layer
(weight N=14336, K=4096, NVFP4 from bf16 ~N(0,0.02) with 4 outlier K-columns
x8; bias ~N(0,0.01); activations M in {1, 8, 32, 64}, K=4096 ~N(0,1)):
  requantize the NVFP4 weight to MXFP4, then for each M quantize the
  activations and run the W4A4 GEMM with bias.
The step is captured once as a CUDA graph (9 kernel launches) and replayed.
Before every timed step L2 is flushed outside the timed events: a 512 MiB
buffer is written, then a second 512 MiB buffer is read, so the previous
step's lines are gone and the write-backs of the flush itself are paid before
the events start.  `value` = GEMM FLOPs of the step / device time of the step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own replica (the path has no exchange
step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 W4A4 GEMM TFLOPS & % FP4 peak; NVFP4→MXFP4 requant GB/s"
N_W, K_W = 14336, 4096
MS = (1, 8, 32, 64)
FP4_NOMINAL_TFLOPS = 15000.0      # dense block-scaled FP4, Blackwell Ultra public figure
WORKLOAD = "decode layer: W[14336,4096] NVFP4->MXFP4 requant + MXFP4 act-quant + W4A4 GEMM (+bias), M in {1,8,32,64}"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--breakdown-reps", type=int, default=200)
    ap.add_argument("--flush-mib", type=int, default=512, help="L2 flush buffer size (0 = no flush)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def step_flops():
    return sum(2.0 * M * N_W * K_W for M in MS)


def requant_bytes():
    return N_W * K_W * (0.5625 + 0.53125)


def act_bytes(M):
    return M * K_W * (2 + 0.53125)


def gemm_bytes(M):
    return 0.53125 * (M + N_W) * K_W + 2.0 * M * N_W + 2.0 * N_W


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch

            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x, device=None):
    if pg is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ our arm
class Layer:
    """Device buffers and the captured step for the decode-shaped layer."""

    def __init__(self, L, torch, flush_mib=512):
        import synth

        self.L, self.torch = L, torch
        dev = torch.device("cuda")
        W = synth.workload1()
        self.inputs_host = W
        wb = torch.from_numpy(W["W"].view(np.int16)).to(dev).view(torch.bfloat16)
        amax = float(torch.from_numpy(synth.bf16_bits_to_f32(W["W"])).abs().max())
        self.g = float(np.float32(amax) / np.float32(6.0 * 448.0))
        # NVFP4 weight made on the device by the library's NVFP4 producer (setup, not timed)
        self.w_packed = torch.empty((N_W, K_W // 2), dtype=torch.uint8, device=dev)
        self.w_scale = torch.empty((N_W, K_W // 16), dtype=torch.uint8, device=dev)
        L.fp4_quant_nvfp4(wb, self.g, self.w_packed, self.w_scale, N_W, K_W)
        del wb
        self.bias = torch.from_numpy(W["bias"].view(np.int16)).to(dev).view(torch.bfloat16)
        self.x = {M: torch.from_numpy(W["X"][M].view(np.int16)).to(dev).view(torch.bfloat16) for M in MS}
        self.b_packed = torch.empty((N_W, K_W // 2), dtype=torch.uint8, device=dev)
        self.b_scale = torch.empty(L.fp4_sf_bytes(N_W, K_W), dtype=torch.uint8, device=dev)
        self.a_packed = {M: torch.empty((M, K_W // 2), dtype=torch.uint8, device=dev) for M in MS}
        self.a_scale = {M: torch.empty(L.fp4_sf_bytes(M, K_W), dtype=torch.uint8, device=dev) for M in MS}
        self.out = {M: torch.empty((M, N_W), dtype=torch.bfloat16, device=dev) for M in MS}
        self.flush_mib = flush_mib
        self.flush_w = torch.empty(max(1, flush_mib) << 20, dtype=torch.uint8, device=dev)
        self.flush_r = torch.ones(max(1, flush_mib) << 20, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.Stream()

    # the kernels of one step
    def requant(self, s):
        self.L.fp4_requant_nvfp4_to_mxfp4(self.w_packed, self.w_scale, self.g, self.b_packed, self.b_scale,
                                          N_W, K_W, stream=s)

    def act(self, M, s):
        self.L.fp4_quant_act_mxfp4(self.x[M], self.a_packed[M], self.a_scale[M], M, K_W, stream=s)

    def gemm(self, M, s):
        self.L.fp4_gemm_mxfp4(self.a_packed[M], self.a_scale[M], self.b_packed, self.b_scale, self.bias,
                              self.out[M], M, N_W, K_W, stream=s)

    def step(self, s):
        self.requant(s)
        for M in MS:
            self.act(M, s)
            self.gemm(M, s)

    def graph(self, fn):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            fn(self.stream)                      # warm (function attributes, module load)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            fn(self.stream)
        torch.cuda.synchronize()
        return g

    def flush(self):
        """Evict L2: write one buffer larger than L2, then read another one."""
        if self.flush_mib > 0:
            with self.torch.cuda.stream(self.stream):
                self.flush_w.fill_(1)
                self.flush_r.sum(dtype=self.torch.int32)

    def time_graph(self, g, reps, flush=True):
        """Mean device ms of one replay, L2 flushed before each replay (outside the events)."""
        torch = self.torch
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        with torch.cuda.stream(self.stream):
            for i in range(reps):
                if flush:
                    self.flush()
                starts[i].record(self.stream)
                g.replay()
                ends[i].record(self.stream)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def run_ours(args):
    import torch

    world, rank, local, pg = dist_setup(args)
    torch.cuda.set_device(local)
    import __graft_entry__

    __graft_entry__.build()
    from nvfp4_mxfp4_w4a4_gb300 import fp4lin as L

    layer = Layer(L, torch, args.flush_mib)
    step_graph = layer.graph(layer.step)
    for _ in range(max(3, args.warmup)):
        layer.flush()
        with torch.cuda.stream(layer.stream):
            step_graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(pg)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    times = layer.time_graph(step_graph, args.steps)
    torch.cuda.synchronize()
    barrier(pg)
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    if L.fp4_get_device_status() != 0:
        raise RuntimeError("device status reports a timeout")

    ms = statistics.fmean(times)
    ms_max = max_over_ranks(pg, ms, device="cuda")
    value = world * step_flops() / (ms_max * 1e-3) / 1e12

    # per-kernel breakdown: each kernel alone as a graph, L2 flushed before each replay
    reps = args.breakdown_reps
    kern = {"requant": (layer.graph(layer.requant), requant_bytes(), 0.0)}
    for M in MS:
        kern[f"act_quant_M{M}"] = (layer.graph(lambda s, M=M: layer.act(M, s)), act_bytes(M), 0.0)
        kern[f"gemm_M{M}"] = (layer.graph(lambda s, M=M: layer.gemm(M, s)), gemm_bytes(M), 2.0 * M * N_W * K_W)
    hbm_peak, peak_kind = peaks()
    breakdown = {}
    for name, (g, nbytes, flops) in kern.items():
        t = statistics.fmean(layer.time_graph(g, reps))
        breakdown[name] = {"us": round(t * 1e3, 2), "GBps": round(nbytes / (t * 1e-3) / 1e9, 1),
                           "hbm_frac": round(nbytes / (t * 1e-3) / 1e9 / hbm_peak, 3)}
        if flops:
            breakdown[name]["TFLOPS"] = round(flops / (t * 1e-3) / 1e12, 2)
            breakdown[name]["pct_fp4_nominal"] = round(100 * flops / (t * 1e-3) / 1e12 / FP4_NOMINAL_TFLOPS, 3)
    total_us = sum(v["us"] for v in breakdown.values())
    for v in breakdown.values():
        v["share"] = round(v["us"] / total_us, 3)
    dom = max(breakdown, key=lambda k: breakdown[k]["us"])
    dom_bytes = kern[dom][1]
    achieved = dom_bytes / (breakdown[dom]["us"] * 1e-6) / 1e9
    traffic = _committed_traffic(dom)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 3), "traffic": traffic,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6800 GB/s"}

    # end to end through the C ABI from pinned host buffers: H2D of the NVFP4
    # weight and the activations, the step, D2H of the outputs
    e2e = _e2e(layer, torch, L, min(args.steps, 50))

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp4 e2m1 (mxfp4) x fp4 -> fp32 acc -> bf16", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "N": N_W, "K": K_W, "M": list(MS), "global_batch": sum(MS),
                   "l2": f"flushed before every timed step ({args.flush_mib} MiB write + {args.flush_mib} MiB "
                         "read of another buffer, outside the events)",
                   "parallelism": f"replicas x{world}", "cuda_graph": True},
        "requant_GBps": breakdown["requant"]["GBps"],
        "gemm_TFLOPS": {M: breakdown[f"gemm_M{M}"]["TFLOPS"] for M in MS},
        "pct_fp4_peak_step": round(100 * value / world / FP4_NOMINAL_TFLOPS, 3),
        "fp4_peak_used": "15000 TFLOPS nominal dense block-scaled FP4 (public Blackwell Ultra figure)",
        "breakdown": breakdown, "roofline": roofline, "e2e": e2e, "gpu_launches": 9 * args.steps,
        "clocks": clk, "wall_s_timed_region": round(t_wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(budget_s=12.0)
    if rank == 0:
        print(json.dumps(result))
    if pg is not None:
        pg.destroy_process_group()


def _committed_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary of this kernel, if any."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get(kernel)
    return None


def _e2e(layer, torch, L, reps):
    dev = torch.device("cuda")
    wp_h = layer.w_packed.cpu().pin_memory()
    ws_h = layer.w_scale.cpu().pin_memory()
    x_h = {M: layer.x[M].cpu().pin_memory() for M in MS}
    out_h = {M: torch.empty((M, N_W), dtype=torch.bfloat16).pin_memory() for M in MS}
    wp_d = torch.empty_like(layer.w_packed)
    ws_d = torch.empty_like(layer.w_scale)
    x_d = {M: torch.empty_like(layer.x[M]) for M in MS}
    s = layer.stream
    h2d = wp_h.numel() + ws_h.numel() + sum(x.numel() * 2 for x in x_h.values())
    d2h = sum(o.numel() * 2 for o in out_h.values())

    def once():
        wp_d.copy_(wp_h, non_blocking=True)
        ws_d.copy_(ws_h, non_blocking=True)
        for M in MS:
            x_d[M].copy_(x_h[M], non_blocking=True)
        L.fp4_requant_nvfp4_to_mxfp4(wp_d, ws_d, layer.g, layer.b_packed, layer.b_scale, N_W, K_W, stream=s)
        for M in MS:
            L.fp4_quant_act_mxfp4(x_d[M], layer.a_packed[M], layer.a_scale[M], M, K_W, stream=s)
            L.fp4_gemm_mxfp4(layer.a_packed[M], layer.a_scale[M], layer.b_packed, layer.b_scale, layer.bias,
                             layer.out[M], M, N_W, K_W, stream=s)
        for M in MS:
            out_h[M].copy_(layer.out[M], non_blocking=True)

    with torch.cuda.stream(s):
        for _ in range(3):
            once()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        layer.flush()
        with torch.cuda.stream(s):
            a.record(s)
            once()
            b.record(s)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.fmean(ts)
    return {"value": round(step_flops() / (ms * 1e-3) / 1e12, 4), "unit": "TFLOPS", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "path": "C ABI, pinned host buffers, H2D + step + D2H inside the events"}


# ------------------------------------------------------------------ CPU oracle
_SAMPLE_CACHE = {}


def _oracle_inputs(rows_w, threads):
    """NVFP4 weight rows and activations for the oracle sample (input
    preparation, not timed).  The global scale is that of the full weight."""
    import oracle
    import synth

    if rows_w not in _SAMPLE_CACHE:
        if "g" not in _SAMPLE_CACHE:
            full = synth.workload1(rows=None)
            _SAMPLE_CACHE["g"] = oracle.nvfp4_global_scale(full["W"])
            del full
        W = synth.workload1(rows=rows_w)
        wp, ws = oracle.nvfp4_quantize(W["W"], _SAMPLE_CACHE["g"], threads=threads)
        _SAMPLE_CACHE[rows_w] = (W, wp, ws)
    return _SAMPLE_CACHE["g"], _SAMPLE_CACHE[rows_w]


def _oracle_sample(rows_w, threads):
    """The oracle on a bounded sample of the step: `rows_w` weight rows are
    requantized and multiplied with all activation rows (M = 1+8+32+64), and
    all activations are quantized.  Returns (seconds, fraction of the step)."""
    import oracle

    g, (W, wp, ws) = _oracle_inputs(rows_w, threads)
    t0 = time.perf_counter()
    bp, bs = oracle.requant(wp, ws, g, threads=threads)
    for M in MS:
        ap, as_ = oracle.act_quant(W["X"][M], threads=threads)
        oracle.gemm(ap, as_, bp, bs, W["bias"][:rows_w], threads=threads)
    dt = time.perf_counter() - t0
    return dt, rows_w / N_W


def cpu_baseline(budget_s=12.0):
    threads = os.cpu_count() or 1
    rows = 128
    dt, frac = _oracle_sample(rows, threads)
    if dt < budget_s / 4:
        rows = int(min(N_W, rows * max(1.0, budget_s / max(dt, 1e-3))))
        rows = max(128, rows // 128 * 128)
        dt, frac = _oracle_sample(rows, threads)
    full_s = dt / frac
    return {"value": round(step_flops() / full_s / 1e12, 6), "unit": "TFLOPS", "cores": threads,
            "kind": "oracle",
            "sample": f"{rows} of {N_W} weight rows requantized and multiplied with all {sum(MS)} activation "
                      f"rows, all activations quantized; step time extrapolated by {N_W}/{rows} "
                      f"({dt:.2f} s measured)"}


def run_reference(args):
    world, rank, local, pg = dist_setup(args)
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    rows = 256
    for _ in range(min(args.warmup, 5)):
        _oracle_sample(rows, threads)
    ts = []
    steps = min(args.steps, 20)      # each step is a bounded sample; cap the run at a few minutes
    for _ in range(steps):
        dt, frac = _oracle_sample(rows, threads)
        ts.append(dt / frac)
    full_s = statistics.fmean(ts)
    value = step_flops() / full_s / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(full_s * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "N": N_W, "K": K_W, "M": list(MS)},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} of {N_W} weight rows per step, extrapolated"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)

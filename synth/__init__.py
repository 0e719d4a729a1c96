"""Seeded synthetic inputs for the W4A4 MXFP4 linear layer.

This module is the only code that both the CUDA path's tests/bench and the
CPU oracle's tests draw from.  It holds no quantization arithmetic: it makes
random numbers, turns them into bf16 tensors, random byte tensors and MoE
routing tables, and nothing else.  NVFP4 weights for the first four
workloads are made from these bf16 tensors by an NVFP4 producer (the oracle
in tests, the library's own producer kernel in the benchmark).

Random numbers: one counter-based generator, SplitMix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014).
Element i of stream (seed, stream) is mix(key + (i + 1) * GOLDEN) with
key = mix(seed * GOLDEN + stream * STREAM_MUL + 1) and mix the SplitMix64
finalizer, all modulo 2^64.  Uniform doubles take the top 53 bits.  Normal
pairs come from Box-Muller over elements (2j, 2j + 1).  Results do not
depend on how the index range is chunked.

Workloads (sizes as the linear layer's (M, N, K); the seed is the index):
  0 tiny:    W[256,512] ~ N(0, 0.02); X[16,512] ~ N(0,1) with 1% of entries x20
  1 decode:  W[14336,4096] ~ N(0, 0.02), 4 of the 4096 K-columns (0.1%) x8;
             X[M,4096] ~ N(0,1) for M in {1, 8, 32, 64}; bias[14336] ~ N(0, 0.01)
  2 prefill: W[18432,7168] ~ N(0, 0.015); X[M,7168] ~ N(0,1) with 0.5% x16,
             M in {2048, 8192}; no bias
  3 MoE:     64 experts, gate_up W[2048,4096] and down W[4096,1024] ~ N(0, 0.02);
             4096 tokens, hidden[4096,4096] ~ N(0,1); router logits [4096,64]
             ~ N(0,1), top-8 per token (ties to the lower expert id); rows
             grouped by (expert, token); the down projection's input is an
             independent [32768,1024] ~ N(0,1) tensor
  4 stream:  60 layers of q,k,v,o [7168,7168] and MLP [18432,7168] NVFP4
             tensors drawn directly as bytes: codes uniform over all 16,
             E4M3 block-scale bytes uniform over 0x38..0x7E (1.0 .. 448),
             global scales log-uniform in [1e-4, 1e-2]; layers 0 and 59 are
             FP8-E4M3 tensors (bytes uniform over the finite codes) that the
             loader passes through unchanged.
"""
from __future__ import annotations

import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
STREAM_MUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# stream ids (one per tensor role)
S_WEIGHT, S_ACT, S_BIAS, S_OUTLIER, S_ROUTER, S_HIDDEN, S_DOWN_IN = 1, 2, 3, 4, 5, 6, 7
S_CODES, S_SCALES, S_GLOBAL, S_FP8 = 8, 9, 10, 11


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.uint64(seed) * GOLDEN + np.uint64(stream) * STREAM_MUL + np.uint64(1)
    return _mix(np.array([z], dtype=np.uint64))[0]


def bits64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Elements [start, start+count) of the stream as uint64."""
    key = _key(seed, stream)
    out = np.empty(count, np.uint64)
    for c0 in range(0, count, _CHUNK):
        c1 = min(count, c0 + _CHUNK)
        idx = np.arange(start + c0 + 1, start + c1 + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            out[c0:c1] = _mix(key + idx * GOLDEN)
    return out


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n doubles in [0, 1)."""
    return (bits64(seed, stream, start, n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def normal(seed: int, stream: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """n standard normals (times sigma) as float64, Box-Muller over pairs."""
    out = np.empty(n, np.float64)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        b = bits64(seed, stream, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
        u1 = ((b[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53   # (0, 1]
        u2 = (b[:, 1] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53           # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1)) * sigma
        t = 2.0 * math.pi * u2
        z = np.empty((p1 - p0, 2), np.float64)
        z[:, 0] = r * np.cos(t)
        z[:, 1] = r * np.sin(t)
        lo, hi = 2 * p0, min(n, 2 * p1)
        out[lo:hi] = z.reshape(-1)[: hi - lo]
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bit patterns (uint16) by the library conversion (round to nearest even)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def random_bytes(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n uniform bytes: the 8 bytes of each 64-bit draw, little-endian, in
    order (byte i is byte i % 8 of draw i // 8).  `start` must be a multiple of 8."""
    assert start % 8 == 0
    draws = bits64(seed, stream, start // 8, (n + 7) // 8)
    return draws.view(np.uint8)[:n].copy()


# ---------------------------------------------------------------- tensors
def bf16_normal(seed, stream, shape, sigma=1.0, outlier_p=0.0, outlier_mul=1.0):
    n = int(np.prod(shape))
    x = normal(seed, stream, n, sigma)
    if outlier_p > 0.0:
        mask = uniform(seed, stream + 100, n) < outlier_p
        x = np.where(mask, x * outlier_mul, x)
    return to_bf16_bits(x).reshape(shape)


def weight_with_column_outliers(seed, shape, sigma, n_cols, mul, rows=None):
    """Weight ~N(0, sigma) with n_cols seeded K-columns (all rows) scaled by mul.
    `rows` limits generation to the first rows (same values as the full tensor)."""
    N, K = shape
    N = N if rows is None else rows
    x = normal(seed, S_WEIGHT, N * K, sigma).reshape(N, K)
    cols = np.sort(np.argsort(uniform(seed, S_OUTLIER, K), kind="stable")[:n_cols])
    x[:, cols] *= mul
    return to_bf16_bits(x), cols


def workload0():
    W = bf16_normal(0, S_WEIGHT, (256, 512), 0.02)
    X = bf16_normal(0, S_ACT, (16, 512), 1.0, 0.01, 20.0)
    return {"W": W, "X": X, "bias": None}


def workload1(Ms=(1, 8, 32, 64), rows=None):
    W, cols = weight_with_column_outliers(1, (14336, 4096), 0.02, 4, 8.0, rows)
    Xs = {M: bf16_normal(1, S_ACT * 1000 + M, (M, 4096), 1.0) for M in Ms}
    bias = bf16_normal(1, S_BIAS, (14336,), 0.01)
    return {"W": W, "X": Xs, "bias": bias, "outlier_cols": cols}


def workload2(Ms=(2048, 8192)):
    W = bf16_normal(2, S_WEIGHT, (18432, 7168), 0.015)
    Xs = {M: bf16_normal(2, S_ACT * 1000 + M, (M, 7168), 1.0, 0.005, 16.0) for M in Ms}
    return {"W": W, "X": Xs, "bias": None}


def moe_routing(seed, T, E, topk):
    """Router logits ~N(0,1) -> top-k experts per token (softmax order == logit
    order; ties go to the lower expert id).  Returns the row -> token map of
    the (expert, token)-sorted grouping and row_offsets[E+1]."""
    logits = normal(seed, S_ROUTER, T * E).astype(np.float32).reshape(T, E)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :topk]          # [T, topk]
    tok = np.repeat(np.arange(T, dtype=np.int64), topk)
    exp = order.reshape(-1).astype(np.int64)
    perm = np.lexsort((tok, exp))                                         # by expert, then token
    row_token = tok[perm]
    counts = np.bincount(exp, minlength=E)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    return row_token, offsets.astype(np.int32), logits


def workload3(E=64, T=4096, topk=8, H=4096, I=1024, N_gu=2048, experts=None):
    """MoE grouped GEMM inputs.  `experts` limits which experts' weights are
    generated (all by default); each expert's weight uses its own stream."""
    row_token, offsets, _ = moe_routing(3, T, E, topk)
    hidden = bf16_normal(3, S_HIDDEN, (T, H), 1.0)
    A_gu = hidden[row_token]
    A_down = bf16_normal(3, S_DOWN_IN, (T * topk, I), 1.0)
    experts = range(E) if experts is None else experts
    W_gu = {e: bf16_normal(3, S_WEIGHT * 1000 + 2 * e, (N_gu, H), 0.02) for e in experts}
    W_down = {e: bf16_normal(3, S_WEIGHT * 1000 + 2 * e + 1, (H, I), 0.02) for e in experts}
    return {"row_offsets": offsets, "row_token": row_token, "A_gu": A_gu, "A_down": A_down,
            "W_gu": W_gu, "W_down": W_down}


# ------------------------------------------------------ layer-stream workload
LAYERS4 = 60
HIDDEN4 = 7168
MLP4 = 18432
EXCLUDED4 = (0, 59)
TENSORS4 = (("q", HIDDEN4), ("k", HIDDEN4), ("v", HIDDEN4), ("o", HIDDEN4), ("mlp", MLP4))


def workload4_tensor(layer: int, t_idx: int, rows: int | None = None):
    """One NVFP4 tensor of layer `layer` (direct byte draw), or the FP8 bytes of
    an excluded layer.  Returns dict(kind, packed, scale, g) / dict(kind, fp8, scale)."""
    name, N = TENSORS4[t_idx]
    K = HIDDEN4
    N = N if rows is None else rows
    stream = (layer * 16 + t_idx) * 64
    if layer in EXCLUDED4:
        b = random_bytes(4, S_FP8 * 100000 + stream, N * K)
        b = np.where((b & 0x7F) == 0x7F, b & 0xFE, b).astype(np.uint8)    # drop the NaN codes
        return {"kind": "fp8", "fp8": b.reshape(N, K), "scale": float(2.0 ** -6)}
    packed = random_bytes(4, S_CODES * 100000 + stream, N * K // 2).reshape(N, K // 2)
    sc = random_bytes(4, S_SCALES * 100000 + stream, N * K // 16)
    scale = (0x38 + (sc.astype(np.uint32) % (0x7E - 0x38 + 1))).astype(np.uint8).reshape(N, K // 16)
    u = uniform(4, S_GLOBAL * 100000 + stream, 1)[0]
    g = float(np.float32(10.0 ** (-4.0 + 2.0 * u)))
    return {"kind": "nvfp4", "packed": packed, "scale": scale, "g": g}

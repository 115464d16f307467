"""Seeded synthetic inputs, shared by the tests, the bench and the smoke check.

This module holds random-number generation and BF16 packing only: none of the
quantize-or-GEMM arithmetic.  Both the oracle and the CUDA path receive the
exact bytes made here.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: the i-th draw of a stream
with start state s is mix(s + (i + 1) * 0x9E3779B97F4A7C15).  A stream's start
state is seed * 2**32 + stream id.  Uniforms take the top 53 bits; normals use
the Box-Muller transform on consecutive uniform pairs (cosine and sine
branches fill consecutive outputs).  FP32 values are cast to BF16 with
round-to-nearest-even.

Workload shapes (dense 8B-class MLP, 30B-A3B-class MoE) and value
distributions follow the configurations the repository measures: activations
~N(0,1) with 0.1% of entries multiplied by 50, weights ~N(0,0.02), output
gradients ~N(0,1e-3), with sigma read as the standard deviation.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids (one per synthetic tensor role)
STREAM = {
    "x": 1, "h": 2, "dy_gate": 3, "dy_up": 4, "dy_down": 5,
    "w_gate": 11, "w_up": 12, "w_down": 13, "w": 14, "dy": 15,
    "outlier": 100, "route": 200, "test": 300,
}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _start(seed: int, stream: int) -> np.uint64:
    return np.uint64(((int(seed) << 32) + int(stream)) & 0xFFFFFFFFFFFFFFFF)


def raw_u64(n: int, seed: int, stream: int, first: int = 0) -> np.ndarray:
    """Draws first .. first+n-1 of a SplitMix64 stream."""
    with np.errstate(over="ignore"):
        i = np.arange(first + 1, first + n + 1, dtype=np.uint64)
        return _mix(_start(seed, stream) + i * GAMMA)


def uniform(n: int, seed: int, stream: int, first: int = 0) -> np.ndarray:
    """Uniform binary64 numbers in [0, 1)."""
    return (raw_u64(n, seed, stream, first) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(n: int, seed: int, stream: int, std: float = 1.0, chunk: int = 1 << 24) -> np.ndarray:
    """n normal deviates (float32) with the given standard deviation."""
    out = np.empty(n, np.float32)
    pairs = (n + 1) // 2
    for p0 in range(0, pairs, chunk):
        p1 = min(pairs, p0 + chunk)
        u = uniform(2 * (p1 - p0), seed, stream, first=2 * p0)
        r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        t = 2.0 * np.pi * u[1::2]
        z = np.empty(2 * (p1 - p0), np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        lo, hi = 2 * p0, min(n, 2 * p1)
        out[lo:hi] = (z[: hi - lo] * std).astype(np.float32)
    return out


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_positions(numel: int, frac: float, seed: int, stream: int) -> np.ndarray:
    """round(frac * numel) distinct positions, uniform, in draw order."""
    k = int(round(frac * numel))
    if k == 0:
        return np.zeros(0, np.int64)
    got = np.zeros(0, np.int64)
    first = 0
    while True:
        m = int(k * 1.25) + 64
        cand = np.minimum((uniform(m, seed, stream, first) * numel).astype(np.int64), numel - 1)
        first += m
        allc = np.concatenate([got, cand])
        _, idx = np.unique(allc, return_index=True)
        got = allc[np.sort(idx)]
        if len(got) >= k:
            return got[:k]


def activation(rows: int, cols: int, seed: int = 0, stream: str | int = "x",
               outlier_frac: float = 0.001, outlier_mult: float = 50.0) -> np.ndarray:
    """BF16 [rows x cols] ~N(0,1) with a fraction of entries scaled by outlier_mult."""
    sid = STREAM[stream] if isinstance(stream, str) else int(stream)
    v = normal(rows * cols, seed, sid)
    pos = outlier_positions(rows * cols, outlier_frac, seed, STREAM["outlier"] + sid)
    v[pos] *= np.float32(outlier_mult)
    return bf16_bits(v).reshape(rows, cols)


def weight(rows: int, cols: int, seed: int = 0, stream: str | int = "w", std: float = 0.02) -> np.ndarray:
    sid = STREAM[stream] if isinstance(stream, str) else int(stream)
    return bf16_bits(normal(rows * cols, seed, sid, std)).reshape(rows, cols)


def gradient(rows: int, cols: int, seed: int = 0, stream: str | int = "dy", std: float = 1e-3) -> np.ndarray:
    sid = STREAM[stream] if isinstance(stream, str) else int(stream)
    return bf16_bits(normal(rows * cols, seed, sid, std)).reshape(rows, cols)


def zipf_topk_routing(tokens: int, experts: int, k: int, s: float, seed: int = 0):
    """Top-k routing with Zipf(s) expert popularity, by Gumbel-top-k.

    Expert r-1 has rank r and weight r**-s.  Each token draws k distinct experts
    (the k largest of log w + Gumbel noise).  Returns (offsets [experts+1],
    token_of_row [tokens*k]) for rows sorted by expert (stable in token order).
    """
    logw = -s * np.log(np.arange(1, experts + 1, dtype=np.float64))
    u = uniform(tokens * experts, seed, STREAM["route"]).reshape(tokens, experts)
    g = -np.log(-np.log(np.clip(u, 1e-300, None)))
    choice = np.argsort(-(logw[None, :] + g), axis=1, kind="stable")[:, :k]
    expert_of_row = choice.reshape(-1)
    token_of_row = np.repeat(np.arange(tokens, dtype=np.int64), k)
    order = np.argsort(expert_of_row, kind="stable")
    counts = np.bincount(expert_of_row, minlength=experts)
    offsets = np.zeros(experts + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    return offsets, token_of_row[order]

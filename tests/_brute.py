"""Brute-force helpers for pinning the oracle (test code only).

These restate the E4M3 format and the group quantizer in the most literal way
available (exhaustive nearest-value search, numpy float32 arithmetic) so that
they share no algorithm with ``oracle/jetq_oracle.c`` (binary search against
exact midpoints).
"""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def e4m3_positive_values():
    """Value of codes 0x00..0x7E, from the OCP definition (bias 7, 3 mantissa bits)."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


_POS = e4m3_positive_values()


def brute_encode(v):
    """Nearest finite E4M3 code by exhaustive search; equal distance -> even code."""
    v = np.asarray(v, dtype=np.float64)
    # beyond 512 every finite code is farther than 448 is; clipping keeps the
    # distances exact in binary64
    a = np.minimum(np.abs(v), 512.0).reshape(-1, 1)
    d = np.abs(a - _POS[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among the (at most two) nearest codes prefer the even one
    even = cand & ((np.arange(0x7F) % 2) == 0)[None, :]
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    sign = np.signbit(v.reshape(-1)).astype(np.uint8) << 7
    return (pick.astype(np.uint8) | sign).reshape(v.shape)


def bf16_f32(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def brute_group(x_bf16):
    """One FP32-scale group: S = fl32(amax/448), q = E4M3(fl32(x/S)) via numpy float32."""
    x = bf16_f32(x_bf16)
    a = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    s = np.float32(a) / np.float32(448.0)
    if s == 0:
        return np.zeros(x.shape, np.uint8), s
    with np.errstate(all="ignore"):
        return brute_encode((x / s).astype(np.float32)), s


def brute_mx_group(x_bf16):
    """One MX group: e = smallest integer with amax <= 448*2^e (search), q = E4M3(x*2^-e)."""
    x = bf16_f32(x_bf16).astype(np.float64)
    a = float(np.max(np.abs(x))) if x.size else 0.0
    if a == 0.0:
        return np.zeros(x.shape, np.uint8), 127
    e = -200
    while a > 448.0 * 2.0 ** e:
        e += 1
    e = max(-127, min(127, e))
    return brute_encode(x * 2.0 ** (-e)), e + 127

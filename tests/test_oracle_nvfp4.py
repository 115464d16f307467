"""Pins for the oracle's NVFP4 quantizer (E2M1 values, E4M3 scale per 16-value
block, FP32 scope scale per token or per tensor), checked against the E2M1
definition, closed forms and invariants rather than against itself."""
import math
import os

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_points.txt")


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_e2m1_code_points_match_the_format():
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        code, value = line.split()
        got = oracle.e2m1_decode([int(code, 16)])[0]
        assert got == float(value) and math.copysign(1, got) == math.copysign(1, float(value)), code


def test_e2m1_rounding_ties_to_even_and_saturates():
    # midpoints of the grid 0, .5, 1, 1.5, 2, 3, 4, 6 go to the code with the even last bit
    ties = {0.25: 0x0, 0.75: 0x2, 1.25: 0x2, 1.75: 0x4, 2.5: 0x4, 3.5: 0x6, 5.0: 0x6}
    for v, code in ties.items():
        assert oracle.e2m1_encode([v])[0] == code, v
        assert oracle.e2m1_encode([-v])[0] == code | 8, v
        lo, hi = np.nextafter(v, 0.0), np.nextafter(v, 10.0)
        assert oracle.e2m1_encode([lo])[0] == oracle.e2m1_encode([v - 1e-6])[0]
        assert oracle.e2m1_encode([hi])[0] == oracle.e2m1_encode([v + 1e-6])[0]
        assert oracle.e2m1_encode([lo])[0] != oracle.e2m1_encode([hi])[0]
    assert oracle.e2m1_encode([6.5, 1e30, -7.0])[0] == 0x7
    assert oracle.e2m1_encode([-7.0])[0] == 0xF
    assert oracle.e2m1_encode([0.0])[0] == 0x0 and oracle.e2m1_encode([-0.0])[0] == 0x8
    # every code value encodes to itself
    vals = oracle.e2m1_decode(np.arange(16))
    assert np.array_equal(oracle.e2m1_encode(vals), np.arange(16, dtype=np.uint8))


def _unpack(q):
    c = np.empty((q.shape[0], q.shape[1] * 2), np.uint8)
    c[:, 0::2], c[:, 1::2] = q & 15, q >> 4
    return c


def test_exact_reconstruction_of_representable_rows():
    """Rows built as e2m1 * E4M3 * 2^-6 with each block's maximum 6 * E4M3 * 2^-6 and
    the row maximum 6 * 448 * 2^-6 = 42: the scope scale is 2^-6, every block scale
    and code is recovered, and dequantization returns the input exactly."""
    rng = np.random.default_rng(3)
    e4m3_vals = oracle.e4m3_decode(np.arange(1, 0x7F))  # positive finite scales
    grid = oracle.e2m1_decode(np.arange(16))
    R, B = 6, 8
    x = np.empty((R, 16 * B), np.float64)
    for r in range(R):
        scales = rng.choice(e4m3_vals[e4m3_vals >= 2.0 ** -3], B)
        scales[rng.integers(B)] = 448.0
        for b in range(B):
            vals = rng.choice(grid, 16)
            vals[rng.integers(16)] = 6.0 * rng.choice([-1.0, 1.0])
            x[r, 16 * b:16 * b + 16] = vals * scales[b] * 2.0 ** -6
    xb = synth.bf16_bits(x.astype(np.float32))
    assert np.array_equal(_f32(xb), x)  # every input is a BF16 value
    q, sb, sg = oracle.quant_nvfp4(xb)
    assert np.all(sg == np.float32(2.0 ** -6))
    assert np.array_equal(oracle.dequant_nvfp4(q, sb, sg), x)
    assert np.array_equal(oracle.dequant_nvfp4_bf16(q, sb, sg), xb)


def test_reconstruction_error_within_half_an_e2m1_step():
    x = synth.activation(64, 256, seed=21, stream="test")
    xv = _f32(x)
    q, sb, sg = oracle.quant_nvfp4(x)
    amax = np.abs(xv).max(axis=1)
    # the scope scale maps the row maximum to 6 * 448 (within binary32 rounding)
    assert np.all(np.abs(sg.astype(np.float64) * 2688.0 - amax) <= 2.0 ** -22 * amax)
    D = np.repeat(oracle.e4m3_decode(sb), 16, axis=1) * sg[:, None].astype(np.float64)
    v = xv / D
    deq = oracle.dequant_nvfp4(q, sb, sg) / D
    a = np.abs(v)
    half = np.where(a < 2.0, 0.25, np.where(a < 4.0, 0.5, 1.0))
    err = np.abs(v - deq)
    assert np.all((err <= half * (1 + 1e-6)) | ((a > 6.0) & (np.abs(deq) == 6.0)))
    # each block's largest element lands on 4 or 6 (the block scale is its max / 6, rounded to E4M3)
    blk = np.abs(deq).reshape(64, -1, 16).max(axis=2)
    assert np.all(blk >= 4.0)
    assert np.all(np.sign(deq[np.abs(deq) > 0]) == np.sign(xv[np.abs(deq) > 0]))


def test_tensor_scope_and_zero_cases():
    x = synth.activation(8, 64, seed=22, stream="test")
    amax = float(np.abs(_f32(x)).max()) * 2.0  # a shared scope wider than this tensor (gate/up pair)
    q, sb, sg = oracle.quant_nvfp4(x, scope_amax=amax)
    assert sg.shape == (1,) and sg[0] == np.float32(np.float32(amax) / np.float32(2688.0))
    assert np.all(np.abs(oracle.dequant_nvfp4(q, sb, sg)) <= amax)
    z = np.zeros((3, 32), np.uint16)
    z[1] = 0x8000
    q, sb, sg = oracle.quant_nvfp4(z)
    assert not q.any() and not sb.any() and not sg.any()
    # a block far below its row's maximum: block scale 0, codes 0
    y = np.zeros((1, 32), np.float32)
    y[0, 0], y[0, 16] = 1.0, 1e-9
    q, sb, sg = oracle.quant_nvfp4(synth.bf16_bits(y))
    assert sb[0, 1] == 0 and not (q[0, 8:] & 0x77).any()


def test_dequant_bf16_rounds_the_exact_product_once():
    # code 0x3 (1.5) with block scale 1.0 (E4M3 0x38) and S = 1 + 2^-7: the product
    # 1.5 + 3 * 2^-8 lies exactly halfway between the BF16 values 0x3FC1 and 0x3FC2,
    # and goes to the even one; one step of S higher it rounds up, one lower down
    q = np.full((1, 8), 0x33, np.uint8)
    sb = np.full((1, 1), 0x38, np.uint8)
    s = np.float32(1.0 + 2.0 ** -7)
    assert np.all(oracle.dequant_nvfp4_bf16(q, sb, np.array([s], np.float32)) == 0x3FC2)
    up = np.nextafter(s, np.float32(2.0))
    down = np.nextafter(s, np.float32(0.0))
    assert np.all(oracle.dequant_nvfp4_bf16(q, sb, np.array([up], np.float32)) == 0x3FC2)
    assert np.all(oracle.dequant_nvfp4_bf16(q, sb, np.array([down], np.float32)) == 0x3FC1)


def test_dequant_fp64_hand_values_and_bf16_relation():
    """Hand values of the binary64 dequantizer (code x E4M3 scale x scope scale), the
    nibble order (element 2j in the low nibble) and the per-row / per-tensor scope; its
    BF16 rounding is the BF16 dequantizer's output."""
    # byte 0x5A: element 0 = code 0xA (-1.0), element 1 = code 0x5 (3.0)
    q = np.array([[0x5A] + [0x00] * 7, [0x71] + [0xFF] * 7], np.uint8)
    sb = np.array([[0x40], [0x30]], np.uint8)   # E4M3 0x40 = 2.0, 0x30 = 0.5
    sg = np.array([0.25, 3.0], np.float32)
    d = oracle.dequant_nvfp4(q, sb, sg)
    assert d[0, 0] == -1.0 * 2.0 * 0.25 and d[0, 1] == 3.0 * 2.0 * 0.25 and not d[0, 2:].any()
    assert d[1, 0] == 0.5 * 0.5 * 3.0 and d[1, 1] == 6.0 * 0.5 * 3.0 and np.all(d[1, 2:] == -6.0 * 0.5 * 3.0)
    dt = oracle.dequant_nvfp4(q, sb, np.array([0.25], np.float32))  # one tensor scope for every row
    assert dt[1, 1] == 6.0 * 0.5 * 0.25
    x = synth.activation(16, 128, seed=23, stream="test")
    q, sb, sg = oracle.quant_nvfp4(x)
    # binary64 -> BF16 rounded once (nearest, ties to even on the 7 kept fraction bits);
    # the values are normal binary32 numbers, so the rounded double converts exactly
    u = oracle.dequant_nvfp4(q, sb, sg).view(np.uint64)
    lsb = (u >> np.uint64(45)) & np.uint64(1)
    r = ((u + np.uint64((1 << 44) - 1) + lsb) >> np.uint64(45)) << np.uint64(45)
    assert np.array_equal(synth.bf16_bits(r.view(np.float64).astype(np.float32)),
                          oracle.dequant_nvfp4_bf16(q, sb, sg))

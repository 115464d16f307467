"""Pins for the oracle's quantizers and dequantizers (no GPU).

Each quantizer is pinned by brute force on small cases (numpy float32
arithmetic plus exhaustive E4M3 search), by the invariants the format fixes
(|q| <= 448, the group maximum maps to +-448, S*448 = amax up to one rounding,
MX: 448*2^(e-1) < amax <= 448*2^e), by exact reconstruction of inputs that are
already E4M3 values times a power of two, and by layout identities (column
copy = row copy of the transpose, transposed weight copy = transposed bytes).
The four input classes (random, boundary, zeros, maxes) follow the byte-exact
quantizer tests described in the Miles Blackwell-recipes post.
"""
import numpy as np
import pytest

import oracle
import synth
from _brute import bf16_f32, brute_encode, brute_group, brute_mx_group, e4m3_positive_values


def _bits(f32):
    return synth.bf16_bits(np.asarray(f32, dtype=np.float32))


def _random_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return _bits(rng.standard_normal(shape) * scale)


def _boundary_bf16(rows, cols, seed, gs=128):
    """Groups whose max is 448*2^k (so S = 2^k exactly) and whose other entries sit
    on E4M3 rounding midpoints (times 2^k) or one BF16 step either side."""
    rng = np.random.default_rng(seed)
    pos = e4m3_positive_values()
    mids = 0.5 * (pos[1:] + pos[:-1])
    out = np.empty((rows, cols), np.uint16)
    for r in range(rows):
        for g in range(cols // gs):
            k = int(rng.integers(-20, 20))
            v = rng.choice(mids, gs) * rng.choice([-1.0, 1.0], gs) * 2.0 ** k
            b = _bits(v)
            b = (b.astype(np.int32) + rng.integers(-1, 2, gs)).astype(np.uint16)  # +-1 BF16 ulp
            b[rng.integers(gs)] = _bits([448.0 * 2.0 ** k])[0]
            out[r, g * gs:(g + 1) * gs] = b
    return out


def _check_rowgroups_brute(x, gs):
    q, s = oracle.quant_rowgroups(x, gs)
    R, C = x.shape
    for r in range(R):
        for g in range(C // gs):
            bq, bs = brute_group(x[r, g * gs:(g + 1) * gs])
            assert s[g, r] == bs or (np.isnan(s[g, r]) and np.isnan(bs))
            assert np.array_equal(q[r, g * gs:(g + 1) * gs], bq), (r, g)
    return q, s


@pytest.mark.parametrize("kind", ["random", "boundary", "zeros", "maxes"])
def test_rowgroups_brute_force_four_classes(kind):
    R, C = 6, 256
    if kind == "random":
        x = _random_bf16((R, C), 1, 3.0)
        x[0, :128] = _random_bf16((1, 128), 9, 1e-30)  # tiny magnitudes
    elif kind == "boundary":
        x = _boundary_bf16(R, C, 2)
    elif kind == "zeros":
        x = np.zeros((R, C), np.uint16)
        x[1] = 0x8000  # -0.0 everywhere: still an all-zero group
    else:
        x = np.where(np.random.default_rng(3).random((R, C)) < 0.5, 0x7F7F, 0xFF7F).astype(np.uint16)
        x[2] = _bits(np.full(C, 448.0 * 2.0 ** 5))
    q, s = _check_rowgroups_brute(x, 128)
    if kind == "zeros":
        assert np.all(q == 0) and np.all(s == 0)


def test_rowgroups_small_group_sizes_brute():
    x = _random_bf16((5, 24), 4, 10.0)
    for gs in (1, 2, 3, 4, 8, 24):
        _check_rowgroups_brute(x, gs)


def test_rowgroup_invariants():
    x = synth.activation(64, 512, seed=0, stream="test")
    q, s = oracle.quant_rowgroups(x)
    deq = oracle.e4m3_decode(q)
    assert np.all(np.abs(deq) <= 448)
    xf = bf16_f32(x).astype(np.float64)
    for g in range(4):
        blk = np.abs(xf[:, g * 128:(g + 1) * 128])
        amax = blk.max(axis=1)
        # S*448 equals the group maximum up to the one rounding of the division
        assert np.all(np.abs(s[g].astype(np.float64) * 448 - amax) <= 2.0 ** -24 * amax + 1e-300)
        # the element(s) that reach the maximum encode to +-448
        hit = blk == amax[:, None]
        assert np.all(np.isin(q[:, g * 128:(g + 1) * 128][hit], [0x7E, 0xFE]))


def test_exact_reconstruction_of_representable_groups():
    rng = np.random.default_rng(5)
    pos = e4m3_positive_values()
    R, C = 8, 256
    x = np.empty((R, C), np.float64)
    ks = rng.integers(-30, 30, size=(R, C // 128))
    for r in range(R):
        for g in range(C // 128):
            v = rng.choice(pos, 128) * rng.choice([-1.0, 1.0], 128)
            v[rng.integers(128)] = 448.0 * rng.choice([-1.0, 1.0])
            x[r, g * 128:(g + 1) * 128] = v * 2.0 ** ks[r, g]
    xb = _bits(x)
    assert np.array_equal(bf16_f32(xb).astype(np.float64), x)
    q, s = oracle.quant_rowgroups(xb)
    assert np.array_equal(s.T, (2.0 ** ks).astype(np.float32))
    assert np.array_equal(oracle.dequant_rowgroups(q, s), x)


def test_batch_invariance_of_row_copy():
    x = synth.activation(40, 256, seed=1, stream="test")
    q, s = oracle.quant_rowgroups(x)
    for sub in (slice(0, 1), slice(3, 11), slice(17, 40)):
        qs, ss = oracle.quant_rowgroups(x[sub])
        assert np.array_equal(qs, q[sub]) and np.array_equal(ss, s[:, sub])


def test_colgroups_is_rowgroups_of_transpose():
    x = synth.activation(256, 384, seed=2, stream="test")
    qc, sc = oracle.quant_colgroups(x)
    qr, sr = oracle.quant_rowgroups(np.ascontiguousarray(x.T))
    assert np.array_equal(qc, qr) and np.array_equal(sc, sr)


def test_colgroups_segments_and_partial_groups():
    x = synth.activation(300, 256, seed=3, stream="test")
    off = [0, 5, 5, 133, 300]  # includes an empty segment and ragged tails
    qc, sc = oracle.quant_colgroups(x, offsets=off)
    P = oracle.colcopy_length(off, 300)
    assert P == 128 + 0 + 128 + 256 and qc.shape == (256, P)
    starts = [0, 128, 128, 256]
    for e in range(4):
        n = off[e + 1] - off[e]
        if n == 0:
            continue
        seg = x[off[e]:off[e + 1]]
        # brute force, group by group
        for t in range(0, n, 128):
            grp = seg[t:t + 128]
            for c in (0, 77, 255):
                bq, bs = brute_group(grp[:, c])
                col = starts[e] + t
                assert sc[col // 128, c] == bs
                assert np.array_equal(qc[c, col:col + len(grp)], bq)
                assert np.all(qc[c, col + len(grp):col + 128] == 0)
    deq = oracle.dequant_colgroups(qc, sc, 300, offsets=off)
    xf = bf16_f32(x).astype(np.float64)
    assert np.all(np.abs(deq - xf) <= 2.0 ** -4 * np.abs(xf) + 1e-3 * np.abs(xf).max())
    # exactly decode(code) * S of the token's own group: row i of segment e is position
    # starts[e] + i of the copy, scaled by that 128-position group's scale of its column
    dec = oracle.e4m3_decode(np.arange(256))
    for e in range(4):
        for i in range(off[e + 1] - off[e]):
            pos = starts[e] + i
            want = dec[qc[:, pos]] * sc[pos // 128].astype(np.float64)
            assert np.array_equal(deq[off[e] + i], want), (e, i)


def test_blocks_brute_and_transpose():
    w = _random_bf16((8, 12), 6, 0.02)
    q, s, qT, sT = oracle.quant_blocks(w, bs=4)
    for bi in range(2):
        for bj in range(3):
            bq, bsc = brute_group(w[bi * 4:(bi + 1) * 4, bj * 4:(bj + 1) * 4])
            assert s[bi, bj] == bsc
            assert np.array_equal(q[bi * 4:(bi + 1) * 4, bj * 4:(bj + 1) * 4], bq)
    assert np.array_equal(qT, q.T) and np.array_equal(sT, s.T)


def test_blocks_full_size_invariants():
    w = synth.weight(256, 384, seed=0)
    q, s, qT, sT = oracle.quant_blocks(w)
    assert np.array_equal(qT, q.T) and np.array_equal(sT, s.T)
    wf = bf16_f32(w).astype(np.float64)
    amax = np.abs(wf).reshape(2, 128, 3, 128).max(axis=(1, 3))
    assert np.all(np.abs(s * 448.0 - amax) <= 2.0 ** -24 * amax)
    deq = oracle.dequant_blocks(q, s)
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 in the normal range, and
    # at most half the subnormal step (2^-10 * S) below it
    S = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)
    assert np.all(np.abs(deq - wf) <= np.maximum(2.0 ** -4 * np.abs(wf), 2.0 ** -10 * S))


# ----------------------------------------------------------------------------- MX

def test_e8m0_exponent_brackets_amax():
    for k in range(-120, 120, 7):
        top = 448.0 * 2.0 ** k
        assert oracle.e8m0_exponent(np.float32(top)) == k  # exactly at the bound: no round-up
        assert oracle.e8m0_exponent(np.float32(np.nextafter(np.float32(top), np.float32(np.inf)))) == k + 1
        assert oracle.e8m0_exponent(np.float32(np.nextafter(np.float32(top), np.float32(0)))) == k
    rng = np.random.default_rng(7)
    for a in np.exp(rng.uniform(-80, 80, 500)).astype(np.float32):
        e = oracle.e8m0_exponent(a)
        assert 448.0 * 2.0 ** (e - 1) < float(a) <= 448.0 * 2.0 ** e
    assert oracle.e8m0_exponent(np.float32(1e-45)) == -127  # clamped
    assert oracle.e8m0_exponent(np.float32(0)) == 0


@pytest.mark.parametrize("kind", ["random", "boundary", "zeros", "maxes"])
def test_mx_rows_brute_force_four_classes(kind):
    R, C = 4, 128
    if kind == "random":
        x = _random_bf16((R, C), 8, 5.0)
    elif kind == "boundary":
        x = _boundary_bf16(R, C, 9, gs=32)
    elif kind == "zeros":
        x = np.zeros((R, C), np.uint16)
    else:
        x = np.full((R, C), 0x7F7F, np.uint16)
        x[1::2] = 0xFF7F
    q, e8 = oracle.quant_mx_rows(x)
    for r in range(R):
        for g in range(C // 32):
            bq, be = brute_mx_group(x[r, g * 32:(g + 1) * 32])
            assert e8[r, g] == be and np.array_equal(q[r, g * 32:(g + 1) * 32], bq), (r, g)


def test_mx_exact_reconstruction_including_sub_max_blocks():
    rng = np.random.default_rng(10)
    pos = e4m3_positive_values()
    R, C = 4, 256
    x = np.empty((R, C))
    for r in range(R):
        for g in range(C // 32):
            k = int(rng.integers(-40, 40))
            v = rng.choice(pos[pos <= 256], 32) * rng.choice([-1.0, 1.0], 32)
            if g % 2 == 0:
                v[rng.integers(32)] = 448.0  # block max exactly 448*2^k
            x[r, g * 32:(g + 1) * 32] = v * 2.0 ** k
    xb = _bits(x)
    q, e8 = oracle.quant_mx_rows(xb)
    assert np.array_equal(oracle.dequant_mx_rows(q, e8), x)


def test_mx_cols_is_rows_of_transpose_and_segments():
    x = synth.activation(256, 128, seed=4, stream="test")
    qc, e8c = oracle.quant_mx_cols(x)
    qr, e8r = oracle.quant_mx_rows(np.ascontiguousarray(x.T))
    assert np.array_equal(qc, qr) and np.array_equal(e8c, e8r)
    off = [0, 40, 40, 200, 256]
    qc, e8c = oracle.quant_mx_cols(x, offsets=off)
    assert qc.shape == (128, 128 + 256 + 128)
    # segment 1 (rows 40..199) starts at column 128: blocks of 32 inside it
    seg = x[40:200]
    for t in range(0, 160, 32):
        for c in (0, 63):
            bq, be = brute_mx_group(seg[t:t + 32, c])
            assert e8c[c, (128 + t) // 32] == be
            assert np.array_equal(qc[c, 128 + t:128 + t + 32], bq)
    # fully padded blocks after segment 0 (40 rows -> blocks 2,3 empty): scale 1, codes 0
    assert np.all(e8c[:, 2:4] == 127) and np.all(qc[:, 40:128] == 0)
    deq = oracle.dequant_mx_cols(qc, e8c, 256, offsets=off)
    xf = bf16_f32(x).astype(np.float64)
    assert np.all(np.abs(deq - xf) <= 2.0 ** -4 * np.abs(xf) + 2.0 ** -9 * np.abs(xf).max())


# ---------------------------------------------------------------- power-of-two blocks
# The blockwise recipe with FP32 scales constrained to powers of two (SkyRL,
# "Deep dive: FP8 quantization with FP32 and power-of-two block scales"): the
# exponent rule is the MX one, applied to 1 x 128 groups (quant_mx_rows with
# bs = 128) and to 128 x 128 weight blocks (quant_blocks_pow2).


@pytest.mark.parametrize("kind", ["random", "boundary", "zeros", "maxes"])
def test_pow2_rows_of_128_brute_force(kind):
    R, C = 3, 256
    if kind == "random":
        x = _random_bf16((R, C), 21, 5.0)
    elif kind == "boundary":
        x = _boundary_bf16(R, C, 22, gs=128)
    elif kind == "zeros":
        x = np.zeros((R, C), np.uint16)
    else:
        x = np.full((R, C), 0x7F7F, np.uint16)
        x[1::2] = 0xFF7F
    q, e8 = oracle.quant_mx_rows(x, bs=128)
    assert e8.shape == (R, 2)
    for r in range(R):
        for g in range(2):
            bq, be = brute_mx_group(x[r, g * 128:(g + 1) * 128])
            assert e8[r, g] == be and np.array_equal(q[r, g * 128:(g + 1) * 128], bq), (r, g)


def test_pow2_blocks_brute_force_and_transpose():
    # two 128 x 128 blocks per side, one all zero, one with an outlier block
    w = synth.weight(256, 256, seed=23, stream="test")
    w[128:, :128] = 0
    w[:128, 128:] = synth.activation(128, 128, seed=23, stream="test")
    q, e8, qT, e8T = oracle.quant_blocks_pow2(w)
    assert np.array_equal(qT, q.T) and np.array_equal(e8T, e8.T)
    for bi in range(2):
        for bj in range(2):
            blk = w[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            bq, be = brute_mx_group(blk.reshape(-1))
            assert e8[bi, bj] == be, (bi, bj)
            assert np.array_equal(q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128], bq.reshape(128, 128))
    assert e8[1, 0] == 127 and not q[128:, :128].any()  # zero block: scale 1, codes 0


def test_pow2_blocks_exact_reconstruction_and_exponent_bracket():
    rng = np.random.default_rng(24)
    pos = e4m3_positive_values()
    x = np.empty((256, 128))
    for bi, k in enumerate((-20, 13)):
        v = rng.choice(pos[pos <= 448], (128, 128)) * rng.choice([-1.0, 1.0], (128, 128))
        v[5, 7] = 448.0  # block max exactly 448 * 2^k: exponent k, no round-up
        x[bi * 128:(bi + 1) * 128] = v * 2.0 ** k
    xb = _bits(x)
    q, e8, _, _ = oracle.quant_blocks_pow2(xb)
    assert list(e8[:, 0]) == [127 - 20, 127 + 13]
    assert np.array_equal(oracle.dequant_blocks_pow2(q, e8), x)


# ---------------------------------------------------------------- re-quantized column copy, BF16 dequantizer

def _decode_f32(codes):
    """E4M3 code -> value from the format table (brute helper), as float32."""
    pos = e4m3_positive_values()
    c = np.asarray(codes, np.uint8)
    v = pos[np.minimum(c & 0x7F, 0x7E)]
    return np.where(c & 0x80, -v, v).astype(np.float32)


def test_requant_colgroups_brute_force():
    x = synth.activation(300, 256, seed=41, stream="test")
    q, s = oracle.quant_rowgroups(x)
    off = [0, 77, 77, 300]
    qc, sc = oracle.requant_colgroups(q, s, offsets=off)
    assert qc.shape == (256, 128 + 256)
    for (lo, hi, p0) in ((0, 77, 0), (77, 205, 128), (205, 300, 256)):
        for c in (0, 1, 127, 128, 255):
            v = _decode_f32(q[lo:hi, c]) * s[c // 128, lo:hi]  # numpy float32 product: IEEE binary32
            a = np.float32(np.max(np.abs(v)))
            S = np.float32(a / np.float32(448.0))
            assert sc[p0 // 128, c] == S
            assert np.array_equal(qc[c, p0:p0 + (hi - lo)], brute_encode(v / S)), (lo, c)
            assert not qc[c, p0 + (hi - lo):p0 + 128].any()


def test_requant_of_exactly_representable_copy_is_the_direct_column_copy():
    # every 1x128 group holds E4M3 grid values times 2^k with its maximum at 448 * 2^k,
    # so the row copy dequantizes back to x exactly and the re-quantized column copy
    # must equal the column copy taken from x directly
    rng = np.random.default_rng(42)
    pos = e4m3_positive_values()
    R, C = 256, 256
    x = np.empty((R, C))
    for r in range(R):
        for g in range(2):
            v = rng.choice(pos, 128) * rng.choice([-1.0, 1.0], 128)
            v[rng.integers(128)] = 448.0
            x[r, g * 128:(g + 1) * 128] = v * 2.0 ** int(rng.integers(-12, 12))
    xb = _bits(x)
    q, s = oracle.quant_rowgroups(xb)
    assert np.array_equal(oracle.dequant_rowgroups(q, s), x)
    qc, sc = oracle.requant_colgroups(q, s)
    qd, sd = oracle.quant_colgroups(xb)
    assert np.array_equal(qc, qd) and np.array_equal(sc, sd)


def _bf16_rne_exact(v):
    """BF16 RNE by exact rational arithmetic (independent of the C oracle)."""
    from fractions import Fraction
    f = Fraction(v)
    if f == 0:
        return 0x8000 if np.signbit(v) else 0
    a = abs(f)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 7)
    m = a / quantum
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = float(n * quantum)
    bits = int(np.array([val], np.float32).view(np.uint32)[0]) >> 16
    return bits | (0x8000 if f < 0 else 0)


def test_dequant_bf16_single_rounding():
    x = synth.activation(64, 256, seed=43, stream="test")
    q, s = oracle.quant_rowgroups(x)
    # scales with full 24-bit significands make the products need the single rounding
    s = (s * np.float32(1.2345678)).astype(np.float32)
    out = oracle.dequant_rowgroups_bf16(q, s)
    rng = np.random.default_rng(44)
    for r, c in zip(rng.integers(0, 64, 400), rng.integers(0, 256, 400)):
        exact = float(_decode_f32(q[r, c])) * float(s[c // 128, r])
        assert out[r, c] == _bf16_rne_exact(exact), (r, c)
    # a product exactly on a bf16 midpoint rounds to even; just above it rounds up
    qq = np.array([[0x38] * 128], np.uint8)  # decode = 1.0
    tie = np.float32(1.0 + 2.0 ** -8)  # halfway between bf16 1.0 and 1.0078125
    above = np.nextafter(tie, np.float32(2))
    o = oracle.dequant_rowgroups_bf16(qq, np.array([[tie]], np.float32))
    assert o[0, 0] == 0x3F80
    o = oracle.dequant_rowgroups_bf16(qq, np.array([[above]], np.float32))
    assert o[0, 0] == 0x3F81
    wq, ws, _, _ = oracle.quant_blocks(synth.weight(256, 256, seed=45, stream="test"))
    ob = oracle.dequant_blocks_bf16(wq, ws)
    for r, c in zip(rng.integers(0, 256, 200), rng.integers(0, 256, 200)):
        exact = float(_decode_f32(wq[r, c])) * float(ws[r // 128, c // 128])
        assert ob[r, c] == _bf16_rne_exact(exact)

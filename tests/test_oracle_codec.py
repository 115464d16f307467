"""Pins for the oracle's E4M3 codec (no GPU).

The codec is pinned against (a) code points printed in the OCP FP8 spec
(tests/golden/e4m3_points.txt), (b) an exhaustive nearest-value search that
shares no algorithm with the oracle, on random values and on every rounding
midpoint and its neighbours, and (c) closed-form properties of the format.
"""
import math
import os

import numpy as np
import pytest

import oracle
from _brute import GOLDEN, brute_encode, e4m3_positive_values


def _golden_points():
    pts = []
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            pts.append((int(code, 16), float(val)))
    return pts


def test_decode_matches_spec_points():
    for code, val in _golden_points():
        got = oracle.e4m3_decode(code)
        if math.isnan(val):
            assert math.isnan(got), hex(code)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_decode_table_shape():
    vals = oracle.e4m3_decode(np.arange(256))
    finite = vals[~np.isnan(vals)]
    assert np.isnan(vals).sum() == 2  # 0x7F and 0xFF only: no infinities
    assert len(finite) == 254
    assert len(np.unique(finite)) == 253  # +0 and -0 compare equal
    assert finite.max() == 448.0 and finite.min() == -448.0
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0)  # codes increase with value
    assert np.array_equal(pos, e4m3_positive_values())
    assert np.array_equal(vals[0x80:0xFF], -pos)


def test_encode_roundtrips_every_finite_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_encode_midpoints_and_neighbours_against_brute_force():
    pos = e4m3_positive_values()
    mids = 0.5 * (pos[1:] + pos[:-1])
    pts = []
    for m in mids:
        f = np.float32(m)
        assert float(f) == m  # midpoints are binary32 numbers
        pts += [float(np.nextafter(f, np.float32(-1))), float(f), float(np.nextafter(f, np.float32(1e9)))]
    pts += [448.0, 448.5, 463.99, 464.0, 464.01, 1e30, 2.0 ** -10, 2.0 ** -11, 0.0]
    pts = np.array(pts)
    pts = np.concatenate([pts, -pts])
    got = oracle.e4m3_encode(pts)
    assert np.array_equal(got, brute_encode(pts))


def test_encode_ties_go_to_even_mantissa():
    # 1.0625 lies halfway between 1.0 (0x38, even) and 1.125 (0x39, odd)
    assert oracle.e4m3_encode(1.0625) == 0x38
    # 1.1875 lies halfway between 1.125 (0x39) and 1.25 (0x3A, even)
    assert oracle.e4m3_encode(1.1875) == 0x3A
    # halfway between the two smallest subnormals: 1.5 * 2^-9 -> 2 * 2^-9 (even)
    assert oracle.e4m3_encode(1.5 * 2.0 ** -9) == 0x02
    # 2^-10 is halfway between 0 and the smallest subnormal: -> 0
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(-(2.0 ** -10)) == 0x80


def test_encode_saturates_and_keeps_zero_sign():
    assert oracle.e4m3_encode(500.0) == 0x7E
    assert oracle.e4m3_encode(-1e38) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(float("nan")) == 0x7F


@pytest.mark.parametrize("seed", [0, 1])
def test_encode_random_values_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    v = np.concatenate([
        rng.standard_normal(4000) * 100,
        rng.uniform(-1, 1, 2000) * 2.0 ** -8,
        rng.uniform(-500, 500, 2000),
    ]).astype(np.float32).astype(np.float64)
    assert np.array_equal(oracle.e4m3_encode(v), brute_encode(v))


def test_encoder_on_every_binary32_pattern_against_a_bit_level_encoder():
    """All 2^32 binary32 patterns: the oracle's encoder (binary search against exact
    midpoints) equals an independent encoder that rounds the pattern's mantissa
    (tests/e4m3_sweep_check.c), so no input of any quantizer can hit a code the
    E4M3 definition does not give."""
    import subprocess
    import tempfile

    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "e4m3_sweep_check.c")
    orc = os.path.join(os.path.dirname(here), "oracle", "jetq_oracle.c")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "sweep")
        subprocess.run(["gcc", "-O2", "-std=gnu99", "-ffp-contract=off", "-pthread", src, orc, "-o", exe, "-lm"],
                       check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches=0" in r.stdout

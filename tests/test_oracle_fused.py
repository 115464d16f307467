"""Pins for the fused-producer definitions in the oracle (RMSNorm and the SwiGLU
product feeding the 1x128 quantizer): the binary32 operation sequence is checked
against binary64 mathematics and closed forms, not against itself."""
import math

import numpy as np

import oracle
import synth


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_ulp(v):
    """Spacing of BF16 values around v (binary64 array)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def test_expf_fixed_within_one_ulp_of_exp():
    for x in np.linspace(-87.0, 88.0, 20001, dtype=np.float32):
        got = oracle.expf_fixed(float(x))
        ref = math.exp(float(x))
        assert abs(got - ref) <= float(np.spacing(np.float32(ref))), x
    assert oracle.expf_fixed(0.0) == 1.0
    assert oracle.expf_fixed(89.0) == math.inf and oracle.expf_fixed(-88.0) == 0.0


def test_swiglu_against_binary64_and_closed_forms():
    g = synth.activation(64, 256, seed=71, stream="test")
    u = synth.activation(64, 256, seed=72, stream="test")
    h = oracle.swiglu_bf16(g, u)
    gv, uv = _f32(g), _f32(u)
    exact = gv / (1.0 + np.exp(-gv)) * uv
    assert np.all(np.abs(_f32(h) - exact) <= _bf16_ulp(exact) + 1e-30)
    # closed forms: silu(0) = 0; sigmoid(30) rounds to 1 in binary32; exp(90) overflows
    gg = synth.bf16_bits(np.array([0.0, 30.0, -90.0, 2.5], np.float32))
    uu = synth.bf16_bits(np.array([7.0, -3.0, 5.0, 0.0], np.float32))
    hh = _f32(oracle.swiglu_bf16(gg, uu))
    assert hh[0] == 0.0 and hh[1] == -90.0 and hh[2] == 0.0 and hh[3] == 0.0


def test_rmsnorm_against_binary64_and_constant_rows():
    x = synth.activation(16, 4096, seed=73, stream="test")
    w = synth.bf16_bits((1.0 + 0.1 * synth.normal(4096, seed=74, stream=synth.STREAM["test"])).astype(np.float32))
    y, rstd = oracle.rmsnorm_bf16(x, w, eps=1e-6)
    xv, wv = _f32(x), _f32(w)
    rs = 1.0 / np.sqrt(np.mean(xv * xv, axis=1) + 1e-6)
    assert np.all(np.abs(rstd - rs) <= 4e-7 * rs)
    exact = xv * rs[:, None] * wv[None, :]
    assert np.all(np.abs(_f32(y) - exact) <= 1.01 * _bf16_ulp(exact))
    # a constant row of 2.0 with unit weights: sum of squares exactly 4 * 4096
    xc = synth.bf16_bits(np.full((1, 4096), 2.0, np.float32))
    wc = synth.bf16_bits(np.ones(4096, np.float32))
    yc, rc = oracle.rmsnorm_bf16(xc, wc, eps=0.0)
    assert rc[0] == np.float32(0.5) and np.all(_f32(yc) == 1.0)

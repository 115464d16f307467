"""GPU quantizers vs the oracle: bit-exact codes and scales.

Input classes follow the byte-exact quantizer tests the Miles Blackwell post
describes (random, quantization-boundary, all-zero, maximum-value), plus
ragged token counts, MoE-style segments and the full dense-8B shapes.
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _brute import e4m3_positive_values
from _gpu import f32bits, mx_atom_offsets, mx_atoms, to_dev_bf16, u8

pytestmark = pytest.mark.gpu


def _classes(kind, rows, cols, seed, gs=128):
    rng = np.random.default_rng(seed)
    if kind == "random":
        return synth.activation(rows, cols, seed=seed, stream="test")
    if kind == "zeros":
        x = np.zeros((rows, cols), np.uint16)
        x[::3] = 0x8000
        return x
    if kind == "maxes":
        x = np.where(rng.random((rows, cols)) < 0.5, 0x7F7F, 0xFF7F).astype(np.uint16)
        x[1::4] = synth.bf16_bits(np.full(cols, 448.0 * 2.0 ** 9, np.float32))
        return x
    if kind == "tiny":  # scales below 2^-96 and subnormal BF16 values
        return synth.bf16_bits((rng.standard_normal((rows, cols)) * 1e-36).astype(np.float32))
    # boundary: every group max = 448 * 2^k, other entries on E4M3 midpoints * 2^k, +-1 BF16 ulp
    pos = e4m3_positive_values()
    mids = 0.5 * (pos[1:] + pos[:-1])
    k = rng.integers(-30, 30, size=(rows, 1))
    v = rng.choice(mids, (rows, cols)) * rng.choice([-1.0, 1.0], (rows, cols)) * 2.0 ** k
    b = synth.bf16_bits(v.astype(np.float32)).astype(np.int32) + rng.integers(-1, 2, (rows, cols))
    b = b.astype(np.uint16)
    b[:, ::gs] = synth.bf16_bits((448.0 * 2.0 ** k[:, 0]).astype(np.float32))[:, None]
    return b


def _check_act(x, offsets=None):
    n, c = x.shape
    seg = None if offsets is None else torch.tensor(offsets, dtype=torch.int64, device="cuda:0")
    out = jq.quant_act(to_dev_bf16(x), seg_offsets=seg)
    torch.cuda.synchronize()
    q, s = oracle.quant_rowgroups(x)
    assert np.array_equal(u8(out["q_row"]), q)
    assert np.array_equal(f32bits(out["s_row"]), f32bits(s))
    qc, sc = oracle.quant_colgroups(x, offsets=offsets)
    P = qc.shape[1]
    assert np.array_equal(u8(out["q_col"])[:, :P], qc)
    assert np.array_equal(f32bits(out["s_col"])[: P // 128], f32bits(sc))


@pytest.mark.parametrize("kind", ["random", "boundary", "zeros", "maxes", "tiny"])
def test_act_quant_classes(kind):
    _check_act(_classes(kind, 384, 512, 11))


@pytest.mark.parametrize("n", [1, 7, 128, 129, 300])
def test_act_quant_ragged_tokens(n):
    _check_act(synth.activation(n, 256, seed=n, stream="test"))


def test_act_quant_segments():
    x = synth.activation(700, 256, seed=5, stream="x")
    _check_act(x, offsets=[0, 0, 5, 133, 133, 400, 700])


def test_act_quant_many_segments():
    off, _ = synth.zipf_topk_routing(256, 32, 4, 1.2, seed=0)  # 1024 routed rows
    x = synth.activation(int(off[-1]), 256, seed=6, stream="x")
    _check_act(x, offsets=list(off))


@pytest.mark.parametrize("kind", ["random", "boundary", "zeros", "maxes", "tiny"])
def test_weight_quant_classes(kind):
    w = _classes(kind, 384, 256, 12) if kind != "random" else synth.weight(384, 256, seed=1)
    q, s, qT, sT = jq.quant_weight(to_dev_bf16(w))
    torch.cuda.synchronize()
    oq, os_, oqT, osT = oracle.quant_blocks(w)
    assert np.array_equal(u8(q), oq) and np.array_equal(u8(qT), oqT)
    assert np.array_equal(f32bits(s), f32bits(os_)) and np.array_equal(f32bits(sT), f32bits(osT))


def _check_mx(x, offsets=None):
    r, c = x.shape
    seg = None if offsets is None else torch.tensor(offsets, dtype=torch.int64, device="cuda:0")
    out = jq.quant_mx(to_dev_bf16(x), seg_offsets=seg)
    torch.cuda.synchronize()
    q, e8 = oracle.quant_mx_rows(x)
    assert np.array_equal(u8(out["q_row"]), q)
    assert np.array_equal(u8(out["e8_row"]), mx_atoms(e8, c))
    qc, e8c = oracle.quant_mx_cols(x, offsets=offsets)
    P = qc.shape[1]
    cap = out["ldq_col"]
    assert np.array_equal(u8(out["q_col"])[:, :P], qc)
    # only the first P/32 blocks of every row are defined
    got = u8(out["e8_col"])
    assert got.size == jq.jetq_mx_scale_bytes(c, cap)
    assert np.array_equal(got[mx_atom_offsets(c, P // 32)], e8c)


@pytest.mark.parametrize("kind", ["random", "boundary", "zeros", "maxes", "tiny"])
def test_mx_quant_classes(kind):
    _check_mx(_classes(kind, 256, 512, 13, gs=32))


def test_mx_quant_ragged_and_segments():
    _check_mx(synth.activation(77, 128, seed=3, stream="x"))
    _check_mx(synth.activation(300, 256, seed=4, stream="x"), offsets=[0, 40, 40, 200, 300])


def test_full_size_dense_8b_quantizers():
    """Dense-8B MLP shapes: X 8192 x 4096 (row + column copies) and W_up 12288 x 4096."""
    x = synth.activation(8192, 4096, seed=0, stream="x")
    _check_act(x)
    w = synth.weight(12288, 4096, seed=0, stream="w_up")
    q, s, qT, sT = jq.quant_weight(to_dev_bf16(w))
    torch.cuda.synchronize()
    oq, os_, oqT, osT = oracle.quant_blocks(w)
    assert np.array_equal(u8(q), oq) and np.array_equal(u8(qT), oqT)
    assert np.array_equal(f32bits(s), f32bits(os_))

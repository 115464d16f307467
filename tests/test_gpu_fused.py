"""The 1x128 quantizer fused with its producer (RMSNorm, the SwiGLU product)
against the oracle: the oracle computes the BF16 producer output operation by
operation, then quantizes it as it quantizes any BF16 tensor; the GPU never
stores that BF16 tensor.  Codes, scales and RMSNorm's rstd must agree bit for
bit, on ragged token counts, more than 32 column groups (two passes of the
statistics warp), MoE-style segments, strided inputs, tiles that take the
general (zero / tiny scale) path and the dense-8B MLP shapes.
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import f32bits, to_dev_bf16, u8

pytestmark = pytest.mark.gpu


def _norm_weight(c, seed):
    return synth.bf16_bits((1.0 + 0.1 * synth.normal(c, seed=seed, stream=synth.STREAM["test"])).astype(np.float32))


def _compare(out, y, offsets=None, row=True, col=True):
    if row:
        q, s = oracle.quant_rowgroups(y)
        assert np.array_equal(u8(out["q_row"]), q)
        assert np.array_equal(f32bits(out["s_row"]), f32bits(s))
    if col:
        qc, sc = oracle.quant_colgroups(y, offsets=offsets)
        P = qc.shape[1]
        assert np.array_equal(u8(out["q_col"])[:, :P], qc)
        assert np.array_equal(f32bits(out["s_col"])[: P // 128], f32bits(sc))


def _seg(offsets):
    return None if offsets is None else torch.tensor(offsets, dtype=torch.int64, device="cuda:0")


def _check_rms(x, w, eps=1e-6, offsets=None, row=True, col=True, pad=0):
    n, c = x.shape
    xd = to_dev_bf16(np.pad(x, ((0, 0), (0, pad)))) if pad else to_dev_bf16(x)
    out = jq.quant_act_rmsnorm(xd[:, :c], to_dev_bf16(w), eps=eps, row=row, col=col, seg_offsets=_seg(offsets))
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    y, rstd = oracle.rmsnorm_bf16(x, w, eps=eps)
    assert np.array_equal(f32bits(out["rstd"]), f32bits(rstd))
    _compare(out, y, offsets, row, col)


def _check_swiglu(g, u, offsets=None, row=True, col=True, pad=0):
    n, c = g.shape
    gd = to_dev_bf16(np.pad(g, ((0, 0), (0, pad)))) if pad else to_dev_bf16(g)
    ud = to_dev_bf16(u)
    out = jq.quant_act_swiglu(gd[:, :c], ud, row=row, col=col, seg_offsets=_seg(offsets))
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    _compare(out, oracle.swiglu_bf16(g, u), offsets, row, col)


@pytest.mark.parametrize("n", [1, 7, 128, 129, 300])
def test_rmsnorm_ragged_tokens(n):
    _check_rms(synth.activation(n, 512, seed=n, stream="x"), _norm_weight(512, n))


def test_rmsnorm_more_than_32_groups_and_strided_rows():
    c = 40 * 128  # 40 column groups: two passes of the statistics warp, the second ragged
    _check_rms(synth.activation(200, c, seed=3, stream="x"), _norm_weight(c, 3), pad=256)


@pytest.mark.parametrize("row,col", [(True, False), (False, True)])
def test_rmsnorm_single_copy(row, col):
    _check_rms(synth.activation(260, 384, seed=4, stream="x"), _norm_weight(384, 4), row=row, col=col)


def test_rmsnorm_segments_and_eps():
    x = synth.activation(700, 256, seed=5, stream="x")
    _check_rms(x, _norm_weight(256, 5), eps=1e-5, offsets=[0, 0, 5, 133, 133, 400, 700])


def test_rmsnorm_zero_rows_take_the_general_path():
    x = synth.activation(256, 256, seed=6, stream="x")
    x[17] = 0  # a zero row: rstd = 1/sqrt(eps), zero groups, zero scales
    x[200:] = 0x8000  # negative zeros
    w = _norm_weight(256, 6)
    w[130:140] = 0  # zero weight columns: zero column groups in the column copy
    _check_rms(x, w)


def test_rmsnorm_rstd_only():
    x = synth.activation(33, 256, seed=7, stream="x")
    w = _norm_weight(256, 7)
    rstd = torch.empty(33, dtype=torch.float32, device="cuda:0")
    jq.jetq_quant_act_1x128_rmsnorm(to_dev_bf16(x), to_dev_bf16(w), 1e-6, rstd, None, None, None, None, 0)
    torch.cuda.synchronize()
    assert np.array_equal(f32bits(rstd), f32bits(oracle.rmsnorm_bf16(x, w)[1]))


@pytest.mark.parametrize("n", [1, 13, 128, 300])
def test_swiglu_ragged_tokens(n):
    g = synth.activation(n, 512, seed=n, stream="x")
    u = synth.activation(n, 512, seed=n + 1000, stream="x")
    _check_swiglu(g, u)


def test_swiglu_saturation_and_tiny_values():
    rng = np.random.default_rng(8)
    g = synth.activation(256, 384, seed=8, stream="x")
    u = synth.activation(256, 384, seed=9, stream="x")
    # gates past both exp clamps (-g > 88: sigmoid 0; -g < -87: sigmoid 1) and at zero
    g[:, 0] = synth.bf16_bits(np.float32(-95.0))
    g[:, 1] = synth.bf16_bits(np.float32(95.0))
    g[:, 2] = 0
    g[3::7] = synth.bf16_bits(rng.uniform(-100, 100, (len(g[3::7]), 384)).astype(np.float32))
    # a tile of tiny products (scales below 2^-96: the general path)
    g[128:, 128:256] = synth.bf16_bits((rng.standard_normal((128, 128)) * 1e-20).astype(np.float32))
    u[128:, 128:256] = synth.bf16_bits((rng.standard_normal((128, 128)) * 1e-20).astype(np.float32))
    _check_swiglu(g, u, pad=128)


def test_swiglu_every_gate_value():
    """Every finite BF16 gate, one binade and sign per row (so each 1x128 group
    resolves its values), against the oracle: covers every sigmoid table slot
    and the directly computed gates (zeros, subnormals, tiny and large
    magnitudes) on both sides of the table's edges."""
    e8 = np.arange(255, dtype=np.uint32)
    rows = []
    for s in (0, 1):
        rows.append((s << 15) | (e8[:, None] << 7) | np.arange(128, dtype=np.uint32)[None, :])
    g = np.concatenate(rows).astype(np.uint16)  # 510 rows x 128
    # |up| <= 1 keeps every product finite (|h| <= |g|): the quantizer's domain
    u = synth.bf16_bits(np.random.default_rng(14).uniform(-1.0, 1.0, g.shape).astype(np.float32))
    _check_swiglu(g, u)
    # up = 1: h = BF16(silu(g)) itself is quantized
    _check_swiglu(g, synth.bf16_bits(np.ones(g.shape, np.float32)))


def test_swiglu_segments():
    off, _ = synth.zipf_topk_routing(64, 16, 4, 1.2, seed=1)  # 256 routed rows
    n = int(off[-1])
    _check_swiglu(synth.activation(n, 256, seed=10, stream="x"), synth.activation(n, 256, seed=11, stream="x"),
                  offsets=list(off))


def test_full_size_dense_8b_producers():
    """Dense-8B MLP: RMSNorm over X 8192 x 4096 before gate/up, SwiGLU over 8192 x 12288 before down."""
    x = synth.activation(8192, 4096, seed=0, stream="x")
    _check_rms(x, _norm_weight(4096, 0))
    g = synth.activation(8192, 12288, seed=1, stream="x")
    u = synth.activation(8192, 12288, seed=2, stream="x")
    _check_swiglu(g, u)


def test_fused_equals_producer_then_quantizer():
    """The fused call equals the unfused pipeline on the GPU: the producer's BF16
    output (the oracle's, uploaded) quantized by the plain 1x128 quantizer."""
    g = synth.activation(300, 640, seed=12, stream="x")
    u = synth.activation(300, 640, seed=13, stream="x")
    fused = jq.quant_act_swiglu(to_dev_bf16(g), to_dev_bf16(u))
    plain = jq.quant_act(to_dev_bf16(oracle.swiglu_bf16(g, u)))
    torch.cuda.synchronize()
    for k in ("q_row", "s_row", "q_col", "s_col"):
        assert torch.equal(fused[k].view(torch.uint8), plain[k].view(torch.uint8))

"""128-block recipe with power-of-two scales on the GPU (the blockwise recipe's
scales constrained to powers of two, run on the native block-scaled MMA).

Quantizers: codes and scale atoms bit-exact against the oracle (the atoms
repeat each 128-group's E8M0 byte over its four 32-element sub-blocks).
GEMMs: |y - y_ref| <= 1e-5 * sum_k |a_k b_k| against the FP64 oracle on the
dequantized operands, including grouped (MoE) launches.
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, mx_atoms, to_dev_bf16, u8

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
P2 = jq.RECIPE_BLOCK128_POW2


def _atoms_rows(e8_groups, k):
    """Per-128-group bytes [R x K/128] -> MX atoms for (R, K): each byte over its 4 sub-blocks."""
    return mx_atoms(np.repeat(e8_groups, 4, axis=1), k)


def _atoms_blocks(e8_blocks, rows, k):
    """Per-block bytes [rows/128 x k/128] -> MX atoms for (rows, k)."""
    return mx_atoms(np.repeat(np.repeat(e8_blocks, 128, axis=0), 4, axis=1), k)


@pytest.mark.parametrize("kind", ["random", "outliers", "zeros", "ragged"])
def test_pow2_activation_quantizer_bit_exact(kind):
    R, C = (300, 384) if kind == "ragged" else (256, 512)
    if kind == "zeros":
        x = np.zeros((R, C), np.uint16)
    elif kind == "outliers":
        x = synth.activation(R, C, seed=31, stream="x")
        x[::7, ::13] = synth.bf16_bits(np.full(((R + 6) // 7, (C + 12) // 13), 3.0e4, np.float32))
    else:
        x = synth.activation(R, C, seed=32, stream="x")
    g = jq.quant_act_pow2(to_dev_bf16(x))
    torch.cuda.synchronize()
    q, e8 = oracle.quant_mx_rows(x, bs=128)
    assert np.array_equal(u8(g["q_row"]), q)
    assert np.array_equal(u8(g["e8_row"]), _atoms_rows(e8, C))
    qc, e8c = oracle.quant_mx_cols(x, bs=128, seg_align=128)
    P = qc.shape[1]
    assert np.array_equal(u8(g["q_col"])[:, :P], qc)
    assert np.array_equal(u8(g["e8_col"]), _atoms_rows(e8c, g["ldq_col"]))


def test_pow2_activation_quantizer_segments():
    off = np.array([0, 40, 40, 200, 333], dtype=np.int64)
    R, C = int(off[-1]), 256
    x = synth.activation(R, C, seed=33, stream="x")
    seg = torch.tensor(off, dtype=torch.int64, device=DEV)
    g = jq.quant_act_pow2(to_dev_bf16(x), row=False, seg_offsets=seg)
    torch.cuda.synchronize()
    qc, e8c = oracle.quant_mx_cols(x, bs=128, offsets=off, seg_align=128)
    P = qc.shape[1]
    assert np.array_equal(u8(g["q_col"])[:, :P], qc)
    assert np.array_equal(u8(g["e8_col"]), _atoms_rows(e8c, g["ldq_col"]))


def test_pow2_weight_quantizer_bit_exact():
    D, C = 384, 512
    w = synth.weight(D, C, seed=34, stream="w")
    w[128:256, 256:384] = 0  # an all-zero block: byte 127, codes 0
    q, e8, qT, e8T = jq.quant_weight_pow2(to_dev_bf16(w))
    torch.cuda.synchronize()
    oq, oe8, oqT, oe8T = oracle.quant_blocks_pow2(w)
    assert np.array_equal(u8(q), oq) and np.array_equal(u8(qT), oqT)
    assert np.array_equal(u8(e8), _atoms_blocks(oe8, D, C))
    assert np.array_equal(u8(e8T), _atoms_blocks(oe8T, C, D))


@pytest.mark.parametrize("N,D,C", [(256, 512, 512), (300, 384, 640), (1, 256, 128), (129, 768, 384)])
def test_pow2_three_gemms_against_oracle(N, D, C):
    x = synth.activation(N, C, seed=N + 35, stream="x")
    w = synth.weight(D, C, seed=N + 35, stream="w")
    dy = synth.gradient(N, D, seed=N + 35, stream="dy")
    gx, gdy = jq.quant_act_pow2(to_dev_bf16(x)), jq.quant_act_pow2(to_dev_bf16(dy))
    qw, ew, qwt, ewt = jq.quant_weight_pow2(to_dev_bf16(w))
    y = jq.fprop(gx["q_row"], gx["e8_row"], qw, ew, recipe=P2)
    dx = jq.dgrad(gdy["q_row"], gdy["e8_row"], qwt, ewt, recipe=P2)
    dw = jq.wgrad(gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], gx["ldq_col"], recipe=P2)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    X = oracle.dequant_mx_rows(*oracle.quant_mx_rows(x, bs=128), bs=128)
    DY = oracle.dequant_mx_rows(*oracle.quant_mx_rows(dy, bs=128), bs=128)
    W = oracle.dequant_blocks_pow2(*oracle.quant_blocks_pow2(w)[:2])
    Xc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(x, bs=128), N, bs=128)
    DYc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(dy, bs=128), N, bs=128)
    assert_gemm_close(y, *oracle.fprop(X, W))
    assert_gemm_close(dx, *oracle.dgrad(DY, W))
    assert_gemm_close(dw, *oracle.wgrad(DYc, Xc))


def test_pow2_grouped_against_oracle():
    off = np.array([0, 0, 5, 133, 133, 260, 700, 701, 701], dtype=np.int64)
    E, R, C, D = len(off) - 1, int(off[-1]), 256, 384
    x = synth.activation(R, C, seed=36, stream="x")
    dy = synth.gradient(R, D, seed=36, stream="dy")
    ws = [synth.weight(D, C, seed=40 + e, stream="w") for e in range(E)]
    seg = torch.tensor(off, dtype=torch.int64, device=DEV)
    gx = jq.quant_act_pow2(to_dev_bf16(x), seg_offsets=seg)
    gdy = jq.quant_act_pow2(to_dev_bf16(dy), seg_offsets=seg)
    qs = [jq.quant_weight_pow2(to_dev_bf16(w)) for w in ws]
    qw, ew = torch.stack([q[0] for q in qs]), torch.cat([q[1] for q in qs])
    qwt, ewt = torch.stack([q[2] for q in qs]), torch.cat([q[3] for q in qs])
    y = jq.grouped(jq.GEMM_FPROP, gx["q_row"], gx["e8_row"], qw, ew, seg, n=D, k=C, recipe=P2)
    dx = jq.grouped(jq.GEMM_DGRAD, gdy["q_row"], gdy["e8_row"], qwt, ewt, seg, n=C, k=D, recipe=P2)
    Pk = oracle.colcopy_length(off, R)
    dw = jq.grouped(jq.GEMM_WGRAD, gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], seg, n=C, k=Pk,
                    recipe=P2)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    X = oracle.dequant_mx_rows(*oracle.quant_mx_rows(x, bs=128), bs=128)
    DY = oracle.dequant_mx_rows(*oracle.quant_mx_rows(dy, bs=128), bs=128)
    Xc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(x, bs=128, offsets=off), R, bs=128, offsets=off)
    DYc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(dy, bs=128, offsets=off), R, bs=128, offsets=off)
    yc, dxc, dwc = y.cpu(), dx.cpu(), dw.cpu()
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        W = oracle.dequant_blocks_pow2(*oracle.quant_blocks_pow2(ws[e])[:2])
        if hi > lo:
            assert_gemm_close(yc[lo:hi], *oracle.fprop(X[lo:hi], W))
            assert_gemm_close(dxc[lo:hi], *oracle.dgrad(DY[lo:hi], W))
            assert_gemm_close(dwc[e], *oracle.wgrad(DYc[lo:hi], Xc[lo:hi]))
        else:
            assert torch.count_nonzero(dwc[e]) == 0

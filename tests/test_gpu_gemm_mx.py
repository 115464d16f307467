"""MXFP8 GEMMs (native block-scaled tensor-core MMA) vs the FP64 oracle.

Operands are the MXFP8 copies the Miles Blackwell post describes: row-wise
1x32 blocks for the FProp/DGrad first operand and FProp weight, column-wise
(32x1) copies for the DGrad weight and both WGrad operands, each quantized
from BF16.  Tolerance: |y - y_ref| <= 1e-5 * sum_k |a_k b_k| elementwise.
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, to_dev_bf16, u8

pytestmark = pytest.mark.gpu


def _operands(N, D, C, seed):
    x = synth.activation(N, C, seed=seed, stream="x")
    w = synth.weight(D, C, seed=seed, stream="w")
    dy = synth.gradient(N, D, seed=seed, stream="dy")
    gx = jq.quant_mx(to_dev_bf16(x))
    gw = jq.quant_mx(to_dev_bf16(w))
    gdy = jq.quant_mx(to_dev_bf16(dy))
    return (x, w, dy), (gx, gw, gdy)


@pytest.mark.parametrize("N,D,C", [(256, 512, 512), (300, 384, 256), (1, 256, 128), (129, 768, 384)])
def test_mx_three_gemms_against_oracle(N, D, C):
    (x, w, dy), (gx, gw, gdy) = _operands(N, D, C, seed=N + 7)
    # the GPU codes are the oracle's (the quantizer tests pin this; re-check the ones used here)
    qx, ex = oracle.quant_mx_rows(x)
    assert np.array_equal(u8(gx["q_row"]), qx)
    X = oracle.dequant_mx_rows(qx, ex)
    W = oracle.dequant_mx_rows(*oracle.quant_mx_rows(w))
    DY = oracle.dequant_mx_rows(*oracle.quant_mx_rows(dy))
    Wc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(w), D)
    Xc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(x), N)
    DYc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(dy), N)

    y = jq.fprop(gx["q_row"], gx["e8_row"], gw["q_row"], gw["e8_row"], recipe=jq.RECIPE_MXFP8)
    dx = jq.dgrad(gdy["q_row"], gdy["e8_row"], gw["q_col"], gw["e8_col"], recipe=jq.RECIPE_MXFP8)
    dw = jq.wgrad(gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], gx["ldq_col"], recipe=jq.RECIPE_MXFP8)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    assert_gemm_close(y, *oracle.fprop(X, W))
    assert_gemm_close(dx, *oracle.dgrad(DY, Wc))
    assert_gemm_close(dw, *oracle.wgrad(DYc, Xc))


def test_mx_bf16_output_and_accumulate():
    (x, w, dy), (gx, gw, gdy) = _operands(200, 256, 256, seed=3)
    y32 = jq.fprop(gx["q_row"], gx["e8_row"], gw["q_row"], gw["e8_row"], recipe=jq.RECIPE_MXFP8)
    y16 = jq.fprop(gx["q_row"], gx["e8_row"], gw["q_row"], gw["e8_row"], out_dtype=torch.bfloat16,
                   recipe=jq.RECIPE_MXFP8)
    dw1 = jq.wgrad(gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], gx["ldq_col"], recipe=jq.RECIPE_MXFP8)
    dw2 = jq.wgrad(gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], gx["ldq_col"], dw=dw1.clone(),
                   accumulate=True, recipe=jq.RECIPE_MXFP8)
    torch.cuda.synchronize()
    assert torch.equal(y32.to(torch.bfloat16), y16)
    assert torch.equal(dw2, dw1 + dw1)


def test_mx_full_size_sampled_dense_8b():
    """Dense-8B shapes (N = 8192, C = 4096, D = 12288), 2048 sampled outputs per GEMM."""
    N, C, D = 8192, 4096, 12288
    x = synth.activation(N, C, seed=0, stream="x")
    w = synth.weight(D, C, seed=0, stream="w_up")
    dy = synth.gradient(N, D, seed=0, stream="dy_up")
    gx, gw, gdy = jq.quant_mx(to_dev_bf16(x)), jq.quant_mx(to_dev_bf16(w)), jq.quant_mx(to_dev_bf16(dy))
    y = jq.fprop(gx["q_row"], gx["e8_row"], gw["q_row"], gw["e8_row"], recipe=jq.RECIPE_MXFP8)
    dx = jq.dgrad(gdy["q_row"], gdy["e8_row"], gw["q_col"], gw["e8_col"], recipe=jq.RECIPE_MXFP8)
    dw = jq.wgrad(gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], gx["ldq_col"], recipe=jq.RECIPE_MXFP8)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    rng = np.random.default_rng(1)

    def pick(R, Cc):
        at = np.stack([rng.integers(0, R, 2048), rng.integers(0, Cc, 2048)], 1)
        at[:2] = [[0, 0], [R - 1, Cc - 1]]
        return at

    def take(t, at):
        return t[torch.as_tensor(at[:, 0], device=t.device), torch.as_tensor(at[:, 1], device=t.device)]

    X = oracle.dequant_mx_rows(*oracle.quant_mx_rows(x))
    W = oracle.dequant_mx_rows(*oracle.quant_mx_rows(w))
    at = pick(N, D)
    assert_gemm_close(take(y, at), *oracle.fprop(X, W, at=at))
    DY = oracle.dequant_mx_rows(*oracle.quant_mx_rows(dy))
    Wc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(w), D)
    at = pick(N, C)
    assert_gemm_close(take(dx, at), *oracle.dgrad(DY, Wc, at=at))
    Xc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(x), N)
    DYc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(dy), N)
    at = pick(D, C)
    assert_gemm_close(take(dw, at), *oracle.wgrad(DYc, Xc, at=at))

"""Rollout-shaped (few-token) GEMMs on weights of at least 32 row blocks: the
decode kernel that streams 128 weight rows per tile with the tokens as the
MMA's narrow operand.

Checked against the FP64 oracle (|y - y_ref| <= 1e-5 * sum|a b|) and, bit for
bit, against the training-shaped kernel on the same quantized operands, for
batch sizes on both sides of each token-column width (16, 32, 64) and K-block
counts that leave a partial multi-K-block copy at the end of each tile.
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, to_dev_bf16

pytestmark = pytest.mark.gpu

NS = (1, 13, 16, 17, 32, 40, 64)


@pytest.fixture(scope="module")
def fprop_case():
    D, C = 4096, 640  # 32 weight row blocks; 5 K-blocks
    x = synth.activation(64, C, seed=5, stream="x")
    w = synth.weight(D, C, seed=5, stream="w")
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(w), transposed=False)
    W = oracle.dequant_blocks(*oracle.quant_blocks(w)[:2])
    return x, qw, sw, W


@pytest.mark.parametrize("n", NS)
def test_decode_fprop_against_oracle_and_training(fprop_case, n):
    x, qw, sw, W = fprop_case
    a = jq.quant_act(to_dev_bf16(x[:n]), col=False)
    y_dec = jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_DECODE)
    y_train = jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_TRAIN)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    X = oracle.dequant_rowgroups(*oracle.quant_rowgroups(x[:n]))
    assert_gemm_close(y_dec, *oracle.fprop(X, W))
    assert torch.equal(y_dec.view(torch.int32), y_train.view(torch.int32))


@pytest.mark.parametrize("n", (1, 24, 64))
def test_decode_dgrad_against_oracle_and_training(n):
    D, C = 384, 4096  # DGrad output width C = 32 row blocks of W^T; 3 K-blocks
    dy = synth.gradient(n, D, seed=6, stream="dy")
    w = synth.weight(D, C, seed=6, stream="w")
    _, _, qwt, swt = jq.quant_weight(to_dev_bf16(w))
    a = jq.quant_act(to_dev_bf16(dy), col=False)
    dx = jq.dgrad(a["q_row"], a["s_row"], qwt, swt)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    DY = oracle.dequant_rowgroups(*oracle.quant_rowgroups(dy))
    W = oracle.dequant_blocks(*oracle.quant_blocks(w)[:2])
    assert_gemm_close(dx, *oracle.dgrad(DY, W))
    # the same product through the FProp entry point's training shape
    dx_train = jq.fprop(a["q_row"], a["s_row"], qwt, swt, path=jq.PATH_TRAIN)
    assert torch.equal(dx.view(torch.int32), dx_train.view(torch.int32))


def test_decode_bf16_output_is_rne_of_f32(fprop_case):
    x, qw, sw, _ = fprop_case
    a = jq.quant_act(to_dev_bf16(x[:9]), col=False)
    y32 = jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_DECODE)
    y16 = jq.fprop(a["q_row"], a["s_row"], qw, sw, out_dtype=torch.bfloat16, path=jq.PATH_DECODE)
    torch.cuda.synchronize()
    assert torch.equal(y16, y32.to(torch.bfloat16))


def test_decode_repeated_launches_identical(fprop_case):
    x, qw, sw, _ = fprop_case
    a = jq.quant_act(to_dev_bf16(x[:40]), col=False)
    ys = [jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_DECODE) for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32))
    assert np.isfinite(ys[0].cpu().numpy()).all()

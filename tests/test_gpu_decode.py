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


# With a workspace, batches of up to 32 tokens against weights of 32-76 row
# blocks take the split-K kernel: a cluster of 4 CTAs per row block (at most 38
# blocks, at least 16 K-blocks) or of 2 (at least 8 K-blocks); the partial
# sums pass through the workspace and the cluster's CTAs fold them in
# ascending K.  K-block counts leave a partial last chunk and cluster members
# with fewer chunks than others; the token counts cover both token-column
# widths (16, 32) and the fold's 1, 2, 4 and 8 elements a thread; 33 and 64
# tokens and a 96-block weight check that the others keep the one-CTA kernel.
SPLIT_CASES = [
    (4096, 2048, 1), (4096, 2176, 16), (4096, 2432, 8), (4096, 2176, 17), (4864, 2688, 32),
    (4096, 3200, 33), (4864, 2176, 64), (4096, 12288, 5),
    (8192, 1024, 1), (8192, 2048, 8), (9728, 1152, 13), (6144, 1408, 24), (12288, 4096, 8),
]


@pytest.mark.parametrize("D,C,n", SPLIT_CASES)
def test_decode_split_k_against_oracle_and_training(D, C, n):
    x = synth.activation(n, C, seed=D + C + n, stream="x")
    w = synth.weight(D, C, seed=D + C, stream="w")
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(w), transposed=False)
    a = jq.quant_act(to_dev_bf16(x), col=False)
    # batches of up to 32 tokens against at most 76 row blocks split K; the
    # others keep one CTA per row band
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    split = n <= 32 and D // 128 <= sms // 2
    assert jq.jetq_decode_workspace_bytes(n, D, C) == (D * (C // 128) * n * 4 if split else 0)
    y_dec = jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_DECODE)  # with a workspace
    y_dec16 = jq.fprop(a["q_row"], a["s_row"], qw, sw, out_dtype=torch.bfloat16, path=jq.PATH_DECODE)
    y_one = torch.empty_like(y_dec)  # no workspace: one CTA per row band
    jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, a["q_row"], a["s_row"], qw, sw, n, D, C, y_one, jq.PATH_DECODE)
    y_train = jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_TRAIN)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    assert torch.equal(y_dec.view(torch.int32), y_train.view(torch.int32))
    assert torch.equal(y_one.view(torch.int32), y_train.view(torch.int32))
    assert torch.equal(y_dec16, y_dec.to(torch.bfloat16))
    X = oracle.dequant_rowgroups(*oracle.quant_rowgroups(x))
    W = oracle.dequant_blocks(*oracle.quant_blocks(w)[:2])
    assert_gemm_close(y_dec, *oracle.fprop(X, W))


def test_decode_split_k_repeated_launches_identical():
    D, C, n = 4096, 2304, 40
    x = synth.activation(n, C, seed=11, stream="x")
    w = synth.weight(D, C, seed=11, stream="w")
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(w), transposed=False)
    a = jq.quant_act(to_dev_bf16(x), col=False)
    ys = [jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_DECODE) for _ in range(4)]
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32))

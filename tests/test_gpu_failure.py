"""Failure detection on the GPU without a fault: the bounded-wait diagnostic
makes a wait run out (an mbarrier nothing completes) and the host reads the
status; the context stays usable for the next kernels."""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_bounded_wait_times_out_and_reports():
    assert jq.jetq_check_device_error() == jq.OK  # nothing pending
    limit = 50_000_000  # 50 ms
    elapsed = torch.full((2,), -1, dtype=torch.int64, device=DEV)
    assert jq.jetq_selftest_bounded_wait(limit, elapsed) == jq.OK
    torch.cuda.synchronize()
    e0, e1 = (int(v) for v in elapsed.cpu())
    # waiter 0 gave up on its own limit; waiter 1 on the abort flag, well
    # before its own limit of 8 x 50 ms
    assert limit <= e0 < 20 * limit
    assert 0 <= e1 < 8 * limit
    assert e1 >= e0 - 5_000_000
    assert jq.jetq_check_device_error() == jq.ERR_TIMEOUT
    assert jq.jetq_check_device_error() == jq.OK  # read and cleared


def test_context_usable_after_timeout():
    elapsed = torch.zeros((2,), dtype=torch.int64, device=DEV)
    assert jq.jetq_selftest_bounded_wait(1_000_000, elapsed) == jq.OK
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.ERR_TIMEOUT
    x = synth.activation(64, 256, seed=11, stream="x")
    w = synth.weight(256, 256, seed=11, stream="w")
    ax = jq.quant_act(to_dev_bf16(x), col=False)
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(w), transposed=False)
    y = jq.fprop(ax["q_row"], ax["s_row"], qw, sw)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    X = oracle.dequant_rowgroups(*oracle.quant_rowgroups(x))
    W = oracle.dequant_blocks(*oracle.quant_blocks(w)[:2])
    assert_gemm_close(y, *oracle.fprop(X, W))
    assert np.isfinite(y.cpu().numpy()).all()

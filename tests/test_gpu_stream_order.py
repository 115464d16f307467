"""Stream order across back-to-back launches that share buffers.

The GEMM, decode and quantizer kernels are launched so that a kernel's
prologue may overlap the previous kernel on the stream (programmatic
dependent launch); each waits for its predecessor before it touches global
memory.  These tests queue, with no host synchronization in between, chains
in which a kernel overwrites what the previous kernel reads (the quantized
copies, the split-K decode workspace) or reads what it writes, and check
every result against the same call made in isolation, bit for bit.
"""
import pytest
import torch

import rollout_x128_act_gb300 as jq
import synth
from _gpu import to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


def test_quantize_then_gemm_chain_on_shared_copies():
    n, c, d = 512, 1024, 2048
    xs = [to_dev_bf16(synth.activation(n, c, seed=70 + i, stream="x")) for i in range(4)]
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(synth.weight(d, c, seed=70, stream="w")), transposed=False)
    # isolated references
    refs = []
    for x in xs:
        a = jq.quant_act(x, col=False)
        refs.append(jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_TRAIN))
        torch.cuda.synchronize()
    # chain: every quantization overwrites the copies the previous GEMM reads
    q = torch.empty((n, c), dtype=torch.uint8, device=DEV)
    s = torch.empty((c // 128, n), dtype=torch.float32, device=DEV)
    ys = [torch.empty((n, d), dtype=torch.float32, device=DEV) for _ in xs]
    for x, y in zip(xs, ys):
        jq.jetq_quant_act_1x128(x, q, s, None, None, 0)
        jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, q, s, qw, sw, n, d, c, y, jq.PATH_TRAIN)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    for y, r in zip(ys, refs):
        assert torch.equal(_bits(y), _bits(r))


@pytest.mark.parametrize("n", [1, 8])
def test_decode_chain_on_one_workspace_and_output(n):
    # the down projection's split-K decode (partials through the workspace):
    # consecutive calls reuse one workspace and one output buffer, which a copy
    # kernel reads after each call
    d, c = 4096, 12288
    wsb = jq.jetq_decode_workspace_bytes(n, d, c)
    assert wsb > 0
    work = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    weights = [jq.quant_weight(to_dev_bf16(synth.weight(d, c, seed=80 + i, stream="w_down")), transposed=False)
               for i in range(3)]
    a = jq.quant_act(to_dev_bf16(synth.activation(n, c, seed=81, stream="h")), col=False)
    refs = []
    for qw, sw, _, _ in weights:
        y = torch.empty((n, d), dtype=torch.float32, device=DEV)
        jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, a["q_row"], a["s_row"], qw, sw, n, d, c, y, jq.PATH_DECODE)
        torch.cuda.synchronize()
        refs.append(y)
    shared = torch.empty((n, d), dtype=torch.float32, device=DEV)
    copies = []
    for qw, sw, _, _ in weights * 2:  # six calls, one workspace, one output buffer copied after each
        jq.jetq_gemm_fprop_ws(jq.RECIPE_BLOCK128, a["q_row"], a["s_row"], qw, sw, n, d, c, shared, work,
                              jq.PATH_DECODE)
        copies.append(shared.clone())
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    for i, y in enumerate(copies):
        assert torch.equal(_bits(y), _bits(refs[i % 3])), i

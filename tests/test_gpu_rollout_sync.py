"""On-policy FP8 weight sync on one GPU (SkyRL "On-Policy FP8 weight sync": the
trainer's FP8 payload and scales reach the rollout engine as-is): the payload is
copied device to device into the rollout engine's own buffers, must arrive
byte-identical, and a rollout decode step of 128 concurrent sequences, replayed
from a CUDA graph, must produce the training kernels' rows bit for bit."""
import numpy as np
import torch

import rollout_x128_act_gb300 as jq
import synth
from _gpu import to_dev_bf16

import pytest

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_payload_sync_and_graph_replayed_rollout_step_match_training():
    C, D, n = 1024, 4096, 128  # hidden, intermediate (>= 32 row blocks: the decode kernels), concurrent sequences
    W = {"gate": synth.weight(D, C, seed=61, stream="w_gate"), "up": synth.weight(D, C, seed=61, stream="w_up"),
         "down": synth.weight(C, D, seed=61, stream="w_down")}
    trainer = {k: jq.quant_weight(to_dev_bf16(w), transposed=False)[:2] for k, w in W.items()}
    # weight sync: device-to-device copies into buffers the rollout side owns
    rollout = {k: (torch.empty_like(q), torch.empty_like(s)) for k, (q, s) in trainer.items()}
    for k in trainer:
        rollout[k][0].copy_(trainer[k][0])
        rollout[k][1].copy_(trainer[k][1])
    torch.cuda.synchronize()
    for k in trainer:
        assert torch.equal(rollout[k][0], trainer[k][0])
        assert torch.equal(rollout[k][1].view(torch.int32), trainer[k][1].view(torch.int32))

    x = to_dev_bf16(synth.activation(n, C, seed=62, stream="x"))
    h = to_dev_bf16(synth.activation(n, D, seed=62, stream="h"))
    ax = jq.quant_act(x, col=False)
    ah = jq.quant_act(h, col=False)
    ys = {k: torch.empty((n, D if k != "down" else C), dtype=torch.bfloat16, device=DEV) for k in W}

    def step():
        jq.jetq_quant_act_1x128(x, ax["q_row"], ax["s_row"], None, None, 0)
        for k in ("gate", "up"):
            q, s = rollout[k]
            jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, ax["q_row"], ax["s_row"], q, s, n, D, C, ys[k], jq.PATH_DECODE)
        jq.jetq_quant_act_1x128(h, ah["q_row"], ah["s_row"], None, None, 0)
        q, s = rollout["down"]
        jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, ah["q_row"], ah["s_row"], q, s, n, C, D, ys["down"], jq.PATH_DECODE)

    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            step()
    for k in ys:
        ys[k].zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    # training kernels on the trainer's payload
    for k, a in (("gate", ax), ("up", ax), ("down", ah)):
        q, s = trainer[k]
        ref = jq.fprop(a["q_row"], a["s_row"], q, s, out_dtype=torch.bfloat16, path=jq.PATH_TRAIN)
        torch.cuda.synchronize()
        assert torch.equal(ys[k].view(torch.int16), ref.view(torch.int16)), k

"""Grouped (MoE expert) GEMMs vs per-expert FP64 oracle GEMMs, both recipes.

Routing is Zipf-skewed top-k (the MoE workload's shape) plus hand-made
offsets with empty experts and ragged segments.  Each expert's block must meet
the same bound as a dense GEMM: |y - y_ref| <= 1e-5 * sum|a b|.
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

ROUTINGS = {
    "zipf": lambda: synth.zipf_topk_routing(160, 8, 4, 1.2, seed=0)[0],  # 640 routed rows
    "ragged": lambda: np.array([0, 0, 5, 133, 133, 260, 700, 701, 701], dtype=np.int64),
}


def _seg(off):
    return torch.tensor(off, dtype=torch.int64, device=DEV)


def _experts_b128(ws):
    qs, ss, qts, sts = zip(*(jq.quant_weight(to_dev_bf16(w)) for w in ws))
    return torch.stack(qs), torch.stack(ss), torch.stack(qts), torch.stack(sts)


@pytest.mark.parametrize("routing", sorted(ROUTINGS))
def test_grouped_block128(routing):
    off = ROUTINGS[routing]()
    E, R = len(off) - 1, int(off[-1])
    C, D = 256, 384
    x = synth.activation(R, C, seed=1, stream="x")
    dy = synth.gradient(R, D, seed=1, stream="dy")
    ws = [synth.weight(D, C, seed=e, stream="w") for e in range(E)]
    seg = _seg(off)
    ax = jq.quant_act(to_dev_bf16(x), seg_offsets=seg)
    ady = jq.quant_act(to_dev_bf16(dy), seg_offsets=seg)
    qw, sw, qwt, swt = _experts_b128(ws)

    y = jq.grouped(jq.GEMM_FPROP, ax["q_row"], ax["s_row"], qw, sw, seg, n=D, k=C)
    dx = jq.grouped(jq.GEMM_DGRAD, ady["q_row"], ady["s_row"], qwt, swt, seg, n=C, k=D)
    P = oracle.colcopy_length(off, R)
    dw = jq.grouped(jq.GEMM_WGRAD, ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], seg, n=C, k=P)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK

    X = oracle.dequant_rowgroups(*oracle.quant_rowgroups(x))
    DY = oracle.dequant_rowgroups(*oracle.quant_rowgroups(dy))
    Xc = oracle.dequant_colgroups(*oracle.quant_colgroups(x, offsets=off), R, offsets=off)
    DYc = oracle.dequant_colgroups(*oracle.quant_colgroups(dy, offsets=off), R, offsets=off)
    yc, dxc, dwc = y.cpu(), dx.cpu(), dw.cpu()
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        W = oracle.dequant_blocks(*oracle.quant_blocks(ws[e])[:2])
        if hi > lo:
            assert_gemm_close(yc[lo:hi], *oracle.fprop(X[lo:hi], W))
            assert_gemm_close(dxc[lo:hi], *oracle.dgrad(DY[lo:hi], W))
            assert_gemm_close(dwc[e], *oracle.wgrad(DYc[lo:hi], Xc[lo:hi]))
        else:
            assert torch.count_nonzero(dwc[e]) == 0


def test_grouped_equals_dense_per_expert_bitwise():
    """An expert's rows of a grouped FProp equal a dense FProp of that expert's rows."""
    off = ROUTINGS["zipf"]()
    E, R, C, D = len(off) - 1, int(off[-1]), 512, 256
    x = synth.activation(R, C, seed=2, stream="x")
    ws = [synth.weight(D, C, seed=10 + e, stream="w") for e in range(E)]
    seg = _seg(off)
    ax = jq.quant_act(to_dev_bf16(x), col=False)
    qw, sw, _, _ = _experts_b128(ws)
    y = jq.grouped(jq.GEMM_FPROP, ax["q_row"], ax["s_row"], qw, sw, seg, n=D, k=C)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        a = jq.quant_act(to_dev_bf16(x[lo:hi]), col=False)
        ye = jq.fprop(a["q_row"], a["s_row"], qw[e], sw[e], path=jq.PATH_TRAIN)
        assert torch.equal(ye.view(torch.int32), y[lo:hi].view(torch.int32)), e


@pytest.mark.parametrize("routing", sorted(ROUTINGS))
def test_grouped_mxfp8(routing):
    off = ROUTINGS[routing]()
    E, R = len(off) - 1, int(off[-1])
    C, D = 256, 384
    x = synth.activation(R, C, seed=3, stream="x")
    dy = synth.gradient(R, D, seed=3, stream="dy")
    ws = [synth.weight(D, C, seed=20 + e, stream="w") for e in range(E)]
    seg = _seg(off)
    gx = jq.quant_mx(to_dev_bf16(x), seg_offsets=seg)
    gdy = jq.quant_mx(to_dev_bf16(dy), seg_offsets=seg)
    gws = [jq.quant_mx(to_dev_bf16(w)) for w in ws]
    qw = torch.stack([g["q_row"] for g in gws])
    ew = torch.cat([g["e8_row"] for g in gws])   # each expert's atoms for (D, C)
    qwc = torch.stack([g["q_col"] for g in gws])  # [E, C, D]: W columns quantized along D
    ewc = torch.cat([g["e8_col"] for g in gws])  # atoms for (C, D)

    y = jq.grouped(jq.GEMM_FPROP, gx["q_row"], gx["e8_row"], qw, ew, seg, n=D, k=C, recipe=jq.RECIPE_MXFP8)
    dx = jq.grouped(jq.GEMM_DGRAD, gdy["q_row"], gdy["e8_row"], qwc, ewc, seg, n=C, k=D, recipe=jq.RECIPE_MXFP8)
    P = oracle.colcopy_length(off, R)
    dw = jq.grouped(jq.GEMM_WGRAD, gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], seg, n=C, k=P,
                    recipe=jq.RECIPE_MXFP8)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK

    X = oracle.dequant_mx_rows(*oracle.quant_mx_rows(x))
    DY = oracle.dequant_mx_rows(*oracle.quant_mx_rows(dy))
    Xc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(x, offsets=off), R, offsets=off)
    DYc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(dy, offsets=off), R, offsets=off)
    yc, dxc, dwc = y.cpu(), dx.cpu(), dw.cpu()
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        W = oracle.dequant_mx_rows(*oracle.quant_mx_rows(ws[e]))
        Wc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(ws[e]), D)
        if hi > lo:
            assert_gemm_close(yc[lo:hi], *oracle.fprop(X[lo:hi], W))
            assert_gemm_close(dxc[lo:hi], *oracle.dgrad(DY[lo:hi], Wc))
            assert_gemm_close(dwc[e], *oracle.wgrad(DYc[lo:hi], Xc[lo:hi]))
        else:
            assert torch.count_nonzero(dwc[e]) == 0


def test_grouped_moe_30b_shapes_sampled():
    """30B-A3B-shaped MoE FProp (gate/up fused, 128 experts, hidden 2048, 1536 out),
    16384 tokens routed top-8 with Zipf(1.2) load; sampled rows of a few experts."""
    off, _ = synth.zipf_topk_routing(16384, 128, 8, 1.2, seed=0)
    E, R, C, D = 128, int(off[-1]), 2048, 1536
    x = synth.activation(R, C, seed=0, stream="x")
    seg = _seg(off)
    ax = jq.quant_act(to_dev_bf16(x), col=False)
    wstack = synth.weight(E * D, C, seed=0, stream="w_gate")
    qw, sw = [], []
    for e in range(E):
        q, s, _, _ = jq.quant_weight(to_dev_bf16(wstack[e * D:(e + 1) * D]), transposed=False)
        qw.append(q)
        sw.append(s)
    qw, sw = torch.stack(qw), torch.stack(sw)
    y = jq.grouped(jq.GEMM_FPROP, ax["q_row"], ax["s_row"], qw, sw, seg, n=D, k=C, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    X = None
    rng = np.random.default_rng(0)
    for e in (0, 1, 63, 127):
        lo, hi = int(off[e]), int(off[e + 1])
        rows = np.unique(np.concatenate([[lo, hi - 1], rng.integers(lo, hi, 6)]))
        xq, xs = oracle.quant_rowgroups(x[rows])
        X = oracle.dequant_rowgroups(xq, xs)
        W = oracle.dequant_blocks(*oracle.quant_blocks(wstack[e * D:(e + 1) * D])[:2])
        ref, bound = oracle.fprop(X, W)
        got = y[torch.as_tensor(rows, device=DEV)].float()
        # BF16 output: the FP32 result rounded once more (half a BF16 ulp)
        assert_gemm_close(got, ref, bound + 2.0 ** -8 * np.abs(ref) / 1e-5)

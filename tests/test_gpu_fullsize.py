"""Full-size parity on the shapes the bench times, on sampled outputs.

* MoE expert GEMMs, 30B-A3B-shaped: 128 experts, hidden 2048, fused gate/up
  projection of 1536 rows, 16384 tokens routed top-8 with Zipf(1.2) expert load
  (131072 routed rows; experts of about 135 to 15,500 rows).  Grouped FProp,
  DGrad and WGrad in the three recipes (FP32 128-block scales, MXFP8, and
  128-block with power-of-two scales).  The Miles post on Blackwell-native RL
  recipes quantizes the MoE expert GEMMs like every other linear layer, so
  each expert's block meets the dense bound |y - y_ref| <= 1e-5 * sum|a b|.
  Sampled experts: the largest, the smallest and two in between; FProp/DGrad
  compare whole sampled rows, WGrad sampled weight-gradient entries over the
  expert's full token range.  BF16 outputs are checked as the round-to-nearest-
  even of the FP32 run, bit for bit, over the whole output.
* The dense-8B layer (8192 tokens, 4096 -> 12288) in the power-of-two recipe:
  4096 sampled outputs of each of the three GEMMs.
* The on-policy identity at full size for both dense-8B weight shapes: the
  rollout (DECODE) FProp of tokens 0:N equals rows 0:N of the 8192-token
  training FProp bit for bit, for the up projection (W 12288 x 4096) and the
  down projection (W 4096 x 12288, K = 12288).
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, to_dev_bf16, u8

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

TOKENS, TOPK, EXPERTS, HID, INTER2 = 16384, 8, 128, 2048, 1536


@pytest.fixture(scope="module")
def moe_inputs():
    off, _ = synth.zipf_topk_routing(TOKENS, EXPERTS, TOPK, 1.2, seed=0)
    R = int(off[-1])
    x = synth.activation(R, HID, seed=0, stream="x")
    dy = synth.gradient(R, INTER2, seed=0, stream="dy_gate")
    wstack = synth.weight(EXPERTS * INTER2, HID, seed=0, stream="w_gate")
    counts = np.diff(off)
    order = np.argsort(counts, kind="stable")
    experts = sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2]), int(order[(3 * len(order)) // 4])})
    return dict(off=off, R=R, x=x, dy=dy, w=wstack, experts=experts, counts=counts)


def _expert_w(inp, e):
    return inp["w"][e * INTER2:(e + 1) * INTER2]


def _quantize_gpu(recipe, inp):
    """GPU copies of X, dY and the stacked expert weights for one recipe."""
    seg = torch.tensor(inp["off"], dtype=torch.int64, device=DEV)
    tx, tdy = to_dev_bf16(inp["x"]), to_dev_bf16(inp["dy"])
    if recipe == jq.RECIPE_BLOCK128:
        ax, ady = jq.quant_act(tx, seg_offsets=seg), jq.quant_act(tdy, seg_offsets=seg)
        sa_x, sa_dy, sc_x, sc_dy = ax["s_row"], ady["s_row"], ax["s_col"], ady["s_col"]
        qs = [jq.quant_weight(to_dev_bf16(_expert_w(inp, e))) for e in range(EXPERTS)]
        qw, sw = torch.stack([q[0] for q in qs]), torch.stack([q[1] for q in qs])
        qwt, swt = torch.stack([q[2] for q in qs]), torch.stack([q[3] for q in qs])
    elif recipe == jq.RECIPE_MXFP8:
        ax, ady = jq.quant_mx(tx, seg_offsets=seg), jq.quant_mx(tdy, seg_offsets=seg)
        sa_x, sa_dy, sc_x, sc_dy = ax["e8_row"], ady["e8_row"], ax["e8_col"], ady["e8_col"]
        gws = [jq.quant_mx(to_dev_bf16(_expert_w(inp, e))) for e in range(EXPERTS)]
        qw, sw = torch.stack([g["q_row"] for g in gws]), torch.cat([g["e8_row"] for g in gws])
        qwt, swt = torch.stack([g["q_col"] for g in gws]), torch.cat([g["e8_col"] for g in gws])
    else:
        ax, ady = jq.quant_act_pow2(tx, seg_offsets=seg), jq.quant_act_pow2(tdy, seg_offsets=seg)
        sa_x, sa_dy, sc_x, sc_dy = ax["e8_row"], ady["e8_row"], ax["e8_col"], ady["e8_col"]
        qs = [jq.quant_weight_pow2(to_dev_bf16(_expert_w(inp, e))) for e in range(EXPERTS)]
        qw, sw = torch.stack([q[0] for q in qs]), torch.cat([q[1] for q in qs])
        qwt, swt = torch.stack([q[2] for q in qs]), torch.cat([q[3] for q in qs])
    del tx, tdy
    return dict(seg=seg, ax=ax, ady=ady, sa_x=sa_x, sa_dy=sa_dy, sc_x=sc_x, sc_dy=sc_dy,
                qw=qw, sw=sw, qwt=qwt, swt=swt)


# oracle operands per recipe: (row copy of rows, weight, weight for DGrad, column copy of a segment)
def _o_rows(recipe, a):
    if recipe == jq.RECIPE_BLOCK128:
        return oracle.dequant_rowgroups(*oracle.quant_rowgroups(a))
    bs = 32 if recipe == jq.RECIPE_MXFP8 else 128
    return oracle.dequant_mx_rows(*oracle.quant_mx_rows(a, bs=bs), bs=bs)


def _o_row_codes(recipe, a):
    if recipe == jq.RECIPE_BLOCK128:
        return oracle.quant_rowgroups(a)[0]
    return oracle.quant_mx_rows(a, bs=32 if recipe == jq.RECIPE_MXFP8 else 128)[0]


def _o_weight(recipe, w):
    """(W for FProp, W for DGrad), both [D x C] dequantized."""
    if recipe == jq.RECIPE_BLOCK128:
        W = oracle.dequant_blocks(*oracle.quant_blocks(w)[:2])
        return W, W
    if recipe == jq.RECIPE_MXFP8:
        # FProp reads W quantized along C; DGrad reads W's column copy, quantized along D
        return (oracle.dequant_mx_rows(*oracle.quant_mx_rows(w)),
                oracle.dequant_mx_cols(*oracle.quant_mx_cols(w), w.shape[0]))
    W = oracle.dequant_blocks_pow2(*oracle.quant_blocks_pow2(w)[:2])
    return W, W


def _o_cols(recipe, a):
    n = a.shape[0]
    if recipe == jq.RECIPE_BLOCK128:
        return oracle.dequant_colgroups(*oracle.quant_colgroups(a), n)
    bs = 32 if recipe == jq.RECIPE_MXFP8 else 128
    return oracle.dequant_mx_cols(*oracle.quant_mx_cols(a, bs=bs), n, bs=bs)


def _sample_rows(lo, hi, rng, k=6):
    return np.unique(np.concatenate([[lo, hi - 1], rng.integers(lo, hi, k)])).astype(np.int64)


RECIPES = {"block128": jq.RECIPE_BLOCK128, "mxfp8": jq.RECIPE_MXFP8, "pow2": jq.RECIPE_BLOCK128_POW2}


@pytest.mark.parametrize("name", sorted(RECIPES))
def test_moe_30b_grouped_three_gemms_full_size(moe_inputs, name):
    recipe = RECIPES[name]
    inp = moe_inputs
    off, R = inp["off"], inp["R"]
    g = _quantize_gpu(recipe, inp)
    ax, ady, seg = g["ax"], g["ady"], g["seg"]

    y = jq.grouped(jq.GEMM_FPROP, ax["q_row"], g["sa_x"], g["qw"], g["sw"], seg, n=INTER2, k=HID, recipe=recipe)
    y16 = jq.grouped(jq.GEMM_FPROP, ax["q_row"], g["sa_x"], g["qw"], g["sw"], seg, n=INTER2, k=HID, recipe=recipe,
                     out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    assert torch.equal(y.to(torch.bfloat16), y16)
    del y16
    dx = jq.grouped(jq.GEMM_DGRAD, ady["q_row"], g["sa_dy"], g["qwt"], g["swt"], seg, n=HID, k=INTER2,
                    recipe=recipe)
    dx16 = jq.grouped(jq.GEMM_DGRAD, ady["q_row"], g["sa_dy"], g["qwt"], g["swt"], seg, n=HID, k=INTER2,
                      recipe=recipe, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    assert torch.equal(dx.to(torch.bfloat16), dx16)
    del dx16
    Pk = oracle.colcopy_length(off, R)
    assert Pk <= ax["ldq_col"]
    dw = jq.grouped(jq.GEMM_WGRAD, ady["q_col"], g["sc_dy"], ax["q_col"], g["sc_x"], seg, n=HID, k=Pk,
                    recipe=recipe)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK

    rng = np.random.default_rng(1)
    for e in inp["experts"]:
        lo, hi = int(off[e]), int(off[e + 1])
        assert hi > lo, e
        W, Wd = _o_weight(recipe, _expert_w(inp, e))
        rows = _sample_rows(lo, hi, rng)
        ti = torch.as_tensor(rows, device=DEV)
        # the sampled rows' codes are the oracle's, so the GEMM check is on the same operands
        assert np.array_equal(u8(ax["q_row"][ti]), _o_row_codes(recipe, inp["x"][rows])), e
        assert_gemm_close(y[ti], *oracle.fprop(_o_rows(recipe, inp["x"][rows]), W))
        assert_gemm_close(dx[ti], *oracle.dgrad(_o_rows(recipe, inp["dy"][rows]), Wd))
        # WGrad over the expert's whole token range (its segment of both column copies)
        DYc = _o_cols(recipe, inp["dy"][lo:hi])
        Xc = _o_cols(recipe, inp["x"][lo:hi])
        at = np.stack([rng.integers(0, INTER2, 512), rng.integers(0, HID, 512)], 1).astype(np.int64)
        at[:2] = [[0, 0], [INTER2 - 1, HID - 1]]
        ref, bound = oracle.wgrad(DYc, Xc, at=at)
        got = dw[e][torch.as_tensor(at[:, 0], device=DEV), torch.as_tensor(at[:, 1], device=DEV)]
        assert_gemm_close(got, ref, bound)
        del DYc, Xc


def test_dense_8b_pow2_full_size_sampled():
    """Power-of-two 128-block recipe on the dense-8B shape: 4096 sampled outputs per GEMM."""
    N, C, D = 8192, 4096, 12288
    P2 = jq.RECIPE_BLOCK128_POW2
    x = synth.activation(N, C, seed=0, stream="x")
    w = synth.weight(D, C, seed=0, stream="w_up")
    dy = synth.gradient(N, D, seed=0, stream="dy_up")
    gx, gdy = jq.quant_act_pow2(to_dev_bf16(x)), jq.quant_act_pow2(to_dev_bf16(dy))
    qw, ew, qwt, ewt = jq.quant_weight_pow2(to_dev_bf16(w))
    y = jq.fprop(gx["q_row"], gx["e8_row"], qw, ew, recipe=P2)
    dx = jq.dgrad(gdy["q_row"], gdy["e8_row"], qwt, ewt, recipe=P2)
    dw = jq.wgrad(gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], gx["ldq_col"], recipe=P2)
    y16 = jq.fprop(gx["q_row"], gx["e8_row"], qw, ew, recipe=P2, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    assert torch.equal(y.to(torch.bfloat16), y16)
    oq, oe = oracle.quant_mx_rows(x, bs=128)
    assert np.array_equal(u8(gx["q_row"]), oq)
    X = oracle.dequant_mx_rows(oq, oe, bs=128)
    W = oracle.dequant_blocks_pow2(*oracle.quant_blocks_pow2(w)[:2])
    DY = oracle.dequant_mx_rows(*oracle.quant_mx_rows(dy, bs=128), bs=128)
    rng = np.random.default_rng(2)

    def pick(R, Cc):
        at = np.stack([rng.integers(0, R, 4096), rng.integers(0, Cc, 4096)], 1).astype(np.int64)
        at[:4] = [[0, 0], [R - 1, Cc - 1], [0, Cc - 1], [R - 1, 0]]
        return at

    def take(t, at):
        return t[torch.as_tensor(at[:, 0], device=DEV), torch.as_tensor(at[:, 1], device=DEV)]

    at = pick(N, D)
    assert_gemm_close(take(y, at), *oracle.fprop(X, W, at=at))
    at = pick(N, C)
    assert_gemm_close(take(dx, at), *oracle.dgrad(DY, W, at=at))
    del X, DY
    Xc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(x, bs=128), N, bs=128)
    DYc = oracle.dequant_mx_cols(*oracle.quant_mx_cols(dy, bs=128), N, bs=128)
    at = pick(D, C)
    assert_gemm_close(take(dw, at), *oracle.wgrad(DYc, Xc, at=at))


@pytest.mark.parametrize("proj", ["up", "down"])
def test_rollout_equals_training_full_size_both_weight_shapes(proj):
    """Rows 0:N of the 8192-token training FProp against the dense-8B up projection
    (W 12288 x 4096) and down projection (W 4096 x 12288, K = 12288) equal the
    rollout-path FProp of tokens 0:N, bit for bit, with the weight payload
    quantized once and reused (on-policy weight sync)."""
    N = 8192
    if proj == "up":
        D, C, xs, ws = 12288, 4096, "x", "w_up"
    else:
        D, C, xs, ws = 4096, 12288, "h", "w_down"
    tx = to_dev_bf16(synth.activation(N, C, seed=0, stream=xs))
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(synth.weight(D, C, seed=0, stream=ws)), transposed=False)
    ax = jq.quant_act(tx, col=False)
    y_train = jq.fprop(ax["q_row"], ax["s_row"], qw, sw, path=jq.PATH_TRAIN)
    torch.cuda.synchronize()
    for n in (1, 8, 64, 256):
        a = jq.quant_act(tx[:n], col=False)  # the rollout batch quantized on its own
        assert torch.equal(a["q_row"], ax["q_row"][:n])
        y_dec = jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_DECODE)
        torch.cuda.synchronize()
        assert torch.equal(y_dec.view(torch.int32), y_train[:n].view(torch.int32)), n
    assert jq.jetq_check_device_error() == jq.OK

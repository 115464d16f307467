"""GPU block-scaled GEMMs vs the FP64 oracle, and the on-policy identity.

Tolerance (the bar the repository states for FP32 outputs):
    |y_gpu - y_ref| <= 1e-5 * sum_k |a_k * b_k|   elementwise,
where y_ref and the bound come from the oracle on the dequantized operands.
The rollout (DECODE) FProp must equal the training (TRAIN) FProp bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, to_dev_bf16, u8

pytestmark = pytest.mark.gpu


def _layer(N, D, C, seed):
    x = synth.activation(N, C, seed=seed, stream="x")
    w = synth.weight(D, C, seed=seed, stream="w")
    dy = synth.gradient(N, D, seed=seed, stream="dy")
    return x, w, dy


def _gpu_quant(x, w, dy):
    ax = jq.quant_act(to_dev_bf16(x))
    ady = jq.quant_act(to_dev_bf16(dy))
    qw, sw, qwt, swt = jq.quant_weight(to_dev_bf16(w))
    return ax, ady, (qw, sw, qwt, swt)


def _oracle_operands(x, w, dy):
    N = x.shape[0]
    X = oracle.dequant_rowgroups(*oracle.quant_rowgroups(x))
    W = oracle.dequant_blocks(*oracle.quant_blocks(w)[:2])
    DY = oracle.dequant_rowgroups(*oracle.quant_rowgroups(dy))
    qc, sc = oracle.quant_colgroups(x)
    Xc = oracle.dequant_colgroups(qc, sc, N)
    qc, sc = oracle.quant_colgroups(dy)
    DYc = oracle.dequant_colgroups(qc, sc, N)
    return X, W, DY, Xc, DYc


# (20, 384, 640) and (48, 256, 896): decode batches whose K-block counts (5, 3;
# 7, 2) leave a partly out-of-range multi-K-block copy at the end of each tile
@pytest.mark.parametrize("N,D,C", [(256, 512, 512), (300, 512, 384), (1, 256, 256), (129, 768, 128),
                                   (20, 384, 640), (48, 256, 896)])
def test_three_gemms_against_oracle(N, D, C):
    x, w, dy = _layer(N, D, C, seed=N + D)
    ax, ady, (qw, sw, qwt, swt) = _gpu_quant(x, w, dy)
    X, W, DY, Xc, DYc = _oracle_operands(x, w, dy)
    for path in (jq.PATH_TRAIN, jq.PATH_DECODE):
        y = jq.fprop(ax["q_row"], ax["s_row"], qw, sw, path=path)
        torch.cuda.synchronize()
        assert_gemm_close(y, *oracle.fprop(X, W))
    dx = jq.dgrad(ady["q_row"], ady["s_row"], qwt, swt)
    dw = jq.wgrad(ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], ax["ldq_col"])
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    assert_gemm_close(dx, *oracle.dgrad(DY, W))
    assert_gemm_close(dw, *oracle.wgrad(DYc, Xc))


@pytest.mark.parametrize("recipe", [jq.RECIPE_BLOCK128, jq.RECIPE_MXFP8])
def test_repeated_launches_are_bitwise_identical(recipe):
    """Every GEMM is deterministic: repeated launches on the same operands give the
    same bits (a pipeline race would show up here as a rare mismatch)."""
    N, D, C = 2048, 4096, 2048
    x, w, dy = _layer(N, D, C, seed=11)
    if recipe == jq.RECIPE_BLOCK128:
        ax, ady, (qw, sw, qwt, swt) = _gpu_quant(x, w, dy)
        f = lambda: jq.fprop(ax["q_row"], ax["s_row"], qw, sw, path=jq.PATH_TRAIN)  # noqa: E731
        g = lambda: jq.dgrad(ady["q_row"], ady["s_row"], qwt, swt)  # noqa: E731
        h = lambda: jq.wgrad(ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], ax["ldq_col"])  # noqa: E731
    else:
        gx, gw, gdy = jq.quant_mx(to_dev_bf16(x)), jq.quant_mx(to_dev_bf16(w)), jq.quant_mx(to_dev_bf16(dy))
        R = jq.RECIPE_MXFP8
        f = lambda: jq.fprop(gx["q_row"], gx["e8_row"], gw["q_row"], gw["e8_row"], recipe=R)  # noqa: E731
        g = lambda: jq.dgrad(gdy["q_row"], gdy["e8_row"], gw["q_col"], gw["e8_col"], recipe=R)  # noqa: E731
        h = lambda: jq.wgrad(gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], gx["ldq_col"],  # noqa: E731
                             recipe=R)
    for fn in (f, g, h):
        first = fn()
        for _ in range(4):
            again = fn()
            torch.cuda.synchronize()
            assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    assert jq.jetq_check_device_error() == jq.OK


@pytest.mark.parametrize("T,D,C", [(1024, 8192, 3072), (2048, 4096, 12288)])
def test_wgrad_repeatable_on_large_grids(T, D, C):
    """WGrad reuses a shared-memory ring of per-column scales that bulk copies refill;
    these grids (tens of tiles per SM) exposed a missing generic-to-async proxy fence
    as run-to-run differences.  Eight launches must agree bit for bit and meet the
    oracle bound on sampled outputs."""
    x = synth.activation(T, C, seed=13, stream="x")
    dy = synth.gradient(T, D, seed=13, stream="dy")
    ax = jq.quant_act(to_dev_bf16(x), row=False)
    ady = jq.quant_act(to_dev_bf16(dy), row=False)
    first = jq.wgrad(ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], ax["ldq_col"])
    for _ in range(7):
        again = jq.wgrad(ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], ax["ldq_col"])
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    assert jq.jetq_check_device_error() == jq.OK
    rng = np.random.default_rng(0)
    at = np.stack([rng.integers(0, D, 64), rng.integers(0, C, 64)], 1).astype(np.int64)
    DYc = oracle.dequant_colgroups(*oracle.quant_colgroups(dy), T)
    Xc = oracle.dequant_colgroups(*oracle.quant_colgroups(x), T)
    ref, bound = oracle.wgrad(DYc, Xc, at=at)
    got = first[torch.as_tensor(at[:, 0], device=first.device), torch.as_tensor(at[:, 1], device=first.device)]
    assert_gemm_close(got, ref, bound)


def test_bf16_output_is_rne_of_f32():
    x, w, _ = _layer(300, 512, 256, 3)
    ax = jq.quant_act(to_dev_bf16(x), col=False)
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(w), transposed=False)
    y32 = jq.fprop(ax["q_row"], ax["s_row"], qw, sw)
    y16 = jq.fprop(ax["q_row"], ax["s_row"], qw, sw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(y32.to(torch.bfloat16), y16)


def test_wgrad_accumulate_and_segments():
    N, D, C = 500, 256, 384
    x, w, dy = _layer(N, D, C, 4)
    off = [0, 100, 100, 356, 500]
    seg = torch.tensor(off, dtype=torch.int64, device="cuda:0")
    ax = jq.quant_act(to_dev_bf16(x), row=False, seg_offsets=seg)
    ady = jq.quant_act(to_dev_bf16(dy), row=False, seg_offsets=seg)
    P = oracle.colcopy_length(off, N)
    dw0 = torch.full((D, C), 0.5, dtype=torch.float32, device="cuda:0")
    dw = jq.wgrad(ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], P, dw=dw0.clone(), accumulate=True)
    torch.cuda.synchronize()
    # sum over segments of per-segment WGrad == WGrad over all rows (zero padding contributes nothing)
    qc, sc = oracle.quant_colgroups(x, offsets=off)
    Xc = oracle.dequant_colgroups(qc, sc, N, offsets=off)
    qc, sc = oracle.quant_colgroups(dy, offsets=off)
    DYc = oracle.dequant_colgroups(qc, sc, N, offsets=off)
    ref, bound = oracle.wgrad(DYc, Xc)
    # the final fl32(0.5 + acc) adds at most half an ulp of ~0.5
    assert_gemm_close(dw.double() - 0.5, ref, bound + 1e5 * 0.5 * 2.0 ** -24)


def test_rollout_fprop_equals_training_fprop_bitwise():
    """Same W payload (quantized once, as on-policy weight sync ships it) and the
    same activations: the decode-shaped kernel must return the training kernel's rows."""
    C, D = 4096, 12288
    x = synth.activation(1024, C, seed=0, stream="x")
    w = synth.weight(D, C, seed=0, stream="w_up")
    tx = to_dev_bf16(x)
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(w), transposed=False)
    ax = jq.quant_act(tx, col=False)
    y_train = jq.fprop(ax["q_row"], ax["s_row"], qw, sw, path=jq.PATH_TRAIN)
    for n in (1, 8, 20, 33, 64, 96, 128, 256):
        a = jq.quant_act(tx[:n], col=False)  # rollout quantizes its own batch
        assert torch.equal(a["q_row"], ax["q_row"][:n])
        y_dec = jq.fprop(a["q_row"], a["s_row"], qw, sw, path=jq.PATH_DECODE)
        torch.cuda.synchronize()
        assert torch.equal(y_dec.view(torch.int32), y_train[:n].view(torch.int32)), n


def test_full_size_sampled_dense_8b():
    """N = 8192, C = 4096, D = 12288: 4096 sampled outputs of each GEMM against the oracle."""
    N, C, D = 8192, 4096, 12288
    x = synth.activation(N, C, seed=0, stream="x")
    w = synth.weight(D, C, seed=0, stream="w_up")
    dy = synth.gradient(N, D, seed=0, stream="dy_up")
    ax, ady, (qw, sw, qwt, swt) = _gpu_quant(x, w, dy)
    y = jq.fprop(ax["q_row"], ax["s_row"], qw, sw)
    dx = jq.dgrad(ady["q_row"], ady["s_row"], qwt, swt)
    dw = jq.wgrad(ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], ax["ldq_col"])
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    # oracle codes must match (so the sampled GEMM check is on the same operands)
    oqx, osx = oracle.quant_rowgroups(x)
    assert np.array_equal(u8(ax["q_row"]), oqx)
    oqw, osw, _, _ = oracle.quant_blocks(w)
    assert np.array_equal(u8(qw), oqw)
    X = oracle.dequant_rowgroups(oqx, osx)
    W = oracle.dequant_blocks(oqw, osw)
    DY = oracle.dequant_rowgroups(*oracle.quant_rowgroups(dy))
    rng = np.random.default_rng(0)

    def pick(R, Cc):
        at = np.stack([rng.integers(0, R, 4096), rng.integers(0, Cc, 4096)], 1)
        at[:4] = [[0, 0], [R - 1, Cc - 1], [0, Cc - 1], [R - 1, 0]]
        return at

    def take(t, at):
        i = torch.as_tensor(at[:, 0], device=t.device)
        j = torch.as_tensor(at[:, 1], device=t.device)
        return t[i, j]

    at = pick(N, D)
    ref, b = oracle.fprop(X, W, at=at)
    assert_gemm_close(take(y, at), ref, b)
    at = pick(N, C)
    ref, b = oracle.dgrad(DY, W, at=at)
    assert_gemm_close(take(dx, at), ref, b)
    qc, sc = oracle.quant_colgroups(x)
    Xc = oracle.dequant_colgroups(qc, sc, N)
    qc, sc = oracle.quant_colgroups(dy)
    DYc = oracle.dequant_colgroups(qc, sc, N)
    at = pick(D, C)
    ref, b = oracle.wgrad(DYc, Xc, at=at)
    assert_gemm_close(take(dw, at), ref, b)

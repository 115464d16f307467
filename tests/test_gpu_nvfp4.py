"""NVFP4 quantizer and BF16 dequantizer on the GPU against the oracle: codes,
E4M3 block scales, FP32 scope scales and dequantized BF16 values bit for bit,
for per-token (row) and per-tensor (gate/up shared) scopes, on ragged widths,
the input classes of the byte-exact quantizer tests (random, boundary, zeros,
maxes) and the 30B-A3B MoE shapes."""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import f32bits, to_dev_bf16, u8

pytestmark = pytest.mark.gpu


def _check(x, scope=None):
    xd = to_dev_bf16(x)
    amax_d = None if scope is None else torch.tensor([scope], dtype=torch.float32, device="cuda:0")
    out = jq.quant_nvfp4(xd, scope_amax=amax_d)
    deq = jq.dequant_nvfp4_bf16(out["q"], out["sb"], out["sg"])
    torch.cuda.synchronize()
    q, sb, sg = oracle.quant_nvfp4(x, scope_amax=scope)
    assert np.array_equal(f32bits(out["sg"]), f32bits(sg))
    assert np.array_equal(u8(out["sb"]), sb)
    assert np.array_equal(u8(out["q"]), q)
    assert np.array_equal(deq.view(torch.int16).cpu().numpy().view(np.uint16), oracle.dequant_nvfp4_bf16(q, sb, sg))


@pytest.mark.parametrize("rows,cols", [(1, 16), (7, 48), (33, 256), (64, 272), (300, 2048), (16, 4096), (5, 784)])
def test_nvfp4_per_token(rows, cols):
    _check(synth.activation(rows, cols, seed=rows + cols, stream="x"))


def _classes(kind, rows, cols, seed):
    rng = np.random.default_rng(seed)
    if kind == "zeros":
        x = np.zeros((rows, cols), np.uint16)
        x[1::3] = 0x8000
        x[2, 5] = synth.bf16_bits(np.array([3.0], np.float32))[0]  # one nonzero row with a single value
        return x
    if kind == "maxes":
        return np.where(rng.random((rows, cols)) < 0.5, 0x7F7F, 0xFF7F).astype(np.uint16)
    if kind == "tiny":
        return synth.bf16_bits((rng.standard_normal((rows, cols)) * 1e-38).astype(np.float32))
    # boundary: each row's max is 2688 * 2^k (scope scale 2^k), every block's max 6 * 2^j * 2^k, the
    # other values on E2M1 midpoints of their block (0.25, 0.75, ... times the block scale), +-1 BF16 ulp
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    k = rng.integers(-20, 20, size=(rows, 1)).astype(np.float64)
    j = rng.integers(-6, 9, size=(rows, cols // 16)).astype(np.float64)
    blockscale = np.repeat(2.0 ** j, 16, axis=1) * 2.0 ** k
    v = rng.choice(mids, (rows, cols)) * rng.choice([-1.0, 1.0], (rows, cols)) * blockscale
    b = synth.bf16_bits(v.astype(np.float32)).astype(np.int32) + rng.integers(-1, 2, (rows, cols))
    b = b.astype(np.uint16)
    b[:, ::16] = synth.bf16_bits((6.0 * blockscale[:, ::16]).astype(np.float32))
    b[:, 0] = synth.bf16_bits((2688.0 * 2.0 ** k[:, 0]).astype(np.float32))
    return b


@pytest.mark.parametrize("kind", ["boundary", "zeros", "maxes", "tiny"])
def test_nvfp4_classes(kind):
    _check(_classes(kind, 96, 512, 31))


def test_nvfp4_tensor_scope_shared_by_gate_and_up():
    g = synth.weight(768, 2048, seed=3, stream="w_gate")
    u = synth.weight(768, 2048, seed=3, stream="w_up")
    gd, ud = to_dev_bf16(g), to_dev_bf16(u)
    amax = jq.amax_bf16(gd, ud)
    torch.cuda.synchronize()
    ref = np.float32(max(np.abs((g.astype(np.uint32) << 16).view(np.float32)).max(),
                         np.abs((u.astype(np.uint32) << 16).view(np.float32)).max()))
    assert amax.item() == ref
    for w in (g, u):
        _check(w, scope=float(ref))


def test_nvfp4_moe_shapes():
    """30B-A3B experts: 16384 routed rows x hidden 2048 per token; an expert's
    W_down 2048 x 768 with its tensor scope."""
    x = synth.activation(16384, 2048, seed=7, stream="x")
    _check(x)
    w = synth.weight(2048, 768, seed=7, stream="w_down")
    _check(w, scope=float(np.abs((w.astype(np.uint32) << 16).view(np.float32)).max()))

"""NVFP4 GEMM on the GPU (block-scaled FP4 MMA, scope scales in the epilogue)
against the FP64 oracle on the exactly dequantized NVFP4 operands.

The Miles post on Blackwell-native RL recipes (NVFP4 section) quantizes MoE
expert activations per token and weights per tensor; each output must meet
the bound every GEMM here meets: |y - y_ref| <= 1e-5 * sum_k |a_k b_k|, with
y_ref and the bound from oracle.fprop on oracle.dequant_nvfp4 operands.  BF16
outputs equal the round-to-nearest-even of the FP32 run.  The scale-atom
conversion is a byte permutation, checked against the layout formula.
"""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, f32bits, to_dev_bf16, u8

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _atoms_reference(sb: np.ndarray, k: int) -> np.ndarray:
    """The documented atom layout, written out with numpy indexing."""
    R = sb.shape[0]
    RB = (R + 127) // 128
    out = np.zeros(RB * (k // 256) * 4 * 512, np.uint8)
    r = np.arange(R)[:, None]
    j = np.arange(k // 16)[None, :]  # 16-value block index
    kk = j * 16
    off = (((kk // 256) * RB + r // 128) * 4 + (kk % 256) // 64) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 \
        + (kk % 64) // 16
    out[off] = sb
    return out


@pytest.mark.parametrize("R,K", [(1, 256), (300, 512), (128, 1024), (257, 2048)])
def test_scale_atoms_are_the_documented_permutation(R, K):
    rng = np.random.default_rng(R + K)
    sb = rng.integers(0, 0x7F, (R, K // 16), dtype=np.uint8)
    atoms = jq.nvfp4_atoms(torch.from_numpy(sb).to(DEV), K)
    torch.cuda.synchronize()
    assert atoms.numel() == jq.jetq_nvfp4_atom_bytes(R, K)
    assert np.array_equal(u8(atoms), _atoms_reference(sb, K))


def _quant(x, scope=None):
    d = to_dev_bf16(x)
    amax = None if scope is None else torch.tensor([scope], dtype=torch.float32, device=DEV)
    g = jq.quant_nvfp4(d, scope_amax=amax)
    g["atoms"] = jq.nvfp4_atoms(g["sb"], x.shape[1])
    return g


def _oracle_operand(x, g, scope=None):
    q, sb, sg = oracle.quant_nvfp4(x, scope_amax=scope)
    # the GPU operands are the oracle's, byte for byte
    assert np.array_equal(u8(g["q"]), q) and np.array_equal(u8(g["sb"]), sb)
    assert np.array_equal(f32bits(g["sg"]), f32bits(sg))
    return oracle.dequant_nvfp4(q, sb, sg)


@pytest.mark.parametrize("M,N,K", [(300, 384, 512), (1, 128, 256), (129, 256, 768), (256, 512, 1024),
                                   (64, 1536, 2048)])
def test_nvfp4_fprop_against_oracle(M, N, K):
    x = synth.activation(M, K, seed=M + K, stream="x")
    w = synth.weight(N, K, seed=N + K, stream="w")
    wscope = float(np.abs(synth.bf16_to_f32(w)).max()) * 1.5  # a tensor scope wider than W (a gate/up pair)
    gx, gw = _quant(x), _quant(w, wscope)
    y = jq.nvfp4_fprop(gx, gw, K)
    y16 = jq.nvfp4_fprop(gx, gw, K, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    X = _oracle_operand(x, gx)
    W = _oracle_operand(w, gw, wscope)
    assert_gemm_close(y, *oracle.fprop(X, W))
    assert torch.equal(y.to(torch.bfloat16), y16)


def test_nvfp4_fprop_zero_rows_and_repeatable():
    M, N, K = 200, 256, 512
    x = synth.activation(M, K, seed=5, stream="x")
    x[17] = 0          # a zero row: scope scale 0, output row 0
    x[18] = 0x8000     # -0.0 everywhere
    w = synth.weight(N, K, seed=6, stream="w")
    gx, gw = _quant(x), _quant(w, float(np.abs(synth.bf16_to_f32(w)).max()))
    ys = [jq.nvfp4_fprop(gx, gw, K) for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32))
    assert not ys[0][17].abs().any() and not ys[0][18].abs().any()


def test_nvfp4_fprop_moe_expert_full_size_sampled():
    """The 30B-A3B MoE shape: the largest expert's routed rows (15539 of 131072)
    x hidden 2048 against the fused gate/up expert weight (1536 x 2048), tensor
    scope shared by gate and up; 4096 sampled outputs."""
    M, N, K = 15539, 1536, 2048
    x = synth.activation(M, K, seed=0, stream="x")
    w = synth.weight(N, K, seed=0, stream="w_gate")
    gx = _quant(x)
    wd = to_dev_bf16(w)
    amax = jq.amax_bf16(wd)
    gw = jq.quant_nvfp4(wd, scope_amax=amax)
    gw["atoms"] = jq.nvfp4_atoms(gw["sb"], K)
    y = jq.nvfp4_fprop(gx, gw, K)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    X = _oracle_operand(x, gx)
    W = _oracle_operand(w, gw, float(amax.item()))
    rng = np.random.default_rng(7)
    at = np.stack([rng.integers(0, M, 4096), rng.integers(0, N, 4096)], 1).astype(np.int64)
    at[:4] = [[0, 0], [M - 1, N - 1], [0, N - 1], [M - 1, 0]]
    got = y[torch.as_tensor(at[:, 0], device=DEV), torch.as_tensor(at[:, 1], device=DEV)]
    assert_gemm_close(got, *oracle.fprop(X, W, at=at))

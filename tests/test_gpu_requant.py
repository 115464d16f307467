"""Column copy re-quantized from the FP8 row copy, and the BF16 dequantizer, on
the GPU: bit-exact against the oracle (both follow the same single-rounding
definitions), and a WGrad on re-quantized copies within the FP64 bound."""
import numpy as np
import pytest
import torch

import oracle
import rollout_x128_act_gb300 as jq
import synth
from _gpu import assert_gemm_close, to_dev_bf16, u8

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _row_copy(x):
    a = jq.quant_act(to_dev_bf16(x), col=False)
    return a["q_row"], a["s_row"]


@pytest.mark.parametrize("kind", ["random", "outliers", "ragged", "segments", "zeros"])
def test_requant_col_bit_exact(kind):
    R, C = (300, 384) if kind in ("ragged", "segments") else (256, 512)
    x = np.zeros((R, C), np.uint16) if kind == "zeros" else synth.activation(R, C, seed=51, stream="x")
    if kind == "zeros":
        x[1::3] = 0x8000  # negative zeros: code 0x80 in both copies
    if kind == "outliers":
        x[::5, ::11] = synth.bf16_bits(np.full(((R + 4) // 5, (C + 10) // 11), -2.5e4, np.float32))
    off = np.array([0, 90, 90, 217, 300], dtype=np.int64) if kind == "segments" else None
    seg = None if off is None else torch.tensor(off, dtype=torch.int64, device=DEV)
    q_row, s_row = _row_copy(x)
    g = jq.requant_col(q_row, s_row, seg_offsets=seg)
    torch.cuda.synchronize()
    qc, sc = oracle.requant_colgroups(u8(q_row), s_row.cpu().numpy(), offsets=off)
    P = qc.shape[1]
    assert np.array_equal(u8(g["q_col"])[:, :P], qc)
    assert np.array_equal(g["s_col"].cpu().numpy()[:P // 128].view(np.uint32), sc.view(np.uint32))


@pytest.mark.parametrize("mids", [
    [1.0625, 1.1875, 1.9375, 0.53125, 3.75, 7.5, 240.0, 416.0, 0.01953125, 0.017578125, 0.0029296875],
    [k * 2.0 ** -10 for k in (1, 3, 5, 7, 9, 11, 13, 15)] + [0.0146484375 * 2, 0.5078125],
], ids=["normal", "subnormal-codes"])
def test_requant_quotients_near_e4m3_midpoints(mids):
    """Codes of 1.0 make each rebuilt value its row scale, so the values can be placed
    at S * m nudged by -4..+4 binary32 ulps for E4M3 midpoints m: both sides of the
    fast quotient's guard, in the normal range and among the subnormal codes (odd
    multiples of 2^-10)."""
    amax = np.float32(448.0 * 1.2345678)
    S = np.float32(amax / np.float32(448.0))
    vals = [amax]
    for m in mids:
        base = np.float32(np.float32(m) * S)
        for k in range(-4, 5):
            v = base
            for _ in range(abs(k)):
                v = np.nextafter(v, np.float32(np.inf) if k > 0 else np.float32(0))
            vals.append(v)
    vals = np.array(vals, np.float32)
    R = 128
    assert len(vals) <= R
    s_row = np.zeros((1, R), np.float32)
    s_row[0, :len(vals)] = vals
    s_row[0, len(vals):] = -vals[1:R - len(vals) + 1]  # negative copies fill the group
    q_row = np.full((R, 128), 0x38, np.uint8)
    g = jq.requant_col(torch.as_tensor(q_row, device=DEV), torch.as_tensor(s_row, device=DEV))
    torch.cuda.synchronize()
    qc, sc = oracle.requant_colgroups(q_row, s_row)
    assert sc[0, 0] == S
    assert np.array_equal(u8(g["q_col"]), qc)


def test_requant_col_full_size_sampled():
    R, C = 8192, 12288
    x = synth.activation(R, C, seed=52, stream="h")
    q_row, s_row = _row_copy(x)
    g = jq.requant_col(q_row, s_row)
    torch.cuda.synchronize()
    qr, sr = u8(q_row), s_row.cpu().numpy()
    rng = np.random.default_rng(0)
    for gi in rng.integers(0, R // 128, 6):
        lo = int(gi) * 128
        cols = np.unique(np.concatenate([[0, C - 1], rng.integers(0, C, 30)]))
        qc, sc = oracle.requant_colgroups(qr[lo:lo + 128], sr[:, lo:lo + 128])
        got = u8(g["q_col"][torch.as_tensor(cols, device=DEV), lo:lo + 128])
        assert np.array_equal(got, qc[cols])
        assert np.array_equal(g["s_col"][gi, torch.as_tensor(cols, device=DEV)].cpu().numpy(), sc[0, cols])


def test_dequant_bf16_bit_exact():
    x = synth.activation(300, 256, seed=53, stream="x")
    q_row, s_row = _row_copy(x)
    # full 24-bit scale significands make the rounding of the product matter
    s_full = (s_row * 1.2345678).contiguous()
    out = jq.dequant_bf16(q_row, s_full)
    w = synth.weight(384, 256, seed=53, stream="w")
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(w), transposed=False)
    sw_full = (sw * 0.987654321).contiguous()
    outw = jq.dequant_bf16(qw, sw_full, jq.SCALES_BLOCKS_128X128)
    torch.cuda.synchronize()
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16),
                          oracle.dequant_rowgroups_bf16(u8(q_row), s_full.cpu().numpy()))
    assert np.array_equal(outw.view(torch.int16).cpu().numpy().view(np.uint16),
                          oracle.dequant_blocks_bf16(u8(qw), sw_full.cpu().numpy()))


def test_dequant_bf16_ties_and_tiny_products():
    # decode(0x38) = 1, so the products are the scales themselves: a BF16 midpoint
    # (ties to even), just above / below it, and products in the binary64 range
    tie = np.float32(1.0 + 2.0 ** -8)
    s = np.array([tie, np.nextafter(tie, np.float32(2)), np.nextafter(tie, np.float32(0)),
                  np.float32(3.0e-35), np.float32(1.17e-38), np.float32(7.0e-39)], np.float32)
    R = len(s)
    q = np.full((R, 128), 0x38, np.uint8)
    q[:, 1] = 0x7E  # 448
    q[:, 2] = 0xB9  # -1.125
    qd = torch.as_tensor(q, device=DEV)
    sd = torch.as_tensor(s.reshape(1, R), device=DEV)
    out = jq.dequant_bf16(qd, sd)
    torch.cuda.synchronize()
    ref = oracle.dequant_rowgroups_bf16(q, s.reshape(1, R))
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), ref)
    assert ref[0, 0] == 0x3F80 and ref[1, 0] == 0x3F81 and ref[2, 0] == 0x3F80


def test_wgrad_on_requantized_copies():
    N, D, C = 384, 256, 512
    x = synth.activation(N, C, seed=54, stream="x")
    dy = synth.gradient(N, D, seed=54, stream="dy")
    gx = jq.requant_col(*_row_copy(x))
    gdy = jq.requant_col(*_row_copy(dy))
    dw = jq.wgrad(gdy["q_col"], gdy["s_col"], gx["q_col"], gx["s_col"], gx["ldq_col"])
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    Xc = oracle.dequant_colgroups(*oracle.requant_colgroups(*oracle.quant_rowgroups(x)), N)
    DYc = oracle.dequant_colgroups(*oracle.requant_colgroups(*oracle.quant_rowgroups(dy)), N)
    assert_gemm_close(dw, *oracle.wgrad(DYc, Xc))

"""The C ABI library: it builds, loads, exports every symbol include/jetq.h
declares, and its host-side validation rejects bad arguments before any
CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "jetq.h")


@pytest.fixture(scope="module")
def L():
    from rollout_x128_act_gb300 import build

    build.build()
    import rollout_x128_act_gb300 as jq

    return jq.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"JETQ_API[^;(]*?\b(jetq_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("jetq_quant_act_1x128", "jetq_quant_w_128x128", "jetq_quant_mx32", "jetq_gemm_fprop",
                     "jetq_gemm_dgrad", "jetq_gemm_wgrad", "jetq_check_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def _declarations():
    text = open(HEADER).read()
    out = {}
    for name, params in re.findall(r"JETQ_API\s+[\w\s\*]+?\b(jetq_\w+)\s*\(([^;]*?)\)\s*;", text, re.S):
        p = " ".join(params.split())
        out[name] = [] if p in ("", "void") else [x.strip() for x in p.split(",")]
    return out


def _ctype_of(param):
    """The ctypes type the binding must pass for one C parameter declaration."""
    if "*" in param:
        return ctypes.c_void_p
    base = param.rsplit(" ", 1)[0].replace("const ", "").strip()
    if base in re.findall(r"}\s*(jetq_\w+)\s*;", open(HEADER).read()):  # the header's enums
        return ctypes.c_int
    return {"int64_t": ctypes.c_int64, "int": ctypes.c_int, "float": ctypes.c_float, "uint64_t": ctypes.c_uint64,
            "size_t": ctypes.c_size_t}[base]


def test_binding_matches_every_declaration(L):
    """The ctypes binding passes exactly the parameters the header declares, with
    matching widths (a pointer, a 64-bit or 32-bit integer, a float)."""
    decl = _declarations()
    assert decl, "no declarations parsed"
    for name, params in decl.items():
        fn = getattr(L, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), len(params))
        for got, param in zip(fn.argtypes, params):
            want = _ctype_of(param)
            assert ctypes.sizeof(got) == ctypes.sizeof(want), (name, param, got, want)
            assert (got is ctypes.c_float) == (want is ctypes.c_float), (name, param)


def test_status_strings_and_sizes(L):
    import rollout_x128_act_gb300 as jq

    assert jq.status_string(0) == "ok"
    assert "aligned" in jq.status_string(3)
    assert jq.jetq_version() >= 100
    assert jq.jetq_colcopy_capacity(0, 1) == 0
    assert jq.jetq_colcopy_capacity(1, 1) == 128
    assert jq.jetq_colcopy_capacity(8192, 1) == 8192
    assert jq.jetq_colcopy_capacity(300, 4) >= 128 + 128 + 256  # worst case of 4 ragged segments
    assert jq.jetq_mx_scale_bytes(1, 128) == 512
    assert jq.jetq_mx_scale_bytes(8192, 4096) == 64 * 32 * 512
    assert jq.jetq_mx_scale_bytes(2048, 768) == 16 * 6 * 512


def test_validation_happens_before_cuda(L):
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: every call below fails validation first
    # C not a multiple of 128
    assert L.jetq_quant_act_1x128(fake, 4, 100, 100, fake, fake, None, None, 0, None, 0, None) == 2
    # q_row without s_row
    assert L.jetq_quant_act_1x128(fake, 4, 128, 128, fake, None, None, None, 0, None, 0, None) == 1
    # column copy too short
    assert L.jetq_quant_act_1x128(fake, 300, 128, 128, None, None, fake, fake, 256, None, 0, None) == 2
    # weight with D not a multiple of 128
    assert L.jetq_quant_w_128x128(fake, 100, 128, 128, fake, fake, None, None, None) == 2
    # misaligned weight pointer
    assert L.jetq_quant_w_128x128(P(4097), 128, 128, 128, fake, fake, None, None, None) == 3
    # GEMM: bad recipe, bad path, bad output stride, misaligned output
    assert L.jetq_gemm_fprop(7, fake, fake, fake, fake, 8, 128, 128, fake, 0, 128, 0, None) == 1
    assert L.jetq_gemm_fprop(0, fake, fake, fake, fake, 8, 128, 128, fake, 0, 128, 9, None) == 1
    assert L.jetq_gemm_fprop(0, fake, fake, fake, fake, 8, 128, 128, fake, 0, 64, 0, None) == 2
    assert L.jetq_gemm_fprop(0, fake, fake, fake, fake, 8, 128, 128, P(4100), 0, 128, 0, None) == 3
    assert L.jetq_gemm_dgrad(0, fake, fake, fake, fake, 8, 100, 128, fake, 0, 128, None) == 2
    # WGrad: K not a multiple of 128, ldk smaller than K
    assert L.jetq_gemm_wgrad(0, fake, fake, fake, fake, 200, 256, 128, 128, fake, 128, 0, None) == 2
    assert L.jetq_gemm_wgrad(0, fake, fake, fake, fake, 256, 128, 128, 128, fake, 128, 0, None) == 2
    # bounded-wait diagnostic: limit outside [1 ms, 1 s], null or misaligned output
    assert L.jetq_selftest_bounded_wait(ctypes.c_uint64(999_999), fake, None) == 1
    assert L.jetq_selftest_bounded_wait(ctypes.c_uint64(2_000_000_000), fake, None) == 1
    assert L.jetq_selftest_bounded_wait(ctypes.c_uint64(50_000_000), None, None) == 1
    assert L.jetq_selftest_bounded_wait(ctypes.c_uint64(50_000_000), P(4100), None) == 3
    # fused producers: c above 32768 (RMSNorm statistics), eps out of range, missing rstd,
    # misaligned weight; SwiGLU up stride below c, misaligned up
    F = ctypes.c_float
    assert L.jetq_quant_act_1x128_rmsnorm(fake, 4, 32896, 32896, fake, F(1e-6), fake, fake, fake, None, None, 0,
                                          None, 0, None) == 2
    assert L.jetq_quant_act_1x128_rmsnorm(fake, 4, 128, 128, fake, F(-1.0), fake, fake, fake, None, None, 0,
                                          None, 0, None) == 1
    assert L.jetq_quant_act_1x128_rmsnorm(fake, 4, 128, 128, fake, F(1e-6), None, fake, fake, None, None, 0,
                                          None, 0, None) == 1
    assert L.jetq_quant_act_1x128_rmsnorm(fake, 4, 128, 128, P(4098), F(1e-6), fake, fake, fake, None, None, 0,
                                          None, 0, None) == 3
    assert L.jetq_quant_act_1x128_swiglu(fake, fake, 4, 256, 256, 128, fake, fake, None, None, 0, None, 0,
                                         None) == 2
    assert L.jetq_quant_act_1x128_swiglu(fake, P(4104), 4, 128, 128, 128, fake, fake, None, None, 0, None, 0,
                                         None) == 3
    # re-quantizer: channels not a multiple of 128; column copy too short
    assert L.jetq_requant_col_from_row(fake, fake, 4, 100, fake, fake, 128, None, 0, None) == 2
    assert L.jetq_requant_col_from_row(fake, fake, 300, 128, fake, fake, 256, None, 0, None) == 2
    # dequantizer: unknown scale layout; 128x128 blocks need rows % 128 == 0
    assert L.jetq_dequant_bf16(fake, fake, 4, 128, 5, fake, 128, None) == 1
    assert L.jetq_dequant_bf16(fake, fake, 100, 128, 1, fake, 128, None) == 2
    # power-of-two weight blocks: a transposed copy without its scales
    assert L.jetq_quant_w_128x128_pow2(fake, 128, 128, 128, fake, fake, fake, None, None) == 1
    # grouped GEMM: unknown kind; more than 256 experts
    #   (kind, recipe, a, sa, b, sb, m, n, k, ldk, seg_offsets, num_experts, out, out_dtype, ldo, accumulate, stream)
    assert L.jetq_gemm_grouped(7, 0, fake, fake, fake, fake, 128, 128, 128, 128, fake, 4, fake, 0, 128, 0,
                               None) == 1
    assert L.jetq_gemm_grouped(0, 0, fake, fake, fake, fake, 128, 128, 128, 128, fake, 300, fake, 0, 128, 0,
                               None) == 2
    # NVFP4: columns not a multiple of 16, misaligned packed codes, bad scope flag
    assert L.jetq_quant_nvfp4(fake, 4, 40, 40, None, fake, fake, fake, None) == 2
    assert L.jetq_quant_nvfp4(fake, 4, 32, 32, None, P(4098), fake, fake, None) == 3
    assert L.jetq_dequant_nvfp4_bf16(fake, fake, fake, 2, 4, 32, fake, 32, None) == 1
    assert L.jetq_amax_bf16(fake, 4, 12, 12, fake, None) == 2
    # MX: columns not a multiple of 128
    assert L.jetq_quant_mx32(fake, 4, 96, 96, fake, fake, None, None, 0, None, 0, None) == 2
    # FProp with a workspace: misaligned workspace; D not a multiple of 128
    assert L.jetq_gemm_fprop_ws(0, fake, fake, fake, fake, 8, 128, 128, fake, 0, 128, P(4100), 1024, 2, None) == 3
    assert L.jetq_gemm_fprop_ws(0, fake, fake, fake, fake, 8, 100, 128, fake, 0, 128, fake, 1024, 2, None) == 2
    # allocation-free FProp: D not a multiple of 128; negative batch
    assert L.jetq_gemm_fprop_noalloc(fake, fake, fake, fake, 8, 100, 128, fake, 0, 128, None) == 2
    assert L.jetq_gemm_fprop_noalloc(fake, fake, fake, fake, -1, 128, 128, fake, 0, 128, None) == 1


def test_decode_workspace_size_is_zero_without_the_device(L):
    """The size query needs the GB300 (its SM count picks the split): on any other
    device, or none, it reports that no workspace is used."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert L.jetq_decode_workspace_bytes(1, 4096, 12288) == 0
    assert L.jetq_decode_workspace_bytes(0, 4096, 12288) == 0

"""The allocation-free rollout FProp, jetq_gemm_fprop_noalloc.

Some callers cannot give the library device memory for a workspace: a
framework whose caching allocator must own every allocation, a serving loop
that cannot stop for the device-wide synchronization of cudaMalloc, or a
plugin host that passes only a stream and its buffers.  For them the split-K
decode keeps its partial sums in a scratch array built into the library.
This file checks, through the C ABI, that two calls in a row give exactly the
output of the existing entry points (the split-K decode with a caller-owned
workspace, and the one-CTA decode), and that a shape whose partials do not fit
the array is refused.  It sits last in the collection order, so a run that
stops at the first failure has run every other test before it.
"""
import pytest
import torch

import rollout_x128_act_gb300 as jq
import synth
from _gpu import to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _operands(n, d, c, seed):
    x = synth.activation(n, c, seed=seed, stream="x")
    w = synth.weight(d, c, seed=seed, stream="w_down")
    qw, sw, _, _ = jq.quant_weight(to_dev_bf16(w), transposed=False)
    a = jq.quant_act(to_dev_bf16(x), col=False)
    return a["q_row"], a["s_row"], qw, sw


def _reference(q, s, qw, sw, n, d, c, dtype):
    """The existing entry points on the same operands: with a workspace, and without."""
    y_ws = torch.empty((n, d), dtype=dtype, device=DEV)
    work = torch.empty(max(jq.jetq_decode_workspace_bytes(n, d, c), 16), dtype=torch.uint8, device=DEV)
    jq.jetq_gemm_fprop_ws(jq.RECIPE_BLOCK128, q, s, qw, sw, n, d, c, y_ws, work, jq.PATH_DECODE)
    y_one = torch.empty((n, d), dtype=dtype, device=DEV)
    jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, q, s, qw, sw, n, d, c, y_one, jq.PATH_DECODE)
    return y_ws, y_one


def _bits(y):
    return y.view(torch.int32 if y.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_two_calls_in_a_row_match_the_workspace_entry_point(dtype):
    # the dense-8B down projection (4096 x 12288, a 4-CTA cluster per row band):
    # 8 tokens then 1 token, so the second call reads the array after the first
    # left other partials in it
    d, c = 4096, 12288
    for n, seed in ((8, 21), (1, 22)):
        assert 0 < jq.jetq_decode_workspace_bytes(n, d, c) <= jq.NOALLOC_SCRATCH_BYTES
        q, s, qw, sw = _operands(n, d, c, seed)
        y = torch.empty((n, d), dtype=dtype, device=DEV)
        jq.jetq_gemm_fprop_noalloc(q, s, qw, sw, n, d, c, y)
        y_ws, y_one = _reference(q, s, qw, sw, n, d, c, dtype)
        torch.cuda.synchronize()
        assert jq.jetq_check_device_error() == jq.OK
        assert torch.equal(_bits(y), _bits(y_ws)), n
        assert torch.equal(_bits(y), _bits(y_one)), n


def test_repeated_calls_on_one_input_are_identical():
    d, c, n = 4096, 2176, 17  # a partial last chunk; 32 token columns
    q, s, qw, sw = _operands(n, d, c, 23)
    ys = [torch.empty((n, d), dtype=torch.float32, device=DEV) for _ in range(2)]
    for y in ys:
        jq.jetq_gemm_fprop_noalloc(q, s, qw, sw, n, d, c, y)
    y_ws, _ = _reference(q, s, qw, sw, n, d, c, torch.float32)
    torch.cuda.synchronize()
    assert jq.jetq_check_device_error() == jq.OK
    assert torch.equal(_bits(ys[0]), _bits(y_ws))
    assert torch.equal(_bits(ys[1]), _bits(y_ws))


def test_a_shape_beyond_the_array_is_refused():
    # 32 tokens against the down projection need 4096 x 96 x 32 x 4 bytes = 48 MiB
    d, c, n = 4096, 12288, 32
    assert jq.jetq_decode_workspace_bytes(n, d, c) > jq.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((n, c), dtype=torch.uint8, device=DEV)
    s = torch.ones((c // 128, n), dtype=torch.float32, device=DEV)
    qw = torch.zeros((d, c), dtype=torch.uint8, device=DEV)
    sw = torch.ones((d // 128, c // 128), dtype=torch.float32, device=DEV)
    y = torch.empty((n, d), dtype=torch.float32, device=DEV)
    with pytest.raises(jq.JetqError) as refused:
        jq.jetq_gemm_fprop_noalloc(q, s, qw, sw, n, d, c, y)
    assert refused.value.status == jq.ERR_UNSUPPORTED_SHAPE  # refused before any launch

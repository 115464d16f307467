"""Python binding of the jetq C ABI (``include/jetq.h``).

Argument marshalling only: every function passes device pointers, sizes and
the current CUDA stream to ``_build/libjetq.so`` and raises ``JetqError`` on a
non-OK status.  PyTorch supplies device memory and streams.  There is no CPU
fallback: without the compiled library every call raises.

The ``jetq_*`` functions mirror the C entry points one to one.  The short
helpers below them (``quant_act``, ``quant_weight``, ``quant_mx``, ``fprop``,
``dgrad``, ``wgrad``) only allocate the output tensors with torch and call the
matching ``jetq_*`` function.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libjetq.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_ARCH, ERR_CUDA, ERR_TIMEOUT = range(7)
RECIPE_BLOCK128, RECIPE_MXFP8, RECIPE_BLOCK128_POW2 = 0, 1, 2
PATH_AUTO, PATH_TRAIN, PATH_DECODE = 0, 1, 2
GEMM_FPROP, GEMM_DGRAD, GEMM_WGRAD = 0, 1, 2
OUT_F32, OUT_BF16 = 0, 1

_lock = threading.Lock()
_lib = None


class JetqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"jetq CUDA library missing ({LIB_PATH}); build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        sig = {
            "jetq_status_string": (ctypes.c_char_p, [I32]),
            "jetq_version": (I32, []),
            "jetq_check_device_error": (I32, [P]),
            "jetq_selftest_bounded_wait": (I32, [ctypes.c_uint64, P, P]),
            "jetq_colcopy_capacity": (I64, [I64, I32]),
            "jetq_mx_scale_bytes": (I64, [I64, I64]),
            "jetq_quant_act_1x128": (I32, [P, I64, I64, I64, P, P, P, P, I64, P, I32, P]),
            "jetq_quant_act_1x128_rmsnorm": (I32, [P, I64, I64, I64, P, ctypes.c_float, P, P, P, P, P, I64, P, I32,
                                                   P]),
            "jetq_quant_act_1x128_swiglu": (I32, [P, P, I64, I64, I64, I64, P, P, P, P, I64, P, I32, P]),
            "jetq_quant_w_128x128": (I32, [P, I64, I64, I64, P, P, P, P, P]),
            "jetq_amax_bf16": (I32, [P, I64, I64, I64, P, P]),
            "jetq_quant_nvfp4": (I32, [P, I64, I64, I64, P, P, P, P, P]),
            "jetq_dequant_nvfp4_bf16": (I32, [P, P, P, I32, I64, I64, P, I64, P]),
            "jetq_quant_mx32": (I32, [P, I64, I64, I64, P, P, P, P, I64, P, I32, P]),
            "jetq_quant_act_1x128_pow2": (I32, [P, I64, I64, I64, P, P, P, P, I64, P, I32, P]),
            "jetq_quant_w_128x128_pow2": (I32, [P, I64, I64, I64, P, P, P, P, P]),
            "jetq_requant_col_from_row": (I32, [P, P, I64, I64, P, P, I64, P, I32, P]),
            "jetq_dequant_bf16": (I32, [P, P, I64, I64, I32, P, I64, P]),
            "jetq_gemm_fprop": (I32, [I32, P, P, P, P, I64, I64, I64, P, I32, I64, I32, P]),
            "jetq_decode_workspace_bytes": (ctypes.c_size_t, [I64, I64, I64]),
            "jetq_gemm_fprop_ws": (I32, [I32, P, P, P, P, I64, I64, I64, P, I32, I64, P, ctypes.c_size_t, I32, P]),
            "jetq_gemm_fprop_noalloc": (I32, [P, P, P, P, I64, I64, I64, P, I32, I64, P]),
            "jetq_gemm_dgrad": (I32, [I32, P, P, P, P, I64, I64, I64, P, I32, I64, P]),
            "jetq_gemm_wgrad": (I32, [I32, P, P, P, P, I64, I64, I64, I64, P, I64, I32, P]),
            "jetq_gemm_grouped": (I32, [I32, I32, P, P, P, P, I64, I64, I64, I64, P, I32, P, I32, I64, I32, P]),
            "jetq_nvfp4_atom_bytes": (I64, [I64, I64]),
            "jetq_nvfp4_scale_atoms": (I32, [P, I64, I64, P, P]),
            "jetq_gemm_nvfp4": (I32, [P, P, P, I32, P, P, P, I64, I64, I64, P, I32, I64, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return lib().jetq_status_string(int(status)).decode()
    except RuntimeError:
        return "unknown"


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != OK:
        raise JetqError(status, where)


# ------------------------------------------------------------------ C entry points

def jetq_version() -> int:
    return int(lib().jetq_version())


def jetq_check_device_error(stream=None) -> int:
    return int(lib().jetq_check_device_error(_s(stream)))


def jetq_selftest_bounded_wait(limit_ns: int, elapsed_ns, stream=None) -> int:
    """Launch the bounded-wait diagnostic; elapsed_ns: int64 CUDA tensor of 2."""
    return int(lib().jetq_selftest_bounded_wait(int(limit_ns), _p(elapsed_ns), _s(stream)))


def jetq_colcopy_capacity(n: int, nseg: int = 1) -> int:
    return int(lib().jetq_colcopy_capacity(n, nseg))


def jetq_mx_scale_bytes(rows: int, k: int) -> int:
    return int(lib().jetq_mx_scale_bytes(rows, k))


def jetq_quant_act_1x128(x, q_row, s_row, q_col, s_col, ldq_col, seg_offsets=None, nseg=0, stream=None):
    n, c = x.shape
    _check(lib().jetq_quant_act_1x128(_p(x), n, c, x.stride(0), _p(q_row), _p(s_row), _p(q_col), _p(s_col),
                                      ldq_col, _p(seg_offsets), nseg, _s(stream)), "jetq_quant_act_1x128")


def jetq_quant_act_1x128_rmsnorm(x, w, eps, rstd, q_row, s_row, q_col, s_col, ldq_col, seg_offsets=None, nseg=0,
                                 stream=None):
    n, c = x.shape
    _check(lib().jetq_quant_act_1x128_rmsnorm(_p(x), n, c, x.stride(0), _p(w), float(eps), _p(rstd), _p(q_row),
                                              _p(s_row), _p(q_col), _p(s_col), ldq_col, _p(seg_offsets), nseg,
                                              _s(stream)), "jetq_quant_act_1x128_rmsnorm")


def jetq_quant_act_1x128_swiglu(gate, up, q_row, s_row, q_col, s_col, ldq_col, seg_offsets=None, nseg=0, stream=None):
    n, c = gate.shape
    assert up.shape == gate.shape
    _check(lib().jetq_quant_act_1x128_swiglu(_p(gate), _p(up), n, c, gate.stride(0), up.stride(0), _p(q_row),
                                             _p(s_row), _p(q_col), _p(s_col), ldq_col, _p(seg_offsets), nseg,
                                             _s(stream)), "jetq_quant_act_1x128_swiglu")


def jetq_amax_bf16(x, amax, stream=None):
    r, c = x.shape
    _check(lib().jetq_amax_bf16(_p(x), r, c, x.stride(0), _p(amax), _s(stream)), "jetq_amax_bf16")


def jetq_quant_nvfp4(x, q, sb, sg, scope_amax=None, stream=None):
    r, c = x.shape
    _check(lib().jetq_quant_nvfp4(_p(x), r, c, x.stride(0), _p(scope_amax), _p(q), _p(sb), _p(sg), _s(stream)),
           "jetq_quant_nvfp4")


def jetq_dequant_nvfp4_bf16(q, sb, sg, per_row, out, stream=None):
    r, c = out.shape
    _check(lib().jetq_dequant_nvfp4_bf16(_p(q), _p(sb), _p(sg), int(per_row), r, c, _p(out), out.stride(0),
                                         _s(stream)), "jetq_dequant_nvfp4_bf16")


def jetq_nvfp4_atom_bytes(rows: int, k: int) -> int:
    return int(lib().jetq_nvfp4_atom_bytes(rows, k))


def jetq_nvfp4_scale_atoms(sb, rows, k, atoms, stream=None):
    _check(lib().jetq_nvfp4_scale_atoms(_p(sb), rows, k, _p(atoms), _s(stream)), "jetq_nvfp4_scale_atoms")


def jetq_gemm_nvfp4(qa, sfa, sga, per_row_a, qb, sfb, sgb, m, n, k, out, stream=None):
    _check(lib().jetq_gemm_nvfp4(_p(qa), _p(sfa), _p(sga), int(per_row_a), _p(qb), _p(sfb), _p(sgb), m, n, k,
                                 _p(out), _out_dtype(out), out.stride(0), _s(stream)), "jetq_gemm_nvfp4")


def jetq_quant_w_128x128(w, q, s, qT=None, sT=None, stream=None):
    d, c = w.shape
    _check(lib().jetq_quant_w_128x128(_p(w), d, c, w.stride(0), _p(q), _p(s), _p(qT), _p(sT), _s(stream)),
           "jetq_quant_w_128x128")


def jetq_quant_mx32(x, q_row, e8_row, q_col, e8_col, ldq_col, seg_offsets=None, nseg=0, stream=None):
    r, c = x.shape
    _check(lib().jetq_quant_mx32(_p(x), r, c, x.stride(0), _p(q_row), _p(e8_row), _p(q_col), _p(e8_col),
                                 ldq_col, _p(seg_offsets), nseg, _s(stream)), "jetq_quant_mx32")


def jetq_quant_act_1x128_pow2(x, q_row, e8_row, q_col, e8_col, ldq_col, seg_offsets=None, nseg=0, stream=None):
    r, c = x.shape
    _check(lib().jetq_quant_act_1x128_pow2(_p(x), r, c, x.stride(0), _p(q_row), _p(e8_row), _p(q_col), _p(e8_col),
                                           ldq_col, _p(seg_offsets), nseg, _s(stream)), "jetq_quant_act_1x128_pow2")


def jetq_quant_w_128x128_pow2(w, q, e8, qT=None, e8T=None, stream=None):
    d, c = w.shape
    _check(lib().jetq_quant_w_128x128_pow2(_p(w), d, c, w.stride(0), _p(q), _p(e8), _p(qT), _p(e8T), _s(stream)),
           "jetq_quant_w_128x128_pow2")


def jetq_requant_col_from_row(q_row, s_row, q_col, s_col, ldq_col, seg_offsets=None, nseg=0, stream=None):
    n, c = q_row.shape
    _check(lib().jetq_requant_col_from_row(_p(q_row), _p(s_row), n, c, _p(q_col), _p(s_col), ldq_col,
                                           _p(seg_offsets), nseg, _s(stream)), "jetq_requant_col_from_row")


SCALES_ROWGROUPS_1X128, SCALES_BLOCKS_128X128 = 0, 1


def jetq_dequant_bf16(q, s, layout, out, stream=None):
    rows, cols = q.shape
    _check(lib().jetq_dequant_bf16(_p(q), _p(s), rows, cols, layout, _p(out), out.stride(0), _s(stream)),
           "jetq_dequant_bf16")


def requant_col(q_row, s_row, seg_offsets=None, stream=None):
    """Column copy (q_col [c x cap], s_col [cap/128 x c], ldq_col) re-quantized from a row copy."""
    n, c = q_row.shape
    nseg = 0 if seg_offsets is None else seg_offsets.numel() - 1
    cap = jetq_colcopy_capacity(n, max(nseg, 1))
    q_col = torch.zeros((c, cap), dtype=torch.uint8, device=q_row.device)
    s_col = torch.zeros((max(cap, 128) // 128, c), dtype=torch.float32, device=q_row.device)
    jetq_requant_col_from_row(q_row, s_row, q_col, s_col, cap, seg_offsets, nseg, stream)
    return dict(q_col=q_col, s_col=s_col, ldq_col=cap)


def dequant_bf16(q, s, layout=SCALES_ROWGROUPS_1X128, stream=None):
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    jetq_dequant_bf16(q, s, layout, out, stream)
    return out


def _out_dtype(t):
    return OUT_BF16 if t.dtype == torch.bfloat16 else OUT_F32


def jetq_gemm_fprop(recipe, qx, sx, qw, sw, n, d, c, y, path=PATH_AUTO, stream=None):
    _check(lib().jetq_gemm_fprop(recipe, _p(qx), _p(sx), _p(qw), _p(sw), n, d, c, _p(y), _out_dtype(y),
                                 y.stride(0), path, _s(stream)), "jetq_gemm_fprop")


def jetq_decode_workspace_bytes(n, d, c):
    return int(lib().jetq_decode_workspace_bytes(n, d, c))


def jetq_gemm_fprop_ws(recipe, qx, sx, qw, sw, n, d, c, y, ws, path=PATH_AUTO, stream=None):
    _check(lib().jetq_gemm_fprop_ws(recipe, _p(qx), _p(sx), _p(qw), _p(sw), n, d, c, _p(y), _out_dtype(y),
                                    y.stride(0), None if ws is None else _p(ws),
                                    0 if ws is None else ws.numel() * ws.element_size(), path, _s(stream)),
           "jetq_gemm_fprop_ws")


NOALLOC_SCRATCH_BYTES = 16 << 20  # JETQ_NOALLOC_SCRATCH_BYTES


def jetq_gemm_fprop_noalloc(qx, sx, qw, sw, n, d, c, y, stream=None):
    """Rollout FProp (128-block recipe, decode path) that allocates nothing: the
    split-K partial sums use a device array built into the library."""
    _check(lib().jetq_gemm_fprop_noalloc(_p(qx), _p(sx), _p(qw), _p(sw), n, d, c, _p(y), _out_dtype(y),
                                         y.stride(0), _s(stream)), "jetq_gemm_fprop_noalloc")


def jetq_gemm_dgrad(recipe, qdy, sdy, qwt, swt, n, d, c, dx, stream=None):
    _check(lib().jetq_gemm_dgrad(recipe, _p(qdy), _p(sdy), _p(qwt), _p(swt), n, d, c, _p(dx), _out_dtype(dx),
                                 dx.stride(0), _s(stream)), "jetq_gemm_dgrad")


def jetq_gemm_wgrad(recipe, qdyc, sdyc, qxc, sxc, k, ldk, d, c, dw, accumulate=False, stream=None):
    _check(lib().jetq_gemm_wgrad(recipe, _p(qdyc), _p(sdyc), _p(qxc), _p(sxc), k, ldk, d, c, _p(dw),
                                 dw.stride(0), 1 if accumulate else 0, _s(stream)), "jetq_gemm_wgrad")


def jetq_gemm_grouped(kind, recipe, a, sa, b, sb, m, n, k, ldk, seg_offsets, num_experts, out, accumulate=False,
                      stream=None):
    _check(lib().jetq_gemm_grouped(kind, recipe, _p(a), _p(sa), _p(b), _p(sb), m, n, k, ldk, _p(seg_offsets),
                                   num_experts, _p(out), _out_dtype(out), out.stride(-2), 1 if accumulate else 0,
                                   _s(stream)), "jetq_gemm_grouped")


# ------------------------------------------------------------------ allocating helpers

def quant_act(x, row=True, col=True, seg_offsets=None, stream=None):
    """BF16 [n x c] -> dict(q_row, s_row, q_col, s_col, ldq_col) (absent copies are None)."""
    n, c = x.shape
    dev = x.device
    nseg = 0 if seg_offsets is None else seg_offsets.numel() - 1
    cap = jetq_colcopy_capacity(n, max(nseg, 1))
    out = dict(q_row=None, s_row=None, q_col=None, s_col=None, ldq_col=cap)
    if row:
        out["q_row"] = torch.empty((n, c), dtype=torch.uint8, device=dev)
        out["s_row"] = torch.empty((c // 128, n), dtype=torch.float32, device=dev)
    if col:
        out["q_col"] = torch.empty((c, cap), dtype=torch.uint8, device=dev)
        out["s_col"] = torch.empty((max(cap, 128) // 128, c), dtype=torch.float32, device=dev)
    jetq_quant_act_1x128(x, out["q_row"], out["s_row"], out["q_col"], out["s_col"], cap, seg_offsets, nseg, stream)
    return out


def _act_copies(n, c, dev, row, col, seg_offsets):
    nseg = 0 if seg_offsets is None else seg_offsets.numel() - 1
    cap = jetq_colcopy_capacity(n, max(nseg, 1))
    out = dict(q_row=None, s_row=None, q_col=None, s_col=None, ldq_col=cap)
    if row:
        out["q_row"] = torch.empty((n, c), dtype=torch.uint8, device=dev)
        out["s_row"] = torch.empty((c // 128, n), dtype=torch.float32, device=dev)
    if col:
        out["q_col"] = torch.empty((c, cap), dtype=torch.uint8, device=dev)
        out["s_col"] = torch.empty((max(cap, 128) // 128, c), dtype=torch.float32, device=dev)
    return out, nseg


def quant_act_rmsnorm(x, w, eps=1e-6, row=True, col=True, seg_offsets=None, stream=None):
    """1x128 copies of RMSNorm(x) * w (BF16, not stored): the quant_act dict plus rstd [n]."""
    n, c = x.shape
    out, nseg = _act_copies(n, c, x.device, row, col, seg_offsets)
    out["rstd"] = torch.empty(n, dtype=torch.float32, device=x.device)
    jetq_quant_act_1x128_rmsnorm(x, w, eps, out["rstd"], out["q_row"], out["s_row"], out["q_col"], out["s_col"],
                                 out["ldq_col"], seg_offsets, nseg, stream)
    return out


def quant_act_swiglu(gate, up, row=True, col=True, seg_offsets=None, stream=None):
    """1x128 copies of silu(gate) * up (BF16, not stored), as the quant_act dict."""
    n, c = gate.shape
    out, nseg = _act_copies(n, c, gate.device, row, col, seg_offsets)
    jetq_quant_act_1x128_swiglu(gate, up, out["q_row"], out["s_row"], out["q_col"], out["s_col"], out["ldq_col"],
                                seg_offsets, nseg, stream)
    return out


def quant_nvfp4(x, scope_amax=None, stream=None):
    """NVFP4 copy of BF16 x: dict(q [r x c/2] u8, sb [r x c/16] u8, sg [r] or [1] f32).
    scope_amax: a device float tensor (tensor scope) or None (one scope per row)."""
    r, c = x.shape
    dev = x.device
    out = dict(q=torch.empty((r, c // 2), dtype=torch.uint8, device=dev),
               sb=torch.empty((r, c // 16), dtype=torch.uint8, device=dev),
               sg=torch.empty(r if scope_amax is None else 1, dtype=torch.float32, device=dev))
    jetq_quant_nvfp4(x, out["q"], out["sb"], out["sg"], scope_amax, stream)
    return out


def amax_bf16(*tensors, stream=None):
    """max |x| over one or more BF16 tensors, as a device float tensor of one element."""
    a = torch.zeros(1, dtype=torch.float32, device=tensors[0].device)
    for t in tensors:
        jetq_amax_bf16(t, a, stream)
    return a


def dequant_nvfp4_bf16(q, sb, sg, stream=None):
    """BF16 values of an NVFP4 copy (per-row scope when sg has one entry per row)."""
    r = q.shape[0]
    out = torch.empty((r, q.shape[1] * 2), dtype=torch.bfloat16, device=q.device)
    jetq_dequant_nvfp4_bf16(q, sb, sg, sg.numel() > 1, out, stream)
    return out


def nvfp4_atoms(sb, k, stream=None):
    """Scale atoms (the block-scaled FP4 MMA's layout) of row-major NVFP4 block scales sb [rows x k/16]."""
    rows = sb.shape[0]
    atoms = torch.empty(jetq_nvfp4_atom_bytes(rows, k), dtype=torch.uint8, device=sb.device)
    jetq_nvfp4_scale_atoms(sb, rows, k, atoms, stream)
    return atoms


def nvfp4_fprop(a, b, k, out_dtype=torch.float32, stream=None):
    """NVFP4 FProp of two quant_nvfp4 dicts (A: activations, B: weight), each with 'atoms' added."""
    m, n = a["q"].shape[0], b["q"].shape[0]
    y = torch.empty((m, n), dtype=out_dtype, device=a["q"].device)
    jetq_gemm_nvfp4(a["q"], a["atoms"], a["sg"], a["sg"].numel() > 1, b["q"], b["atoms"], b["sg"], m, n, k, y,
                    stream)
    return y


def quant_weight(w, transposed=True, stream=None):
    """BF16 [d x c] -> (q [d x c], s [d/128 x c/128], qT [c x d] | None, sT | None)."""
    d, c = w.shape
    dev = w.device
    q = torch.empty((d, c), dtype=torch.uint8, device=dev)
    s = torch.empty((d // 128, c // 128), dtype=torch.float32, device=dev)
    qT = torch.empty((c, d), dtype=torch.uint8, device=dev) if transposed else None
    sT = torch.empty((c // 128, d // 128), dtype=torch.float32, device=dev) if transposed else None
    jetq_quant_w_128x128(w, q, s, qT, sT, stream)
    return q, s, qT, sT


def quant_mx(x, row=True, col=True, seg_offsets=None, stream=None):
    """MXFP8 copies: dict(q_row, e8_row, q_col, e8_col, ldq_col); scales in the atom layout."""
    r, c = x.shape
    dev = x.device
    nseg = 0 if seg_offsets is None else seg_offsets.numel() - 1
    cap = jetq_colcopy_capacity(r, max(nseg, 1))
    out = dict(q_row=None, e8_row=None, q_col=None, e8_col=None, ldq_col=cap)
    if row:
        out["q_row"] = torch.empty((r, c), dtype=torch.uint8, device=dev)
        out["e8_row"] = torch.zeros(jetq_mx_scale_bytes(r, c), dtype=torch.uint8, device=dev)
    if col:
        out["q_col"] = torch.empty((c, cap), dtype=torch.uint8, device=dev)
        out["e8_col"] = torch.zeros(jetq_mx_scale_bytes(c, cap), dtype=torch.uint8, device=dev)
    jetq_quant_mx32(x, out["q_row"], out["e8_row"], out["q_col"], out["e8_col"], cap, seg_offsets, nseg, stream)
    return out


def quant_act_pow2(x, row=True, col=True, seg_offsets=None, stream=None):
    """Power-of-two 1x128 / 128x1 copies: dict(q_row, e8_row, q_col, e8_col, ldq_col), MX atom layout."""
    r, c = x.shape
    dev = x.device
    nseg = 0 if seg_offsets is None else seg_offsets.numel() - 1
    cap = jetq_colcopy_capacity(r, max(nseg, 1))
    out = dict(q_row=None, e8_row=None, q_col=None, e8_col=None, ldq_col=cap)
    if row:
        out["q_row"] = torch.empty((r, c), dtype=torch.uint8, device=dev)
        out["e8_row"] = torch.zeros(jetq_mx_scale_bytes(r, c), dtype=torch.uint8, device=dev)
    if col:
        out["q_col"] = torch.empty((c, cap), dtype=torch.uint8, device=dev)
        out["e8_col"] = torch.zeros(jetq_mx_scale_bytes(c, cap), dtype=torch.uint8, device=dev)
    jetq_quant_act_1x128_pow2(x, out["q_row"], out["e8_row"], out["q_col"], out["e8_col"], cap, seg_offsets, nseg,
                              stream)
    return out


def quant_weight_pow2(w, transposed=True, stream=None):
    """Power-of-two 128x128 blocks: (q [d x c], e8 atoms (d, c), qT [c x d] | None, e8T atoms (c, d) | None)."""
    d, c = w.shape
    dev = w.device
    q = torch.empty((d, c), dtype=torch.uint8, device=dev)
    e8 = torch.zeros(jetq_mx_scale_bytes(d, c), dtype=torch.uint8, device=dev)
    qT = torch.empty((c, d), dtype=torch.uint8, device=dev) if transposed else None
    e8T = torch.zeros(jetq_mx_scale_bytes(c, d), dtype=torch.uint8, device=dev) if transposed else None
    jetq_quant_w_128x128_pow2(w, q, e8, qT, e8T, stream)
    return q, e8, qT, e8T


def fprop(qx, sx, qw, sw, out_dtype=torch.float32, path=PATH_AUTO, recipe=RECIPE_BLOCK128, stream=None,
          workspace=None):
    """Y = X W^T.  Rollout-sized calls that can spread a weight band over several
    SMs get a workspace (the caller's, if large enough, else a fresh one)."""
    n, c = qx.shape
    d = qw.shape[0]
    y = torch.empty((n, d), dtype=out_dtype, device=qx.device)
    wsb = jetq_decode_workspace_bytes(n, d, c) if recipe == RECIPE_BLOCK128 and path != PATH_TRAIN else 0
    if wsb:
        if workspace is None or workspace.numel() * workspace.element_size() < wsb:
            workspace = torch.empty(wsb, dtype=torch.uint8, device=qx.device)
        jetq_gemm_fprop_ws(recipe, qx, sx, qw, sw, n, d, c, y, workspace, path, stream)
    else:
        jetq_gemm_fprop(recipe, qx, sx, qw, sw, n, d, c, y, path, stream)
    return y


def dgrad(qdy, sdy, qwt, swt, out_dtype=torch.float32, recipe=RECIPE_BLOCK128, stream=None):
    n, d = qdy.shape
    c = qwt.shape[0]
    dx = torch.empty((n, c), dtype=out_dtype, device=qdy.device)
    jetq_gemm_dgrad(recipe, qdy, sdy, qwt, swt, n, d, c, dx, stream)
    return dx


def wgrad(qdyc, sdyc, qxc, sxc, k, dw=None, accumulate=False, recipe=RECIPE_BLOCK128, stream=None):
    d, ldk = qdyc.shape
    c = qxc.shape[0]
    if dw is None:
        dw = torch.empty((d, c), dtype=torch.float32, device=qdyc.device)
    jetq_gemm_wgrad(recipe, qdyc, sdyc, qxc, sxc, k, ldk, d, c, dw, accumulate, stream)
    return dw


def grouped(kind, a, sa, b, sb, seg_offsets, n, k, out_dtype=torch.float32, recipe=RECIPE_BLOCK128, out=None,
            accumulate=False, stream=None):
    """Per-expert GEMMs over routed rows (see jetq_gemm_grouped).

    FPROP/DGRAD: a [m x k] routed row copy, b stacked [E*n x k] (or [E, n, k]); returns [m x n].
    WGRAD: a, b column copies [m x ldk], [n x ldk]; k = column-copy length; returns [E x m x n] FP32.
    """
    E = seg_offsets.numel() - 1
    m, ldk = a.shape[0], a.shape[1]
    if out is None:
        if kind == GEMM_WGRAD:
            out = torch.empty((E, m, n), dtype=torch.float32, device=a.device)
        else:
            out = torch.empty((m, n), dtype=out_dtype, device=a.device)
    jetq_gemm_grouped(kind, recipe, a, sa, b, sb, m, n, k, ldk, seg_offsets, E, out, accumulate, stream)
    return out

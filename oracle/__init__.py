"""The jetq oracle: a plain CPU statement of the FP8 quantize-and-GEMM path.

TEST INFRASTRUCTURE ONLY.  The product library never imports this package.
Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it, to check and time the CUDA path.  It shares no code with
the CUDA path; its arithmetic lives in ``jetq_oracle.c`` (plain C99), and this
module only marshals numpy arrays into it.

What each function computes, and which page passage it follows, is stated in
``jetq_oracle.c``.  Conventions: BF16 tensors are ``numpy.uint16`` bit
patterns; codes are ``numpy.uint8``; FP32 scales are ``numpy.float32``;
dequantized tensors and GEMM results are ``numpy.float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jetq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libjetq_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libjetq_oracle.so`` with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.jo_e4m3_decode.restype = ctypes.c_double
        lib.jo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.jo_e4m3_encode.restype = ctypes.c_uint8
        lib.jo_e4m3_encode.argtypes = [ctypes.c_double]
        lib.jo_e8m0_exponent.restype = ctypes.c_int
        lib.jo_e8m0_exponent.argtypes = [ctypes.c_float]
        lib.jo_colcopy_length.restype = I
        lib.jo_colcopy_length.argtypes = [P, ctypes.c_int, I]
        lib.jo_quant_rowgroups.argtypes = [P, I, I, I, I, P, I, P]
        lib.jo_quant_colgroups.argtypes = [P, I, I, I, I, P, ctypes.c_int, P, I, P]
        lib.jo_quant_blocks.argtypes = [P, I, I, I, I, P, P, P, P]
        lib.jo_quant_blocks_pow2.argtypes = [P, I, I, I, I, P, P, P, P]
        lib.jo_expf_fixed.restype = ctypes.c_float
        lib.jo_expf_fixed.argtypes = [ctypes.c_float]
        lib.jo_swiglu_bf16.argtypes = [P, P, I, P]
        lib.jo_rmsnorm_bf16.argtypes = [P, P, I, I, I, ctypes.c_float, P, P]
        lib.jo_requant_colgroups.argtypes = [P, P, I, I, I, P, ctypes.c_int, P, I, P]
        lib.jo_dequant_rowgroups_bf16.argtypes = [P, I, I, I, P, P]
        lib.jo_dequant_blocks_bf16.argtypes = [P, I, I, I, P, P]
        lib.jo_quant_mx_rows.argtypes = [P, I, I, I, I, P, I, P]
        lib.jo_quant_mx_cols.argtypes = [P, I, I, I, I, I, P, ctypes.c_int, P, I, P]
        lib.jo_dequant_rowgroups.argtypes = [P, I, I, I, I, P, P]
        lib.jo_dequant_colgroups.argtypes = [P, I, P, I, I, I, P, ctypes.c_int, P]
        lib.jo_dequant_blocks.argtypes = [P, I, I, I, P, P]
        lib.jo_dequant_blocks_pow2.argtypes = [P, I, I, I, P, P]
        lib.jo_dequant_mx_rows.argtypes = [P, I, I, I, I, P, P]
        lib.jo_dequant_mx_cols.argtypes = [P, I, P, I, I, I, I, I, P, ctypes.c_int, P]
        lib.jo_e2m1_decode.restype = ctypes.c_double
        lib.jo_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.jo_e2m1_encode.restype = ctypes.c_uint8
        lib.jo_e2m1_encode.argtypes = [ctypes.c_double]
        lib.jo_quant_nvfp4.argtypes = [P, I, I, I, P, P, P, P]
        lib.jo_quant_nvfp4.restype = None
        lib.jo_dequant_nvfp4_bf16.argtypes = [P, P, P, I, I, ctypes.c_int, P]
        lib.jo_dequant_nvfp4_bf16.restype = None
        lib.jo_dequant_nvfp4.argtypes = [P, P, P, I, I, ctypes.c_int, P]
        lib.jo_dequant_nvfp4.restype = None
        for f in ("jo_fprop", "jo_dgrad", "jo_wgrad"):
            getattr(lib, f).argtypes = [P, P, I, I, I, P, I, P, P]
        for f in ("jo_quant_rowgroups", "jo_quant_colgroups", "jo_quant_blocks", "jo_quant_mx_rows",
                  "jo_quant_mx_cols", "jo_dequant_rowgroups", "jo_dequant_colgroups",
                  "jo_dequant_blocks", "jo_dequant_mx_rows", "jo_dequant_mx_cols",
                  "jo_fprop", "jo_dgrad", "jo_wgrad"):
            getattr(lib, f).restype = None
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _offsets(offsets, rows):
    if offsets is None:
        return np.array([0, rows], dtype=np.int64)
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    if off[0] != 0 or off[-1] != rows or np.any(np.diff(off) < 0):
        raise ValueError("segment offsets must rise from 0 to the row count")
    return off


# --------------------------------------------------------------------------- codec

def e4m3_decode(codes) -> np.ndarray:
    """Value of every E4M3 code (NaN for 0x7F / 0xFF)."""
    lib = _load()
    table = np.array([lib.jo_e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(values) -> np.ndarray:
    """Round each value to the nearest E4M3 code (ties to even, saturating)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.array([lib.jo_e4m3_encode(float(x)) for x in v.ravel()], dtype=np.uint8).reshape(v.shape)


def e2m1_decode(codes) -> np.ndarray:
    """Value of every E2M1 code (4 bits: sign, 2 exponent bits, 1 mantissa bit)."""
    lib = _load()
    table = np.array([lib.jo_e2m1_decode(c) for c in range(16)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8) & 15]


def e2m1_encode(values) -> np.ndarray:
    """Round each value to the nearest E2M1 code (ties to even, saturating at 6)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.array([lib.jo_e2m1_encode(float(x)) for x in v.ravel()], dtype=np.uint8).reshape(v.shape)


def e8m0_exponent(amax: float) -> int:
    """Smallest e with amax <= 448 * 2**e, clamped to [-127, 127] (0 for amax 0)."""
    return int(_load().jo_e8m0_exponent(ctypes.c_float(amax)))


def colcopy_length(offsets, rows: int, gs: int = 128) -> int:
    """Length P of a column copy whose segments each start on a multiple of gs."""
    off = _offsets(offsets, rows)
    return int(_load().jo_colcopy_length(_p(off), len(off) - 1, gs))


# ----------------------------------------------------------------------- quantizers

def quant_rowgroups(x, gs: int = 128):
    """1 x gs groups along each row: returns (q [R x C] u8, s [C/gs x R] f32)."""
    x = _c(x, np.uint16)
    R, C = x.shape
    if C % gs:
        raise ValueError("columns must be a multiple of the group size")
    q = np.empty((R, C), np.uint8)
    s = np.empty((C // gs, R), np.float32)
    _load().jo_quant_rowgroups(_p(x), R, C, C, gs, _p(q), C, _p(s))
    return q, s


def quant_colgroups(x, gs: int = 128, offsets=None):
    """gs x 1 groups down each column inside each segment, stored transposed.

    Returns (qc [C x P] u8, sc [P/gs x C] f32) where P = colcopy_length.
    """
    x = _c(x, np.uint16)
    R, C = x.shape
    off = _offsets(offsets, R)
    P = colcopy_length(off, R, gs)
    qc = np.zeros((C, P), np.uint8)
    sc = np.zeros((P // gs, C), np.float32)
    _load().jo_quant_colgroups(_p(x), R, C, C, gs, _p(off), len(off) - 1, _p(qc), P, _p(sc))
    return qc, sc


def quant_blocks(w, bs: int = 128):
    """bs x bs blocks: returns (q [D x C], s [D/bs x C/bs], qT [C x D], sT [C/bs x D/bs])."""
    w = _c(w, np.uint16)
    D, C = w.shape
    if D % bs or C % bs:
        raise ValueError("both dimensions must be multiples of the block size")
    q = np.empty((D, C), np.uint8)
    s = np.empty((D // bs, C // bs), np.float32)
    qT = np.empty((C, D), np.uint8)
    sT = np.empty((C // bs, D // bs), np.float32)
    _load().jo_quant_blocks(_p(w), D, C, C, bs, _p(q), _p(s), _p(qT), _p(sT))
    return q, s, qT, sT


def requant_colgroups(q_row, s_row, offsets=None, gs: int = 128):
    """Column copy re-quantized from a row copy (q_row [R x C], s_row [C/gs x R]):
    v = fl32(decode(q) * S_row), then gs x 1 groups as quant_colgroups.
    Returns (qc [C x P], sc [P/gs x C])."""
    q_row = _c(q_row, np.uint8)
    s_row = _c(s_row, np.float32)
    R, C = q_row.shape
    off = _offsets(offsets, R)
    P = colcopy_length(off, R, gs)
    qc = np.zeros((C, P), np.uint8)
    sc = np.zeros((P // gs, C), np.float32)
    _load().jo_requant_colgroups(_p(q_row), _p(s_row), R, C, gs, _p(off), len(off) - 1, _p(qc), P, _p(sc))
    return qc, sc


def dequant_rowgroups_bf16(q, s, gs: int = 128):
    """BF16 bit patterns of decode(q) * S for a row copy (q [R x C], s [C/gs x R]), rounded once."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    R, C = q.shape
    out = np.empty((R, C), np.uint16)
    _load().jo_dequant_rowgroups_bf16(_p(q), R, C, gs, _p(s), _p(out))
    return out


def dequant_blocks_bf16(q, s, bs: int = 128):
    """BF16 bit patterns of decode(q) * S for bs x bs blocks (s [D/bs x C/bs]), rounded once."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    D, C = q.shape
    out = np.empty((D, C), np.uint16)
    _load().jo_dequant_blocks_bf16(_p(q), D, C, bs, _p(s), _p(out))
    return out


def expf_fixed(x: float) -> float:
    """The binary32 exp of the fused SwiGLU producer (Cody-Waite + Taylor, fmaf)."""
    return float(_load().jo_expf_fixed(ctypes.c_float(x)))


def swiglu_bf16(gate, up):
    """BF16 bits of silu(gate) * up, operation by operation in binary32."""
    gate = _c(gate, np.uint16)
    up = _c(up, np.uint16)
    if gate.shape != up.shape:
        raise ValueError("gate and up must have the same shape")
    h = np.empty(gate.shape, np.uint16)
    _load().jo_swiglu_bf16(_p(gate), _p(up), gate.size, _p(h))
    return h


def rmsnorm_bf16(x, w, eps: float = 1e-6):
    """BF16 bits of RMSNorm(x) * w and the per-row rstd (fixed binary32 summation order)."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    R, C = x.shape
    if C % 128 or w.shape != (C,):
        raise ValueError("columns must be a multiple of 128 and w must have one entry per column")
    y = np.empty((R, C), np.uint16)
    rstd = np.empty(R, np.float32)
    _load().jo_rmsnorm_bf16(_p(x), _p(w), R, C, C, ctypes.c_float(eps), _p(y), _p(rstd))
    return y, rstd


def quant_blocks_pow2(w, bs: int = 128):
    """Power-of-two bs x bs blocks: returns (q [D x C], e8 [D/bs x C/bs], qT [C x D], e8T [C/bs x D/bs]);
    e8 holds the E8M0 byte e + 127 of each block's scale 2^e."""
    w = _c(w, np.uint16)
    D, C = w.shape
    if D % bs or C % bs:
        raise ValueError("both dimensions must be multiples of the block size")
    q = np.empty((D, C), np.uint8)
    e8 = np.empty((D // bs, C // bs), np.uint8)
    qT = np.empty((C, D), np.uint8)
    e8T = np.empty((C // bs, D // bs), np.uint8)
    _load().jo_quant_blocks_pow2(_p(w), D, C, C, bs, _p(q), _p(e8), _p(qT), _p(e8T))
    return q, e8, qT, e8T


def quant_mx_rows(x, bs: int = 32):
    """MX 1 x bs blocks along each row: returns (q [R x C] u8, e8 [R x C/bs] u8)."""
    x = _c(x, np.uint16)
    R, C = x.shape
    if C % bs:
        raise ValueError("columns must be a multiple of the block size")
    q = np.empty((R, C), np.uint8)
    e8 = np.empty((R, C // bs), np.uint8)
    _load().jo_quant_mx_rows(_p(x), R, C, C, bs, _p(q), C, _p(e8))
    return q, e8


def quant_mx_cols(x, bs: int = 32, offsets=None, seg_align: int = 128):
    """MX bs x 1 blocks down each column inside each segment, stored transposed.

    Segments start on multiples of seg_align.  Returns (qc [C x P], e8 [C x P/bs]).
    """
    x = _c(x, np.uint16)
    R, C = x.shape
    off = _offsets(offsets, R)
    P = colcopy_length(off, R, seg_align)
    qc = np.zeros((C, P), np.uint8)
    e8 = np.zeros((C, P // bs), np.uint8)
    _load().jo_quant_mx_cols(_p(x), R, C, C, bs, seg_align, _p(off), len(off) - 1, _p(qc), P, _p(e8))
    return qc, e8


# ---------------------------------------------------------------------- dequantizers

def dequant_rowgroups(q, s, gs: int = 128):
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    R, C = q.shape
    out = np.empty((R, C), np.float64)
    _load().jo_dequant_rowgroups(_p(q), R, C, C, gs, _p(s), _p(out))
    return out


def dequant_colgroups(qc, sc, rows: int, gs: int = 128, offsets=None):
    """Back to the natural [rows x C] layout."""
    qc = _c(qc, np.uint8)
    sc = _c(sc, np.float32)
    C, P = qc.shape
    off = _offsets(offsets, rows)
    out = np.zeros((rows, C), np.float64)
    _load().jo_dequant_colgroups(_p(qc), P, _p(sc), rows, C, gs, _p(off), len(off) - 1, _p(out))
    return out


def dequant_blocks(q, s, bs: int = 128):
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    D, C = q.shape
    out = np.empty((D, C), np.float64)
    _load().jo_dequant_blocks(_p(q), D, C, bs, _p(s), _p(out))
    return out


def dequant_blocks_pow2(q, e8, bs: int = 128):
    q = _c(q, np.uint8)
    e8 = _c(e8, np.uint8)
    D, C = q.shape
    out = np.empty((D, C), np.float64)
    _load().jo_dequant_blocks_pow2(_p(q), D, C, bs, _p(e8), _p(out))
    return out


def dequant_mx_rows(q, e8, bs: int = 32):
    q = _c(q, np.uint8)
    e8 = _c(e8, np.uint8)
    R, C = q.shape
    out = np.empty((R, C), np.float64)
    _load().jo_dequant_mx_rows(_p(q), R, C, C, bs, _p(e8), _p(out))
    return out


def dequant_mx_cols(qc, e8, rows: int, bs: int = 32, offsets=None, seg_align: int = 128):
    qc = _c(qc, np.uint8)
    e8 = _c(e8, np.uint8)
    C, P = qc.shape
    off = _offsets(offsets, rows)
    out = np.zeros((rows, C), np.float64)
    _load().jo_dequant_mx_cols(_p(qc), P, _p(e8), P, rows, C, bs, seg_align, _p(off), len(off) - 1,
                               _p(out))
    return out


# ---------------------------------------------------------------------------- GEMMs

def _gemm(name, A, B, N, D, C, at, out_shape):
    A = _c(A, np.float64)
    B = _c(B, np.float64)
    if at is None:
        y = np.empty(out_shape, np.float64)
        b = np.empty(out_shape, np.float64)
        getattr(_load(), name)(_p(A), _p(B), N, D, C, None, 0, _p(y), _p(b))
        return y, b
    at = np.ascontiguousarray(np.asarray(at, dtype=np.int64).reshape(-1, 2))
    y = np.empty(len(at), np.float64)
    b = np.empty(len(at), np.float64)
    getattr(_load(), name)(_p(A), _p(B), N, D, C, _p(at), len(at), _p(y), _p(b))
    return y, b


def fprop(X, W, at=None):
    """Y = X W^T on dequantized X [N x C], W [D x C]; returns (Y, sum|terms|)."""
    N, C = X.shape
    D = W.shape[0]
    assert W.shape[1] == C
    return _gemm("jo_fprop", X, W, N, D, C, at, (N, D))


def dgrad(dY, W, at=None):
    """dX = dY W on dequantized dY [N x D], W [D x C]; returns (dX, sum|terms|)."""
    N, D = dY.shape
    C = W.shape[1]
    assert W.shape[0] == D
    return _gemm("jo_dgrad", dY, W, N, D, C, at, (N, C))


def wgrad(dY, X, at=None):
    """dW = dY^T X on dequantized dY [N x D], X [N x C]; returns (dW, sum|terms|)."""
    N, D = dY.shape
    C = X.shape[1]
    assert X.shape[0] == N
    return _gemm("jo_wgrad", dY, X, N, D, C, at, (D, C))


# --------------------------------------------------------------------------- NVFP4

def quant_nvfp4(x, scope_amax=None):
    """NVFP4: (q [R x C/2] u8 packed E2M1, sb [R x C/16] u8 E4M3 block scales,
    sg f32 scope scales: [R] per row when scope_amax is None, else [1] from the
    given tensor-scope max |x|)."""
    x = _c(x, np.uint16)
    R, C = x.shape
    if C % 16:
        raise ValueError("columns must be a multiple of 16")
    q = np.empty((R, C // 2), np.uint8)
    sb = np.empty((R, C // 16), np.uint8)
    sg = np.empty(R if scope_amax is None else 1, np.float32)
    amax = None if scope_amax is None else np.array([scope_amax], np.float32)
    _load().jo_quant_nvfp4(_p(x), R, C, C, _p(amax), _p(q), _p(sb), _p(sg))
    return q, sb, sg


def dequant_nvfp4_bf16(q, sb, sg):
    """BF16 bits of e2m1 * decode(e_b) * S_g, rounded once; per-row scales when sg has R entries."""
    q = _c(q, np.uint8)
    sb = _c(sb, np.uint8)
    sg = _c(sg, np.float32)
    R, C = q.shape[0], q.shape[1] * 2
    out = np.empty((R, C), np.uint16)
    _load().jo_dequant_nvfp4_bf16(_p(q), _p(sb), _p(sg), R, C, int(sg.size > 1), _p(out))
    return out


def dequant_nvfp4(q, sb, sg) -> np.ndarray:
    """Exact binary64 values e2m1 * decode(e_b) * S_g (per-row scales when sg has one entry per row)."""
    q = _c(q, np.uint8)
    sb = _c(sb, np.uint8)
    sg = _c(sg, np.float32)
    R, C = q.shape[0], q.shape[1] * 2
    out = np.empty((R, C), np.float64)
    _load().jo_dequant_nvfp4(_p(q), _p(sb), _p(sg), R, C, int(sg.size > 1), _p(out))
    return out

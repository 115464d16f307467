"""Helpers shared by the GPU parity tests (test code only)."""
import numpy as np
import torch

DEV = "cuda:0"


def to_dev_bf16(h: np.ndarray) -> torch.Tensor:
    """uint16 BF16 bit patterns -> a bfloat16 tensor on the GPU (same bytes)."""
    return torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).to(DEV).view(torch.bfloat16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def f32bits(t) -> np.ndarray:
    a = t.cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def mx_atom_offsets(R: int, J: int) -> np.ndarray:
    """Byte offset of logical MX scale (r, j) in the documented 512-byte atom layout."""
    rb = (R + 127) // 128
    r = np.arange(R)[:, None]
    j = np.arange(J)[None, :]
    return ((j // 4) * rb + r // 128) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4


def mx_atoms(e8_logical: np.ndarray, k: int) -> np.ndarray:
    """Places logical MX scale bytes [R x K/32] into the atom layout for a K-column payload."""
    R, J = e8_logical.shape
    out = np.zeros(((R + 127) // 128) * (k // 128) * 512, np.uint8)
    out[mx_atom_offsets(R, J)] = e8_logical
    return out


def assert_gemm_close(got: torch.Tensor, ref: np.ndarray, bound: np.ndarray, rel: float = 1e-5):
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    ok = err <= rel * bound
    if not np.all(ok):
        idx = np.argwhere(~ok)[:5]
        worst = float(np.max(err / np.maximum(bound, 1e-300)))
        raise AssertionError(f"{(~ok).sum()} outputs outside {rel}*sum|ab|; worst ratio {worst:.3g}; "
                             f"first {idx.tolist()} got {g[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")

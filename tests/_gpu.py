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


def mx_atoms(e8_logical: np.ndarray, k: int) -> np.ndarray:
    """Places logical MX scale bytes [R x K/32] into the documented 2048-byte atom layout."""
    R, J = e8_logical.shape
    ka = (k + 511) // 512
    out = np.zeros(((R + 127) // 128) * ka * 2048, np.uint8)
    r = np.arange(R)[:, None]
    j = np.arange(J)[None, :]
    off = ((r // 128) * ka + j // 16) * 2048 + (r % 128) * 16 + j % 16
    out[off] = e8_logical
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

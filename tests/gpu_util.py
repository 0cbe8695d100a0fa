"""Helpers for the GPU parity tests: host <-> device conversions and the documented scale layout.

Nothing here computes the method: it only moves bits between numpy (the oracle's side) and
torch device tensors (the library's side), and applies the byte permutation that
include/adahop.h documents for scale_layout = 1.
"""
import numpy as np
import torch

from synthetic import bf16_bits


def dev_bf16_from_bits(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return bf16_bits(t)


def tiled_scale_permutation(lines, J: int) -> np.ndarray:
    """offset[l, b] of scale (line l, block b) in the tensor-core layout (include/adahop.h), for
    lines 0 .. lines - 1 (an int) or for the given line numbers (an array)."""
    ids = np.arange(lines) if np.isscalar(lines) else np.asarray(lines)
    l = ids.astype(np.int64)[:, None]
    b = np.arange(J // 32, dtype=np.int64)[None, :]
    return ((l >> 7) * (J >> 7) + (b >> 2)) * 512 + (l & 31) * 16 + ((l >> 5) & 3) * 4 + (b & 3)


def to_tiled(scales: np.ndarray) -> np.ndarray:
    lines, nb = scales.shape
    out = np.zeros(lines * nb, dtype=np.uint8)
    out[tiled_scale_permutation(lines, nb * 32).ravel()] = scales.ravel()
    return out


def from_tiled(flat: np.ndarray, lines, J: int) -> np.ndarray:
    """The scales of lines 0 .. lines - 1 (an int) or of the given line numbers (an array)."""
    return np.asarray(flat)[tiled_scale_permutation(lines, J)]


def bitmap(lines: int, idx) -> np.ndarray:
    words = np.zeros((lines + 31) // 32, dtype=np.uint32)
    for i in np.asarray(idx, dtype=np.int64):
        words[i >> 5] |= np.uint32(1) << np.uint32(i & 31)
    return words


_SIGNED = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32, np.dtype(np.uint64): np.int64}


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Upload a numpy array bit for bit (unsigned 16/32/64-bit arrays travel as signed views)."""
    a = np.ascontiguousarray(a)
    if a.dtype in _SIGNED:
        a = a.view(_SIGNED[a.dtype])
    return torch.from_numpy(a).to(device)


def to_host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint8)

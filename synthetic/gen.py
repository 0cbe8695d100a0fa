"""Seeded tensor draws.

Recipe (the same on every machine for a given device kind):
  * base values: ``torch.randn`` (float32) from a ``torch.Generator`` on the target device,
    seeded with ``seed``, times ``std``;
  * outlier lines: the first ``count`` entries of ``torch.randperm(dim)`` drawn from a CPU
    generator seeded with ``seed + 7919`` (so the choice does not depend on the device), sorted;
    those whole rows (or columns) are multiplied by ``scale``;
  * the float32 tensor is rounded to bfloat16 by PyTorch's round-to-nearest-even cast.

CPU and CUDA generators give different streams; tests that compare the two paths always hand
the very same bf16 tensor to both sides.
"""
from __future__ import annotations

import numpy as np
import torch

_OUTLIER_SEED_OFFSET = 7919


def outlier_lines(dim: int, count: int, seed: int) -> torch.Tensor:
    """Sorted indices of ``count`` distinct lines out of ``dim`` (int64, CPU)."""
    if count <= 0:
        return torch.empty(0, dtype=torch.long)
    if count > dim:
        raise ValueError(f"cannot pick {count} outlier lines out of {dim}")
    g = torch.Generator(device="cpu").manual_seed(seed + _OUTLIER_SEED_OFFSET)
    return torch.randperm(dim, generator=g)[:count].sort().values


def normal_bf16(rows: int, cols: int, std: float, seed: int, *, outlier_axis: str | None = None,
                outlier_count: int = 0, outlier_scale: float = 1.0,
                device: str | torch.device = "cpu") -> torch.Tensor:
    """A ``rows x cols`` row-major bf16 tensor ~ N(0, std^2) with optional scaled lines.

    ``outlier_axis`` is ``"row"`` (whole rows scaled: a Row-wise tensor), ``"col"`` (whole
    columns scaled: Column-wise) or ``None``.
    """
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn((rows, cols), generator=g, dtype=torch.float32, device=device)
    x.mul_(std)
    if outlier_axis is not None and outlier_count > 0:
        if outlier_axis == "row":
            idx = outlier_lines(rows, outlier_count, seed).to(device)
            x[idx, :] *= outlier_scale
        elif outlier_axis == "col":
            idx = outlier_lines(cols, outlier_count, seed).to(device)
            x[:, idx] *= outlier_scale
        else:
            raise ValueError(f"outlier_axis must be 'row', 'col' or None, not {outlier_axis!r}")
    return x.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of ``t`` as a host uint16 array of the same shape."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)

"""Workload shapes and tensor recipes for the synthetic stand-ins of the pages' models.

The AdaHOP pages train Llama3.2-1B, Instella-3B and Llama3.1-8B on C4 (AdaHOP paper, Table 1,
Table 3).  Neither the dataset nor trained tensors are available, so every linear layer is fed
seeded Gaussian tensors with planted outlier lines that give each operand the pattern the pages
report for it (weights None, activations Column-wise, gradients Row-wise or None; Table 1 caption,
Fig. 8 caption).

Shapes: W is N x K (out x in features), X is M x K, G_Y is M x N, M = sequence x batch.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from .gen import normal_bf16


@dataclass(frozen=True)
class TensorRecipe:
    std: float
    outlier_axis: str | None = None   # "row", "col" or None
    outlier_count: int = 0
    outlier_scale: float = 1.0

    def draw(self, rows: int, cols: int, seed: int, device="cpu") -> torch.Tensor:
        return normal_bf16(rows, cols, self.std, seed, outlier_axis=self.outlier_axis,
                           outlier_count=self.outlier_count, outlier_scale=self.outlier_scale,
                           device=device)


W_RECIPE = TensorRecipe(std=0.02)


@dataclass(frozen=True)
class Linear:
    name: str
    N: int                 # out features
    K: int                 # in features
    x: TensorRecipe
    gy: TensorRecipe | None
    w: TensorRecipe = W_RECIPE


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    linears: tuple
    description: str
    seed: int = 0
    fwd_only: bool = False
    extra: dict = field(default_factory=dict)

    def flops_fwd_bwd(self) -> int:
        """6*M*N*K summed over the linears (Fwd + dX + dW)."""
        return sum(6 * self.M * lin.N * lin.K for lin in self.linears)


def tensor_recipes(wl: Workload, li: int, device="cpu"):
    """Draw (X, W, G_Y) for linear ``li`` of workload ``wl`` (G_Y is None for fwd-only)."""
    lin = wl.linears[li]
    base = wl.seed * 1000 + li * 3
    X = lin.x.draw(wl.M, lin.K, base + 0, device)
    W = lin.w.draw(lin.N, lin.K, base + 1, device)
    GY = lin.gy.draw(wl.M, lin.N, base + 2, device) if lin.gy is not None else None
    return X, W, GY


def _block(prefix, hidden, kv, ffn, x, gy):
    return (
        Linear(f"{prefix}q", hidden, hidden, x, gy),
        Linear(f"{prefix}k", kv, hidden, x, gy),
        Linear(f"{prefix}v", kv, hidden, x, gy),
        Linear(f"{prefix}o", hidden, hidden, x, gy),
        Linear(f"{prefix}gate", ffn, hidden, x, gy),
        Linear(f"{prefix}up", ffn, hidden, x, gy),
        Linear(f"{prefix}down", hidden, ffn, x, gy),
    )


_X1B = TensorRecipe(1.0, "col", 16, 30.0)
_G1B = TensorRecipe(1e-3, "row", 32, 40.0)
_X3B_C = TensorRecipe(1.0, "col", 24, 50.0)
_X3B_N = TensorRecipe(1.0)
_G3B_R = TensorRecipe(1e-3, "row", 32, 40.0)
_G3B_N = TensorRecipe(1e-3)
_X8B = TensorRecipe(1.0, "col", 32, 50.0)
_G8B = TensorRecipe(1e-3, "row", 64, 40.0)

WORKLOADS = {
    # 256 x 256 x 512 forward GEMM, CN pair (X Column-wise, W None).
    "tiny": Workload(
        "tiny", 256,
        (Linear("fc", 256, 512, TensorRecipe(1.0, "col", 8, 50.0), None),),
        "X 256x512 ~N(0,1), 8 columns x50; W 256x512 ~N(0,0.02); Y = X.W^T",
        fwd_only=True),
    # Llama3.2-1B-shaped block: seq 2048 x batch 2, hidden 2048, 8 KV heads x 64, FFN 8192.
    "llama3.2-1b": Workload(
        "llama3.2-1b", 4096, _block("", 2048, 512, 8192, _X1B, _G1B),
        "M=4096; X 16 cols x30; W ~N(0,0.02); G_Y ~N(0,1e-3) 32 rows x40"),
    # Instella-3B-shaped block: seq 4096 x batch 2, hidden 3072 (k/v taken as full width), FFN 8192.
    # Four synthetic layers cover the pairs RN, RC, NN, NC and CN.
    "instella-3b": Workload(
        "instella-3b", 8192,
        _block("L0.", 3072, 3072, 8192, _X3B_C, _G3B_R)[:1]
        + _block("L1.", 3072, 3072, 8192, _X3B_C, _G3B_N)[4:5]
        + _block("L2.", 3072, 3072, 8192, _X3B_N, _G3B_R)[6:7]
        + _block("L3.", 3072, 3072, 8192, _X3B_N, _G3B_N)[3:4],
        "M=8192; X Column-wise (24 cols x50) or None; G_Y Row-wise (32 rows x40) or None"),
    # Llama3.1-8B-shaped block: seq 4096 x batch 8, hidden 4096, 8 KV heads x 128, FFN 14336.
    "llama3.1-8b": Workload(
        "llama3.1-8b", 32768, _block("", 4096, 1024, 14336, _X8B, _G8B),
        "M=32768; X 32 cols x50; W ~N(0,0.02); G_Y ~N(0,1e-3) 64 rows x40"),
}

# OE rank / batch sweep on the Llama3.1-8B down projection (K=14336, N=4096).
SWEEP_M = (4096, 8192, 16384, 32768, 65536)
SWEEP_RANKS = (0, 16, 32, 64, 128, 256)


def sweep_workload(M: int, rank: int, control: bool = False) -> Workload:
    """Down projection with ``rank`` Column-wise outlier columns x50 (or a None control)."""
    x = TensorRecipe(1.0) if (control or rank == 0) else TensorRecipe(1.0, "col", rank, 50.0)
    return Workload(f"sweep-M{M}-r{rank}{'-none' if control else ''}", M,
                    (Linear("down", 4096, 14336, x, None),),
                    "Llama3.1-8B down projection, forward OE-Right sweep", fwd_only=True,
                    extra={"rank": rank})

"""Saved context: adahop_linear_fwd_save writes X and W in the backward orientations and
adahop_linear_bwd_saved reads them (AdaHOP appendix, IHT and Quantization: the forward pass saves
the quantised operands for backpropagation).

The saved operands carry exactly the zero mask and Hadamard setting the backward GEMM would apply,
so every output must be bit-identical to the plain adahop_linear_fwd / adahop_linear_bwd calls.
The strategy / pattern grid routes the saved operands through both paths of the forward call:
the dual-orientation pass (forward and backward agree on mask and Hadamard) and the separate pass
(they differ: e.g. wgrad OE-Right zeroes X's outlier columns while the forward IHT does not).
"""
import numpy as np
import pytest
import torch

import oracle as O
from synthetic import normal_bf16

pytestmark = pytest.mark.gpu

S = (O.IHT, O.MXFP4_PLAIN, O.BF16, O.OE_LEFT, O.OE_RIGHT)
PATTERNS = {
    "CNR": (O.PAT_COL, O.PAT_NONE, O.PAT_ROW),
    "RCC": (O.PAT_ROW, O.PAT_COL, O.PAT_COL),
}
AXES = {O.PAT_ROW: "row", O.PAT_COL: "col", O.PAT_NONE: None}


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as lib
    return lib


def _tensors(M, N, K, pats, seed=11):
    px, pw, pg = pats
    X = normal_bf16(M, K, 1.0, seed, outlier_axis=AXES[px], outlier_count=12, outlier_scale=50.0)
    W = normal_bf16(N, K, 0.02, seed + 1, outlier_axis=AXES[pw], outlier_count=12, outlier_scale=50.0)
    GY = normal_bf16(M, N, 1e-3, seed + 2, outlier_axis=AXES[pg], outlier_count=16, outlier_scale=40.0)
    return X.cuda(), W.cuda(), GY.cuda()


def _nan(shape, dtype):
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


@pytest.mark.parametrize("pset", list(PATTERNS))
@pytest.mark.parametrize("fwd", S)
@pytest.mark.parametrize("dgrad,wgrad", [(O.OE_LEFT, O.OE_LEFT), (O.OE_RIGHT, O.OE_RIGHT), (O.IHT, O.MXFP4_PLAIN),
                                         (O.MXFP4_PLAIN, O.IHT), (O.BF16, O.OE_RIGHT), (O.OE_LEFT, O.BF16)])
def test_saved_context_bit_identical(q, pset, fwd, dgrad, wgrad):
    M, N, K, r = 256, 384, 512, 32
    pats = PATTERNS[pset]
    plan = q.make_plan(*pats, fwd, dgrad, wgrad, r)
    X, W, GY = _tensors(M, N, K, pats)
    ws = q.new_workspace(q.adahop_workspace_size(plan, M, N, K))
    dt = torch.bfloat16
    Y0, dX0, dW0 = _nan((M, N), dt), _nan((M, K), dt), _nan((N, K), dt)
    q.adahop_linear_fwd(plan, X, W, Y0, ws)
    q.adahop_linear_bwd(plan, GY, X, W, dX0, dW0, ws)
    saved = q.new_saved(plan, M, N, K)
    Y1, dX1, dW1 = _nan((M, N), dt), _nan((M, K), dt), _nan((N, K), dt)
    q.adahop_linear_fwd_save(plan, X, W, Y1, saved, ws)
    q.adahop_linear_bwd_saved(plan, GY, X, W, saved, dX1, dW1, ws)
    assert q.adahop_get_device_status(ws) == 0
    assert torch.equal(Y0, Y1)
    assert torch.equal(dX0, dX1)
    assert torch.equal(dW0, dW1)


def test_saved_context_fp32_and_single_output(q):
    M, N, K, r = 384, 256, 640, 16
    pats = PATTERNS["CNR"]
    plan = q.make_plan(*pats, O.IHT, O.OE_LEFT, O.OE_LEFT, r)
    X, W, GY = _tensors(M, N, K, pats, seed=5)
    ws = q.new_workspace(q.adahop_workspace_size(plan, M, N, K))
    saved = q.new_saved(plan, M, N, K)
    Y = _nan((M, N), torch.float32)
    q.adahop_linear_fwd_save(plan, X, W, Y, saved, ws)
    for which in ("dX", "dW"):
        ref = _nan((M, K) if which == "dX" else (N, K), torch.float32)
        got = _nan(ref.shape, torch.float32)
        args = (ref, None) if which == "dX" else (None, ref)
        q.adahop_linear_bwd(plan, GY, X, W, *args, ws)
        args = (got, None) if which == "dX" else (None, got)
        q.adahop_linear_bwd_saved(plan, GY, X, W, saved, *args, ws)
        assert torch.equal(ref, got)
    assert q.adahop_get_device_status(ws) == 0

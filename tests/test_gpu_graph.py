"""The linear calls inside a CUDA graph.

Every entry point is stream-ordered, allocates nothing and synchronises nothing (per-device
set-up happens on a device's first call), so a training step can capture a layer's forward and
backward calls once and replay them.  A replay must give bit for bit what the eager calls give,
including after the captured input buffers are refilled with new values.
"""
import pytest
import torch

import oracle as O
from synthetic import normal_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as lib
    return lib


def _draw(M, N, K, seed):
    X = normal_bf16(M, K, 1.0, seed, outlier_axis="col", outlier_count=12, outlier_scale=50.0)
    W = normal_bf16(N, K, 0.02, seed + 1)
    GY = normal_bf16(M, N, 1e-3, seed + 2, outlier_axis="row", outlier_count=16, outlier_scale=40.0)
    return X.cuda(), W.cuda(), GY.cuda()


@pytest.mark.parametrize("dgrad,wgrad", [(O.OE_LEFT, O.OE_LEFT), (O.IHT, O.IHT)])
def test_captured_step_replays_bit_identical(q, dgrad, wgrad):
    M, N, K = 512, 384, 640
    plan = q.make_plan(q.PAT_COL, q.PAT_NONE, q.PAT_ROW, q.IHT, dgrad, wgrad, 64)
    X, W, GY = _draw(M, N, K, 31)
    ws = q.new_workspace(q.adahop_workspace_size(plan, M, N, K))
    saved = q.new_saved(plan, M, N, K)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dX = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dW = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")

    def step():
        q.adahop_linear_fwd_save(plan, X, W, Y, saved, ws)
        q.adahop_linear_bwd_saved(plan, GY, X, W, saved, dX, dW, ws)

    def load(x, w, gy):
        X.copy_(x)
        W.copy_(w)
        GY.copy_(gy)

    def eager(x, w, gy):
        load(x, w, gy)
        step()
        torch.cuda.synchronize()
        assert q.adahop_get_device_status(ws) == 0
        return [t.clone() for t in (Y, dX, dW)]

    x0, w0, g0 = X.clone(), W.clone(), GY.clone()
    want0 = eager(x0, w0, g0)
    x1, w1, g1 = _draw(M, N, K, 47)
    want1 = eager(x1, w1, g1)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step()                                   # warm on the capture stream
        s.synchronize()
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.synchronize()
    for x, w, gy, want in ((x0, w0, g0, want0), (x1, w1, g1, want1)):
        load(x, w, gy)
        for t in (Y, dX, dW):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert q.adahop_get_device_status(ws) == 0
        for got, ref in zip((Y, dX, dW), want):
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16))

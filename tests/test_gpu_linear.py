"""End-to-end parity of adahop_linear_fwd / adahop_linear_bwd (C ABI) with the CPU oracle.

Every strategy (IHT, plain MXFP4, BF16, OE-Left, OE-Right) is run on each of the three GEMMs,
with operand patterns that put the extracted lines in each geometric role: inner (a rank-r
BF16 term inside the fused GEMM), outer rows and outer columns (BF16 outlier GEMM + scatter-add).
Tolerances: relative Frobenius 2e-3 (float32 output) / 4e-3 (bf16 output) against the oracle's
float64 product of the same quantised operands (Fig. 5 pipeline, appendix implementation notes).
Config-size cases compare sampled output rows (the oracle quantises the full B operand and the
sampled rows of A); the sampled rows always include extracted rows when OE is outer.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synthetic import WORKLOADS, bf16_bits, normal_bf16, tensor_recipes

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 2e-3, torch.bfloat16: 4e-3}
GEMM_ID = {"fwd": 0, "dgrad": 1, "wgrad": 2}


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as lib
    return lib


def _tensors(M, N, K, seed, x_axis="col", gy_axis="row", w_axis=None):
    X = normal_bf16(M, K, 1.0, seed, outlier_axis=x_axis, outlier_count=12, outlier_scale=50.0)
    W = normal_bf16(N, K, 0.02, seed + 1, outlier_axis=w_axis, outlier_count=12, outlier_scale=50.0)
    GY = normal_bf16(M, N, 1e-3, seed + 2, outlier_axis=gy_axis, outlier_count=16, outlier_scale=40.0)
    return X, W, GY


def _run(q, plan, X, W, GY, gemm, dtype):
    M, K = X.shape
    N = W.shape[0]
    ws = q.new_workspace(q.adahop_workspace_size(plan, M, N, K))
    dX_, dW_, dG_ = X.cuda(), W.cuda(), GY.cuda()
    if gemm == "fwd":
        out = torch.full((M, N), float("nan"), dtype=dtype, device="cuda")
        q.adahop_linear_fwd(plan, dX_, dW_, out, ws)
    elif gemm == "dgrad":
        out = torch.full((M, K), float("nan"), dtype=dtype, device="cuda")
        q.adahop_linear_bwd(plan, dG_, dX_, dW_, out, None, ws)
    else:
        out = torch.full((N, K), float("nan"), dtype=dtype, device="cuda")
        q.adahop_linear_bwd(plan, dG_, dX_, dW_, None, out, ws)
    assert q.adahop_get_device_status(ws) == 0
    return out.float().cpu().numpy().astype(np.float64)


# (x pattern, w pattern, gy pattern) choices that place OE in every role
PATTERN_SETS = {
    "CNR": (O.PAT_COL, O.PAT_NONE, O.PAT_ROW),   # fwd OE-R inner (X cols), dgrad OE-L outer rows,
                                                 # wgrad OE-L inner (G_Y rows), wgrad OE-R outer cols
    "RCC": (O.PAT_ROW, O.PAT_COL, O.PAT_COL),    # fwd OE-L outer rows (X rows), fwd OE-R inner (W cols),
                                                 # dgrad OE-R outer cols (W cols)
}


@pytest.mark.parametrize("gemm", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("strategy", [O.IHT, O.MXFP4_PLAIN, O.BF16, O.OE_LEFT, O.OE_RIGHT])
@pytest.mark.parametrize("pset", ["CNR", "RCC"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_linear_strategies_small(q, gemm, strategy, pset, dtype):
    M, N, K = 256, 384, 512
    px, pw, pg = PATTERN_SETS[pset]
    axes = {O.PAT_ROW: "row", O.PAT_COL: "col", O.PAT_NONE: None}
    X, W, GY = _tensors(M, N, K, 3, x_axis=axes[px], gy_axis=axes[pg], w_axis=axes[pw])
    r = 32
    strat = {"fwd": O.IHT, "dgrad": O.IHT, "wgrad": O.IHT}
    strat[gemm] = strategy
    plan = q.make_plan(px, pw, pg, strat["fwd"], strat["dgrad"], strat["wgrad"], r)
    got = _run(q, plan, X, W, GY, gemm, dtype)
    pats = {"X": px, "W": pw, "GY": pg}
    ref = O.gemm_oracle(gemm, strategy, bf16_bits(X), bf16_bits(W), bf16_bits(GY), patterns=pats, r=r)
    assert O.rel_frobenius(got, ref["C"]) <= TOL[dtype]
    if dtype == torch.float32:
        assert O.rel_frobenius(got, ref["C"]) <= 1e-5


@pytest.mark.parametrize("r", [0, 1, 8, 13, 50, 64, 256])
def test_linear_rank_edges(q, r):
    """r = 0 (plain IHT), one line, ranks that are not multiples of 8 or 64 (inner slices padded
    with zero columns), the default 64 and the maximum 256."""
    M, N, K = 512, 256, 384
    X, W, GY = _tensors(M, N, K, 9)
    plan = q.make_plan(O.PAT_COL, O.PAT_NONE, O.PAT_ROW, O.OE_RIGHT, O.OE_LEFT, O.OE_LEFT, r)
    pats = {"X": O.PAT_COL, "W": O.PAT_NONE, "GY": O.PAT_ROW}
    for gemm in ("fwd", "dgrad", "wgrad"):
        got = _run(q, plan, X, W, GY, gemm, torch.float32)
        strategy = {"fwd": O.OE_RIGHT, "dgrad": O.OE_LEFT, "wgrad": O.OE_LEFT}[gemm]
        ref = O.gemm_oracle(gemm, strategy, bf16_bits(X), bf16_bits(W), bf16_bits(GY), patterns=pats, r=r)
        assert O.rel_frobenius(got, ref["C"]) <= 1e-5, gemm


def test_linear_bwd_both_outputs_share_foid(q):
    """dX and dW in one call (FOID computed once for G_Y rows) match two separate calls."""
    M, N, K = 384, 256, 512
    X, W, GY = _tensors(M, N, K, 12)
    plan = q.make_plan(O.PAT_COL, O.PAT_NONE, O.PAT_ROW, O.IHT, O.OE_LEFT, O.OE_LEFT, 64)
    ws = q.new_workspace(q.adahop_workspace_size(plan, M, N, K))
    dX = torch.empty((M, K), dtype=torch.float32, device="cuda")
    dW = torch.empty((N, K), dtype=torch.float32, device="cuda")
    q.adahop_linear_bwd(plan, GY.cuda(), X.cuda(), W.cuda(), dX, dW, ws)
    assert q.adahop_get_device_status(ws) == 0
    np.testing.assert_array_equal(dX.cpu().numpy(), _run(q, plan, X, W, GY, "dgrad", torch.float32))
    np.testing.assert_array_equal(dW.cpu().numpy(), _run(q, plan, X, W, GY, "wgrad", torch.float32))


def test_tiny_config(q):
    """256 x 256 x 512 forward, CN pair: IHT, and the OE-Right variant with 16 columns."""
    X, W, _ = tensor_recipes(WORKLOADS["tiny"], 0)
    cal_ws = q.new_workspace(1 << 20)
    plan = q.adahop_calibrate(X.cuda(), W.cuda(), None, cal_ws)
    assert (plan.x, plan.w, plan.fwd) == (O.PAT_COL, O.PAT_NONE, O.IHT)
    pats = {"X": O.PAT_COL, "W": O.PAT_NONE, "GY": O.PAT_NONE}
    GY = torch.zeros((256, 256), dtype=torch.bfloat16)
    for strategy, r in ((O.IHT, 0), (O.OE_RIGHT, 16)):
        plan.fwd, plan.oe_rank = strategy, r
        for dtype in (torch.float32, torch.bfloat16):
            got = _run(q, plan, X, W, GY, "fwd", dtype)
            ref = O.gemm_oracle("fwd", strategy, bf16_bits(X), bf16_bits(W), None, patterns=pats, r=r)
            assert O.rel_frobenius(got, ref["C"]) <= TOL[dtype]


def _sampled_parity(q, wl_name, li, n_rows=48, n_cols=None, dtype=torch.float32):
    """The three GEMMs of linear `li` of a workload through the C ABI, compared with the oracle on
    sampled rows (and, with n_cols, sampled columns: the oracle then quantises only the operand
    lines of that block, so full-size shapes stay quick on the host)."""
    wl = WORKLOADS[wl_name]
    X, W, GY = tensor_recipes(wl, li, device="cuda")
    M, K = X.shape
    N = W.shape[0]
    cal_ws = q.new_workspace(1 << 22)
    plan = q.adahop_calibrate(X, W, GY, cal_ws)
    Xb, Wb, Gb = bf16_bits(X), bf16_bits(W), bf16_bits(GY)
    want = O.calibrate(Xb, Wb, Gb)
    assert (plan.x, plan.w, plan.gy) == (want["patterns"]["X"], want["patterns"]["W"], want["patterns"]["GY"])
    ws = q.new_workspace(q.adahop_workspace_size(plan, M, N, K))
    Y = torch.empty((M, N), dtype=dtype, device="cuda")
    dX = torch.empty((M, K), dtype=dtype, device="cuda")
    dW = torch.empty((N, K), dtype=dtype, device="cuda")
    q.adahop_linear_fwd(plan, X, W, Y, ws)
    q.adahop_linear_bwd(plan, GY, X, W, dX, dW, ws)
    assert q.adahop_get_device_status(ws) == 0
    rng = np.random.default_rng(li)
    strategies = {"fwd": plan.fwd, "dgrad": plan.dgrad, "wgrad": plan.wgrad}
    for gemm, out in (("fwd", Y), ("dgrad", dX), ("wgrad", dW)):
        P, Qn = out.shape
        rows = np.sort(rng.choice(P, n_rows, replace=False))
        cols = None if n_cols is None else np.sort(rng.choice(Qn, n_cols, replace=False))
        oe = O.gemm_plan(gemm, strategies[gemm], want["patterns"], plan.oe_rank, {"X": Xb, "W": Wb, "GY": Gb})
        if oe is not None and oe["role"] == "P":
            rows = np.unique(np.concatenate([rows, oe["idx"][:8]]))
        if oe is not None and oe["role"] == "Q" and cols is not None:
            cols = np.unique(np.concatenate([cols, oe["idx"][:8]]))
        ref = O.gemm_oracle(gemm, strategies[gemm], Xb, Wb, Gb, patterns=want["patterns"], r=plan.oe_rank,
                            rows=rows, cols=cols, oe=oe)
        got = out[torch.from_numpy(rows).cuda()]
        if cols is not None:
            got = got[:, torch.from_numpy(cols).cuda()]
        got = got.float().cpu().numpy().astype(np.float64)
        err = O.rel_frobenius(got, ref["C"])
        assert err <= TOL[dtype], (wl_name, li, gemm, err)


@pytest.mark.parametrize("li", [0, 1, 4, 6])
def test_llama_1b_config_sampled(q, li):
    _sampled_parity(q, "llama3.2-1b", li)


@pytest.mark.parametrize("li", [0, 1, 2, 3])
def test_instella_3b_config_sampled(q, li):
    _sampled_parity(q, "instella-3b", li, dtype=torch.bfloat16)


@pytest.mark.parametrize("li", [1, 3, 4, 6])
def test_llama_8b_config_sampled(q, li):
    """Full-size Llama3.1-8B linears in the bench's launch configuration, checked on sampled rows
    of all three GEMMs: k (N = 1024: the J = 1024 dgrad), o (N = K = 4096: its wgrad, 4096 x 4096
    x 32768 with the rank-64 tail, runs stream-K), gate (N = 14336, K = 4096) and down (N = 4096,
    K = 14336: J = 14336 in Fwd, Q = 14336 in dgrad)."""
    _sampled_parity(q, "llama3.1-8b", li, n_rows=32, n_cols=96, dtype=torch.bfloat16)

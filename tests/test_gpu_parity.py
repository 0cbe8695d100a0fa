"""GPU <-> oracle parity through the C ABI (sm_103a library), on small and ragged shapes.

Bar (from the method's statement of the target): bit-exact FOID indices, pattern classes, MXFP4
codes and scales; GEMM outputs within relative Frobenius error 2e-3 of the oracle's float64
product of the same dequantised operands for float32 output, 4e-3 for bf16 output (one extra
bf16 rounding, 2^-9 relative per element).
"""
import numpy as np
import pytest
import torch

import oracle as O
from synthetic import normal_bf16, bf16_bits
from tests.gpu_util import (bitmap, dev_bf16_from_bits, from_tiled, to_dev, to_host_u8, to_tiled)

pytestmark = pytest.mark.gpu

TOL_FP32 = 2e-3
TOL_BF16 = 4e-3


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as lib
    return lib


def _bits(shape, seed, std=1.0, axis=None, count=0, scale=1.0):
    return bf16_bits(normal_bf16(*shape, std, seed, outlier_axis=axis, outlier_count=count,
                                 outlier_scale=scale))


# ------------------------------------------------------------------------------ K2 quantiser
@pytest.mark.parametrize("shape", [(128, 128), (256, 512), (384, 1152)])
@pytest.mark.parametrize("hadamard", [1, 0])
@pytest.mark.parametrize("inner_axis", [1, 0])
def test_quantize_bitexact(q, shape, hadamard, inner_axis):
    T = _bits(shape, 11, axis="col", count=5, scale=50.0)
    rows, cols = shape
    zr = [0, 7, rows - 1]
    zc = [3, 64, cols - 2]
    ref_in = T if inner_axis == 1 else np.ascontiguousarray(T.T)
    lines, J = ref_in.shape
    dT = dev_bf16_from_bits(T)
    for zero_rows, zero_cols in ((None, None), (zr, None), (None, zc), (zr, zc)):
        codes = torch.zeros(lines * J // 2, dtype=torch.uint8, device="cuda")
        scales = torch.zeros(lines * J // 32, dtype=torch.uint8, device="cuda")
        mr = to_dev(bitmap(rows, zero_rows)) if zero_rows else None
        mc = to_dev(bitmap(cols, zero_cols)) if zero_cols else None
        q.adahop_quantize_mxfp4(dT, inner_axis, hadamard, mr, mc, codes, scales, 0)
        torch.cuda.synchronize()
        # the oracle's line/J view of the same zeroing
        o_rows, o_cols = (zero_rows, zero_cols) if inner_axis == 1 else (zero_cols, zero_rows)
        want_codes, want_scales = O.quantize_operand(ref_in, bool(hadamard), zero_rows=o_rows,
                                                     zero_cols=o_cols)
        got_codes = to_host_u8(codes).reshape(lines, J // 2)
        got_scales = to_host_u8(scales).reshape(lines, J // 32)
        assert np.array_equal(got_scales, want_scales)
        assert np.array_equal(got_codes, want_codes)
        # the tensor-core scale layout is the documented permutation of the canonical one
        tiled = torch.zeros_like(scales)
        q.adahop_quantize_mxfp4(dT, inner_axis, hadamard, mr, mc, codes, tiled, 1)
        torch.cuda.synchronize()
        assert np.array_equal(from_tiled(to_host_u8(tiled), lines, J), want_scales)


@pytest.mark.parametrize("shape", [(128, 128), (384, 256), (256, 640)])
@pytest.mark.parametrize("hadamard", [1, 0])
def test_quantize_dual_bitexact(q, shape, hadamard):
    """One pass, both orientations: each equals the oracle's quantisation of that orientation."""
    T = _bits(shape, 12, axis="row", count=6, scale=40.0)
    rows, cols = shape
    dT = dev_bf16_from_bits(T)
    for zero_rows, zero_cols in ((None, None), ([1, 33, rows - 1], None), (None, [0, 95, cols - 1])):
        mr = to_dev(bitmap(rows, zero_rows)) if zero_rows else None
        mc = to_dev(bitmap(cols, zero_cols)) if zero_cols else None
        for layout in (0, 1):
            cr = torch.zeros(rows * cols // 2, dtype=torch.uint8, device="cuda")
            sr = torch.zeros(rows * cols // 32, dtype=torch.uint8, device="cuda")
            cc = torch.zeros_like(cr)
            sc = torch.zeros_like(sr)
            q.adahop_quantize_mxfp4_dual(dT, hadamard, mr, mc, cr, sr, cc, sc, layout)
            torch.cuda.synchronize()
            wcr, wsr = O.quantize_operand(T, bool(hadamard), zero_rows=zero_rows, zero_cols=zero_cols)
            wcc, wsc = O.quantize_operand(np.ascontiguousarray(T.T), bool(hadamard), zero_rows=zero_cols,
                                          zero_cols=zero_rows)
            assert np.array_equal(to_host_u8(cr).reshape(rows, cols // 2), wcr)
            assert np.array_equal(to_host_u8(cc).reshape(cols, rows // 2), wcc)
            got_sr, got_sc = to_host_u8(sr), to_host_u8(sc)
            if layout == 1:
                got_sr, got_sc = from_tiled(got_sr, rows, cols), from_tiled(got_sc, cols, rows)
            assert np.array_equal(got_sr.reshape(rows, -1), wsr)
            assert np.array_equal(got_sc.reshape(cols, -1), wsc)


def test_quantize_edge_values(q):
    """All-zero blocks, tiny (subnormal-scale) blocks, exact ties and huge values."""
    rows, cols = 128, 256
    x = np.zeros((rows, cols), np.float32)
    x[1, :32] = 2.0 ** -130 * np.arange(32)                    # subnormal amax
    x[2, :32] = np.array([6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25] * 4, np.float32)
    x[3, :32] = -x[2, :32]
    # large but finite through the Hadamard: 32 summands of at most 1e37 stay below 3.4e38
    # (inputs whose block transform overflows float32 are outside the documented domain)
    x[4, :] = 1.0e37 * np.cos(np.arange(cols))
    x[5, :] = np.float32(1.5) ** (np.arange(cols) % 64 - 32)
    T = O.f32_to_bf16_bits(x)
    dT = dev_bf16_from_bits(T)
    for had in (0, 1):
        for inner in (1, 0):
            ref_in = T if inner == 1 else np.ascontiguousarray(T.T)
            lines, J = ref_in.shape
            codes = torch.zeros(lines * J // 2, dtype=torch.uint8, device="cuda")
            scales = torch.zeros(lines * J // 32, dtype=torch.uint8, device="cuda")
            q.adahop_quantize_mxfp4(dT, inner, had, None, None, codes, scales, 0)
            torch.cuda.synchronize()
            wc, ws = O.quantize_operand(ref_in, bool(had))
            assert np.array_equal(to_host_u8(scales).reshape(lines, -1), ws)
            assert np.array_equal(to_host_u8(codes).reshape(lines, -1), wc)


def test_quantize_dual_edge_values(q):
    """The dual kernel on the edge values of both orientations: constant blocks (31 exact zeros
    after the transform, where the sign of zero decides the code), negative zeros, subnormal-scale,
    tie and huge blocks, along rows and along columns, in both 32-row halves of the staged tile."""
    rows, cols = 128, 256
    x = np.zeros((rows, cols), np.float32)
    x[1, :32] = 2.0 ** -130 * np.arange(32)
    x[2, :32] = np.array([6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25] * 4, np.float32)
    x[3, 32:64] = -x[2, :32]
    x[4, 64:96] = 0.5                                          # constant along a row block
    x[5, 96:128] = -0.0
    x[6, :] = 1.0e37 * np.cos(np.arange(cols))
    x[40, 128:160] = -3.0
    x[33:65, 7] = 0.75                                         # constant along a column block
    x[64:96, 9] = np.array([6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25] * 4, np.float32)
    x[96:128, 130] = 2.0 ** -135 * np.arange(32)
    x[32:64, 200] = -0.0
    x[:, 255] = np.float32(1.5) ** (np.arange(rows) % 64 - 32)
    T = O.f32_to_bf16_bits(x)
    dT = dev_bf16_from_bits(T)
    for had in (1, 0):
        cr = torch.zeros(rows * cols // 2, dtype=torch.uint8, device="cuda")
        sr = torch.zeros(rows * cols // 32, dtype=torch.uint8, device="cuda")
        cc = torch.zeros_like(cr)
        sc = torch.zeros_like(sr)
        q.adahop_quantize_mxfp4_dual(dT, had, None, None, cr, sr, cc, sc, 0)
        torch.cuda.synchronize()
        wcr, wsr = O.quantize_operand(T, bool(had))
        wcc, wsc = O.quantize_operand(np.ascontiguousarray(T.T), bool(had))
        assert np.array_equal(to_host_u8(cr).reshape(rows, -1), wcr)
        assert np.array_equal(to_host_u8(sr).reshape(rows, -1), wsr)
        assert np.array_equal(to_host_u8(cc).reshape(cols, -1), wcc)
        assert np.array_equal(to_host_u8(sc).reshape(cols, -1), wsc)


# ------------------------------------------------------------------------------ K1 FOID
@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("shape,r", [((256, 512), 16), ((4096, 640), 64), ((128, 2560), 1),
                                     ((640, 4224), 256), ((1024, 256), 0)])
def test_foid_bitexact(q, axis, shape, r):
    lines = shape[axis]
    if r > lines:
        pytest.skip("rank beyond lines")
    T = _bits(shape, 21, axis="col" if axis else "row", count=min(8, r + 1), scale=40.0)
    dT = dev_bf16_from_bits(T)
    idx = torch.full((max(r, 1),), -1, dtype=torch.int32, device="cuda")
    mask = torch.full(((lines + 31) // 32,), -1, dtype=torch.int32, device="cuda")
    ws = q.new_workspace(q.adahop_foid_workspace_size(lines, r))
    q.adahop_foid(dT, axis, r, idx, mask, ws)
    torch.cuda.synchronize()
    want = O.foid(T, "row" if axis == 0 else "col", r)
    assert idx.cpu().numpy()[:r].tolist() == want.tolist()
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), bitmap(lines, want))


def test_foid_ties_and_duplicates(q):
    alt = np.where(np.arange(64) % 2, -1.0, 1.0)
    x = np.tile(np.concatenate([alt, np.zeros(64)]), (300, 1)).astype(np.float32)
    x[[5, 77, 150], :64] *= 3.0        # three clear winners, the rest tie
    T = O.f32_to_bf16_bits(x)
    dT = dev_bf16_from_bits(T)
    for r in (3, 10, 64):
        idx = torch.zeros(r, dtype=torch.int32, device="cuda")
        ws = q.new_workspace(q.adahop_foid_workspace_size(300, r))
        q.adahop_foid(dT, 0, r, idx, None, ws)
        torch.cuda.synchronize()
        assert idx.cpu().numpy().tolist() == O.foid(T, "row", r).tolist()


@pytest.mark.parametrize("axis", [0, 1])
def test_foid_ties_across_chunks_at_scale(q, axis):
    """32768 lines whose probes tie in three classes (variance 1, 4, 9): the top-r cut falls inside
    a tied band that straddles stage-1 chunk boundaries (256, 1024 and 2048 lines per chunk for
    r = 64 / 256), so the merge must break ties to the lower index across runs.  Bit-exact
    against the oracle and against the set fixed by construction."""
    L = 32768
    alt = np.where(np.arange(64) % 2, -1.0, 1.0)
    probe = np.tile(alt, (L, 1))
    winners = np.array([7, 9000, 20000, 32767])
    mid = np.concatenate([np.arange(250, 263), np.arange(1020, 1031), np.arange(2040, 2057),
                          np.arange(32752, 32760), [4095, 4096, 16383, 16384]])
    probe[mid] *= 2.0                            # variance 4
    probe[winners] *= 3.0                        # variance 9
    bits = O.f32_to_bf16_bits(probe.astype(np.float32))            # L x 64: line l = row l
    T = bits if axis == 0 else np.ascontiguousarray(bits.T)        # 64 x L: line l = column l
    dT = dev_bf16_from_bits(T)
    mid_sorted = np.sort(mid)
    for r in (1, 4, 33, 40, 64, 77, 256):
        # by construction: the winners, then the lowest-indexed tied lines of each class in turn
        base = np.setdiff1d(np.arange(L), np.concatenate([winners, mid]))
        ranked = np.concatenate([winners, mid_sorted, base])[:r]
        want = np.sort(ranked)
        assert np.array_equal(O.foid(T, "row" if axis == 0 else "col", r), want)
        idx = torch.full((r,), -1, dtype=torch.int32, device="cuda")
        mask = torch.full(((L + 31) // 32,), -1, dtype=torch.int32, device="cuda")
        ws = q.new_workspace(q.adahop_foid_workspace_size(L, r))
        q.adahop_foid(dT, axis, r, idx, mask, ws)
        torch.cuda.synchronize()
        assert q.adahop_get_device_status(ws) == 0
        assert np.array_equal(idx.cpu().numpy(), want), (axis, r)
        assert np.array_equal(mask.cpu().numpy().view(np.uint32), bitmap(L, want)), (axis, r)
    # every line tied: the r lowest indices
    flat = O.f32_to_bf16_bits(np.tile(alt, (L, 1)).astype(np.float32))
    dflat = dev_bf16_from_bits(flat if axis == 0 else np.ascontiguousarray(flat.T))
    for r in (64, 256):
        idx = torch.full((r,), -1, dtype=torch.int32, device="cuda")
        ws = q.new_workspace(q.adahop_foid_workspace_size(L, r))
        q.adahop_foid(dflat, axis, r, idx, None, ws)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), np.arange(r)), (axis, r)


# ------------------------------------------------------------------------------ calibration
def test_calibration_classes(q):
    from synthetic import WORKLOADS, tensor_recipes
    wl = WORKLOADS["llama3.2-1b"]
    for li in (0, 4):
        X, W, GY = tensor_recipes(wl, li)
        want = O.calibrate(bf16_bits(X), bf16_bits(W), bf16_bits(GY))
        dX, dW, dG = X.cuda(), W.cuda(), GY.cuda()
        M, K = X.shape
        N = W.shape[0]
        ws = q.new_workspace(16384 + 4 * (max(M, N) + max(N, K)) + 512)   # zeroed header + statistics
        plan = q.adahop_calibrate(dX, dW, dG, ws)
        assert (plan.x, plan.w, plan.gy) == (want["patterns"]["X"], want["patterns"]["W"],
                                             want["patterns"]["GY"])
        assert (plan.fwd, plan.dgrad, plan.wgrad) == (want["fwd"], want["dgrad"], want["wgrad"])


# ------------------------------------------------------------------------------ GEMMs
def _rel(got, ref):
    return O.rel_frobenius(got, ref)


# J <= 2048 and J > 2048 run different pipeline configurations of the kernel (384, 2176 and 2432:
# odd multiples of 128, whose last 256-wide slice of J is half full)
@pytest.mark.parametrize("P,Q,J", [(128, 256, 256), (256, 512, 384), (384, 384, 1024), (128, 128, 128),
                                   (128, 256, 2176), (256, 384, 2304), (256, 128, 2432), (384, 256, 4096)])
@pytest.mark.parametrize("r", [0, 16, 64, 128])
@pytest.mark.parametrize("out", ["fp32", "bf16"])
@pytest.mark.parametrize("stream_k", [False, True])
def test_gemm_mxfp4_against_oracle(q, P, Q, J, r, out, stream_k):
    """With a 4 KB workspace and with the one that allows stream-K (these shapes have too few tiles
    for it, so both run whole tiles: the larger workspace changes nothing here)."""
    A = _bits((P, J), 31, axis="col", count=4, scale=30.0)
    Bt = _bits((Q, J), 32, std=0.02)
    ac, asf = O.quantize_operand(A, True)
    bc, bsf = O.quantize_operand(Bt, True)
    ref = O.dequantize_operand(ac, asf) @ O.dequantize_operand(bc, bsf).T
    Ao = Bo = None
    if r:
        Ao_bits = _bits((P, r), 33, std=5.0)
        Bo_bits = _bits((Q, r), 34, std=0.02)
        ref = ref + O.bf16_to_f32(Ao_bits).astype(np.float64) @ O.bf16_to_f32(Bo_bits).astype(np.float64).T
        Ao, Bo = dev_bf16_from_bits(Ao_bits), dev_bf16_from_bits(Bo_bits)
    C = torch.zeros((P, Q), dtype=torch.float32 if out == "fp32" else torch.bfloat16, device="cuda")
    ws = q.new_workspace(q.adahop_gemm_mxfp4_workspace_size() if stream_k else 4096)
    args = (to_dev(ac), to_dev(to_tiled(asf)), to_dev(bc), to_dev(to_tiled(bsf)), P, Q, J, Ao, Bo, r)
    q.adahop_gemm_mxfp4(*args, C, ws)
    assert q.adahop_get_device_status(ws) == 0
    got = C.float().cpu().numpy().astype(np.float64)
    assert _rel(got, ref) <= (TOL_FP32 if out == "fp32" else TOL_BF16)
    if out == "fp32":
        assert _rel(got, ref) <= 1e-5          # float32 accumulation of exact products
    if stream_k:
        C2 = torch.full_like(C, 7.0)
        q.adahop_gemm_mxfp4(*args, C2, ws)
        assert q.adahop_get_device_status(ws) == 0
        assert torch.equal(C, C2)


# at least two whole rounds of 256 x 256 tiles over the CTA pairs, a short last round and a long J:
# the shapes the fused GEMM balances with stream-K (160 tiles; 256 tiles like the q / o wgrad)
@pytest.mark.parametrize("P,Q,J,r", [(4096, 2560, 16384, 0), (4096, 2560, 16384, 64), (4096, 4096, 32768, 64)])
def test_gemm_mxfp4_stream_k_matches_whole_tiles(q, P, Q, J, r):
    """Stream-K (the workspace the entry point asks for) against whole tiles (a 4 KB workspace,
    itself checked against the oracle above): equal to float32 rounding of the reordered sums,
    bit-identical on a second call, and the counters left at zero."""
    A = normal_bf16(P, J, 1.0, 41, device="cuda")
    B = normal_bf16(Q, J, 0.02, 42, device="cuda")
    ac = torch.empty(P * J // 2, dtype=torch.uint8, device="cuda")
    asf = torch.empty(P * J // 32, dtype=torch.uint8, device="cuda")
    bc = torch.empty(Q * J // 2, dtype=torch.uint8, device="cuda")
    bsf = torch.empty(Q * J // 32, dtype=torch.uint8, device="cuda")
    q.adahop_quantize_mxfp4(A, 1, 1, None, None, ac, asf, 1)
    q.adahop_quantize_mxfp4(B, 1, 1, None, None, bc, bsf, 1)
    del A, B
    Ao = normal_bf16(P, r, 5.0, 43, device="cuda") if r else None
    Bo = normal_bf16(Q, r, 0.02, 44, device="cuda") if r else None
    Cw = torch.empty((P, Q), dtype=torch.float32, device="cuda")
    Cs = torch.empty((P, Q), dtype=torch.float32, device="cuda")
    ws_w = q.new_workspace(4096)
    ws_s = q.new_workspace(q.adahop_gemm_mxfp4_workspace_size())
    q.adahop_gemm_mxfp4(ac, asf, bc, bsf, P, Q, J, Ao, Bo, r, Cw, ws_w)
    q.adahop_gemm_mxfp4(ac, asf, bc, bsf, P, Q, J, Ao, Bo, r, Cs, ws_s)
    assert q.adahop_get_device_status(ws_w) == 0 and q.adahop_get_device_status(ws_s) == 0
    diff = (Cs.double() - Cw.double()).norm() / Cw.double().norm()
    assert float(diff) <= 1e-6
    Cs2 = torch.full_like(Cs, 3.0)
    q.adahop_gemm_mxfp4(ac, asf, bc, bsf, P, Q, J, Ao, Bo, r, Cs2, ws_s)
    assert q.adahop_get_device_status(ws_s) == 0
    assert torch.equal(Cs, Cs2)
    assert int(ws_s[:16384].count_nonzero()) == 0


@pytest.mark.parametrize("a_kmajor,b_kmajor", [(1, 1), (1, 0), (0, 0), (0, 1)])
@pytest.mark.parametrize("P,Q,J", [(128, 256, 128), (256, 512, 320), (64, 192, 256)])
def test_gemm_bf16_layouts(q, a_kmajor, b_kmajor, P, Q, J):
    A = _bits((P, J), 41)              # logical A: P x J
    B = _bits((J, Q), 42, std=0.5)     # logical B: J x Q
    ref = O.bf16_to_f32(A).astype(np.float64) @ O.bf16_to_f32(B).astype(np.float64)
    dA = dev_bf16_from_bits(A if a_kmajor else np.ascontiguousarray(A.T))
    dB = dev_bf16_from_bits(np.ascontiguousarray(B.T) if b_kmajor else B)
    C = torch.zeros((P, Q), dtype=torch.float32, device="cuda")
    ws = q.new_workspace(4096)
    q.adahop_gemm_bf16(dA, a_kmajor, dB, b_kmajor, P, Q, J, C, ws)
    assert q.adahop_get_device_status(ws) == 0
    assert _rel(C.cpu().numpy(), ref) <= 1e-5


@pytest.mark.parametrize("J,S", [(1024, 4), (128, 5)])
def test_gemm_bf16_split_partials(q, J, S):
    # (128, 5): J holds two 64-wide K stages, so splits 1..4 have empty ranges and must hold zeros
    P, Q = 64, 256
    A = _bits((P, J), 51)
    B = _bits((J, Q), 52)
    ref = O.bf16_to_f32(A).astype(np.float64) @ O.bf16_to_f32(B).astype(np.float64)
    part = torch.full((S, P, Q), float("nan"), dtype=torch.float32, device="cuda")
    ws = q.new_workspace(4096)
    q.adahop_gemm_bf16(dev_bf16_from_bits(A), 1, dev_bf16_from_bits(B), 0, P, Q, J, None, ws, splits=S,
                       c_partial=part)
    torch.cuda.synchronize()
    assert _rel(part.sum(0).cpu().numpy(), ref) <= 1e-5
    per = -(-(J // 64) // S)
    for s in range(S):
        if s * per >= J // 64:
            assert torch.count_nonzero(part[s]).item() == 0


# ------------------------------------------------------------------------------ scatter-add
# (P or Q, the other dimension, J): the cluster's split count runs through 1, 2, 4 and 8
@pytest.mark.parametrize("axis,other,J,b_kmajor", [
    (0, 256, 128, 1), (0, 512, 512, 0), (0, 256, 2048, 1), (0, 4096, 2048, 0),
    (1, 320, 256, 1), (1, 1024, 4096, 1), (1, 384, 1024, 0)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gemm_bf16_scatter_add(q, axis, other, J, b_kmajor, dtype):
    """The outer-OE outlier GEMM with the scatter-add fused: C[idx, :] += A . B (axis 0) or
    C[:, idx] += A . B (axis 1) against the float64 product added to C's previous values; every
    other element of C is left bit for bit as it was."""
    r = 64
    rng = np.random.default_rng(J + other + axis)
    if axis == 0:
        P, Q = r, other
        c_rows, c_cols = 1024, Q
        idx = np.sort(rng.choice(c_rows, r, replace=False)).astype(np.int32)
    else:
        P, Q = other, r
        c_rows, c_cols = P, 768
        idx = np.sort(rng.choice(c_cols, r, replace=False)).astype(np.int32)
    A = _bits((P, J), 3, std=1.0)                            # K-major: P x J
    B = _bits((Q, J) if b_kmajor else (J, Q), 4, std=0.05)   # K-major Q x J, or stored J x Q
    C0 = torch.randn((c_rows, c_cols), generator=torch.Generator().manual_seed(5)).to(dtype)
    C = C0.cuda()
    ws = q.new_workspace(256)
    q.adahop_gemm_bf16_scatter_add(dev_bf16_from_bits(A), 1, dev_bf16_from_bits(B), b_kmajor, P, Q, J, C,
                                   torch.from_numpy(idx).cuda(), r, axis, ws)
    torch.cuda.synchronize()
    assert q.adahop_get_device_status(ws) == 0
    f = lambda b: O.bf16_to_f32(b).astype(np.float64)
    prod = f(A) @ (f(B).T if b_kmajor else f(B))             # P x Q
    got = C.float().cpu().numpy().astype(np.float64)
    before = C0.float().numpy().astype(np.float64)
    want = before.copy()
    if axis == 0:
        want[idx, :] += prod
        touched = np.zeros(c_rows, bool)
        touched[idx] = True
        assert np.array_equal(got[~touched], before[~touched])
        err = O.rel_frobenius(got[idx] - before[idx], want[idx] - before[idx])
    else:
        want[:, idx] += prod
        touched = np.zeros(c_cols, bool)
        touched[idx] = True
        assert np.array_equal(got[:, ~touched], before[:, ~touched])
        err = O.rel_frobenius(got[:, idx] - before[:, idx], want[:, idx] - before[:, idx])
    # the added part, measured against the exact product: one float32 sum, one rounding of C
    tol = TOL_FP32 if dtype == torch.float32 else 2e-2
    assert err <= tol, err
    if dtype == torch.float32:
        assert O.rel_frobenius(got, want) <= 1e-5


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_scatter_add(q, axis, dtype):
    P, Q, r, S = 256, 384, 24, 3
    rng = np.random.default_rng(5)
    idx = np.sort(rng.choice(P if axis == 0 else Q, r, replace=False)).astype(np.int32)
    C0 = rng.standard_normal((P, Q)).astype(np.float32)
    part = rng.standard_normal((S, r, Q) if axis == 0 else (S, P, r)).astype(np.float32)
    dC = torch.from_numpy(C0).to(dtype).cuda()
    base = dC.float().cpu().numpy().astype(np.float64)
    q.adahop_scatter_add(dC, to_dev(part), S, to_dev(idx), r, axis)
    torch.cuda.synchronize()
    want = base.copy()
    summed = part.astype(np.float32).sum(0, dtype=np.float32)
    if axis == 0:
        want[idx, :] = (base[idx, :].astype(np.float32) + summed).astype(np.float64)
    else:
        want[:, idx] = (base[:, idx].astype(np.float32) + summed).astype(np.float64)
    got = dC.float().cpu().numpy()
    tol = 1e-6 if dtype == torch.float32 else 2 ** -8
    assert np.allclose(got, want, rtol=tol, atol=tol)


# ------------------------------------------------------------------------------ outlier-slice gathers
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("shape,r", [((256, 512), 64), ((384, 1152), 32), ((320, 96), 24), ((128, 256), 8),
                                     ((4096, 14336), 64)])
def test_gather_bitexact(q, mode, shape, r):
    """adahop_gather moves bf16 values without arithmetic, so every mode must match plain indexing
    bit for bit (mode 2 covers both its vectorised path, columns % 64 == 0 and r % 32 == 0, and
    the general one)."""
    rows, cols = shape
    lines = rows if mode in (0, 2) else cols
    T = torch.randn(shape, generator=torch.Generator().manual_seed(rows + cols + r)).to(torch.bfloat16)
    sel = torch.randperm(lines, generator=torch.Generator().manual_seed(r))[:r].sort().values
    if r > 1:
        sel[1] = sel[0]                                  # a repeated index is gathered twice
    idx = sel.to(torch.int32).cuda()
    dT = T.cuda()
    if mode == 0:
        want = T[sel.long(), :]
    elif mode == 1:
        want = T[:, sel.long()]
    elif mode == 2:
        want = T[sel.long(), :].t()
    else:
        want = T[:, sel.long()].t()
    out = torch.full(tuple(want.shape), float("nan"), dtype=torch.bfloat16, device="cuda")
    q.adahop_gather(dT, idx, r, mode, out)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().view(torch.int16), want.contiguous().view(torch.int16))

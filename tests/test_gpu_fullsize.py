"""Bit-exact parity of K1 (FOID) and K2 (the dual-orientation IHT + MXFP4 quantiser) at the full
size of the Llama3.1-8B gate projection's G_Y (32768 x 14336, Row-wise: 64 rows x40), in the
launch configuration the bench times (tensor-core scale layout, FOID's zero mask), checked on
sampled lines that the oracle computes one by one.  The GEMMs at this size are covered by
test_gpu_linear.py::test_llama_8b_config_sampled."""
import numpy as np
import pytest
import torch

import oracle as O
from synthetic import WORKLOADS, bf16_bits, tensor_recipes
from tests.gpu_util import from_tiled, to_host_u8

pytestmark = pytest.mark.gpu

GATE = 4                     # the gate projection of the block: N = 14336, K = 4096
R = 64


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as lib
    return lib


@pytest.fixture(scope="module")
def gate_gy():
    _, _, GY = tensor_recipes(WORKLOADS["llama3.1-8b"], GATE, device="cuda")
    return GY


@pytest.fixture(scope="module")
def foid_rows(q, gate_gy):
    M = gate_gy.shape[0]
    idx = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    mask = torch.full(((M + 31) // 32,), -1, dtype=torch.int32, device="cuda")
    ws = q.new_workspace(q.adahop_foid_workspace_size(M, R))
    q.adahop_foid(gate_gy, 0, R, idx, mask, ws)
    torch.cuda.synchronize()
    assert q.adahop_get_device_status(ws) == 0
    return idx, mask


def test_foid_full_size(q, gate_gy, foid_rows):
    idx, mask = foid_rows
    M = gate_gy.shape[0]
    want = O.foid(bf16_bits(gate_gy[:, :64]), "row", R)        # the probe is the first 64 columns
    assert np.array_equal(idx.cpu().numpy(), want)
    words = mask.cpu().numpy().view(np.uint32)
    got_lines = np.nonzero((words[np.arange(M) >> 5] >> (np.arange(M) & 31).astype(np.uint32)) & 1)[0]
    assert np.array_equal(got_lines, want)


def test_quantize_dual_full_size_sampled_lines(q, gate_gy, foid_rows):
    idx, mask = foid_rows
    M, N = gate_gy.shape
    n = M * N
    cr = torch.empty(n // 2, dtype=torch.uint8, device="cuda")
    sr = torch.empty(n // 32, dtype=torch.uint8, device="cuda")
    cc = torch.empty(n // 2, dtype=torch.uint8, device="cuda")
    sc = torch.empty(n // 32, dtype=torch.uint8, device="cuda")
    q.adahop_quantize_mxfp4_dual(gate_gy, 1, mask, None, cr, sr, cc, sc, 1)
    torch.cuda.synchronize()
    zeroed = idx.cpu().numpy().astype(np.int64)
    rng = np.random.default_rng(5)

    # rows (lines = rows of G_Y, J = N): some extracted rows, rows from both halves of a 64-row
    # tile, the last row, and random ones
    rows = np.unique(np.concatenate([zeroed[:4], [0, 31, 32, 63, 64, M - 1], rng.choice(M, 24, replace=False)]))
    T_rows = bf16_bits(gate_gy[torch.from_numpy(rows).cuda()])
    wc, ws = O.quantize_operand(T_rows, True, zero_rows=np.nonzero(np.isin(rows, zeroed))[0])
    got_c = cr.view(M, N // 2)[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(got_c, wc)
    assert np.array_equal(from_tiled(to_host_u8(sr), rows, N), ws)

    # columns (lines = columns of G_Y, J = M): every extracted row is zeroed along J
    cols = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.choice(N, 24, replace=False)]))
    T_cols = bf16_bits(gate_gy[:, torch.from_numpy(cols).cuda()].t().contiguous())
    wc, ws = O.quantize_operand(T_cols, True, zero_cols=zeroed)
    got_c = cc.view(N, M // 2)[torch.from_numpy(cols).cuda()].cpu().numpy()
    assert np.array_equal(got_c, wc)
    assert np.array_equal(from_tiled(to_host_u8(sc), cols, M), ws)


def test_quantize_dual_64bit_offsets():
    """A tensor of 2^31 elements (32768 x 65536, 4 GiB of bf16), which takes the dual quantiser's
    64-bit-offset instantiation (below 2^31 elements it computes offsets in 32 bits): both
    orientations equal the single-orientation kernels bit for bit, and sampled lines near the
    ends of the tensor, where the offsets pass 2^31, equal the oracle's.  About 17 GB on the
    device at the peak (the float32 draw of the tensor)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as q
    from synthetic import normal_bf16
    M, N = 32768, 65536
    n = M * N
    assert n == 1 << 31
    T = normal_bf16(M, N, 1.0, 11, device="cuda")
    bufs = [torch.empty(k, dtype=torch.uint8, device="cuda") for k in (n // 2, n // 32, n // 2, n // 32)]
    cr, sr, cc, sc = bufs
    q.adahop_quantize_mxfp4_dual(T, 1, None, None, cr, sr, cc, sc, 1)
    for axis, codes, scales in ((1, cr, sr), (0, cc, sc)):
        c1 = torch.empty_like(codes)
        s1 = torch.empty_like(scales)
        q.adahop_quantize_mxfp4(T, axis, 1, None, None, c1, s1, 1)
        torch.cuda.synchronize()
        assert torch.equal(c1, codes) and torch.equal(s1, scales)
        del c1, s1
    rows = np.array([0, 1, M // 2, M - 65, M - 2, M - 1])
    wc, ws = O.quantize_operand(bf16_bits(T[torch.from_numpy(rows).cuda()]), True)
    assert np.array_equal(cr.view(M, N // 2)[torch.from_numpy(rows).cuda()].cpu().numpy(), wc)
    assert np.array_equal(from_tiled(to_host_u8(sr), rows, N), ws)
    cols = np.array([0, 127, N // 2, N - 129, N - 1])
    wc, ws = O.quantize_operand(bf16_bits(T[:, torch.from_numpy(cols).cuda()].t().contiguous()), True)
    assert np.array_equal(cc.view(N, M // 2)[torch.from_numpy(cols).cuda()].cpu().numpy(), wc)
    assert np.array_equal(from_tiled(to_host_u8(sc), cols, M), ws)

"""The allocation-free FOID entry point (adahop_foid_noalloc) against the workspace one.

adahop_foid_noalloc serves callers that cannot allocate device memory (code handed only its
inputs and outputs, or that must not call cudaMalloc); it keeps its scratch in a fixed device
array inside the library.  Its results must equal adahop_foid's exactly (FOID is integer work:
indices and a bitmap), on consecutive calls that reuse the same array, in a fresh process or
after every other test.  This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synthetic import bf16_bits, normal_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as lib
    return lib


def _both(q, T, axis, r):
    lines = T.shape[axis]
    words = (lines + 31) // 32
    idx_ref = torch.full((max(r, 1),), -7, dtype=torch.int32, device="cuda")
    mask_ref = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    ws = q.new_workspace(q.adahop_foid_workspace_size(lines, r))
    q.adahop_foid(T, axis, r, idx_ref, mask_ref, ws)
    idx = torch.full((max(r, 1),), -9, dtype=torch.int32, device="cuda")
    mask = torch.full((words,), -9, dtype=torch.int32, device="cuda")
    q.adahop_foid_noalloc(T, axis, r, idx, mask)
    torch.cuda.synchronize()
    return idx_ref.cpu().numpy()[:r], mask_ref.cpu().numpy(), idx.cpu().numpy()[:r], mask.cpu().numpy()


def test_noalloc_foid_matches_workspace_foid_on_two_calls_in_a_row(q):
    # two consecutive calls with different inputs and ranks: the second reuses the fixed array
    cases = [((4096, 640), 0, 64, 1), ((640, 4224), 1, 256, 2)]
    for (rows, cols), axis, r, seed in cases:
        T = normal_bf16(rows, cols, 1.0, seed, outlier_axis="row" if axis == 0 else "col",
                        outlier_count=12, outlier_scale=40.0, device="cuda")
        idx_ref, mask_ref, idx, mask = _both(q, T, axis, r)
        assert np.array_equal(idx, idx_ref)
        assert np.array_equal(mask, mask_ref)
        assert len(np.unique(idx)) == r and np.all(np.diff(idx) > 0)
        # and directly against the CPU oracle's FOID (appendix FOID paragraph), bit for bit
        assert np.array_equal(idx, O.foid(bf16_bits(T), "row" if axis == 0 else "col", r))


def test_noalloc_foid_rejects_requests_beyond_its_scratch(q):
    # ceil(67584 / 2048) * 256 = 33 * 256 = 8448 candidates > 8192: refused before any launch
    T = torch.zeros((67584, 64), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(256, dtype=torch.int32, device="cuda")
    with pytest.raises(q.AdahopError) as err:
        q.adahop_foid_noalloc(T, 0, 256, idx, None)
    assert err.value.status == 2           # ADAHOP_ERR_SHAPE
    # the same lines with a smaller rank fit (33 * 248 = 8184)
    q.adahop_foid_noalloc(T, 0, 248, idx, None)
    torch.cuda.synchronize()

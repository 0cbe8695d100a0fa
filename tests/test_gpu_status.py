"""The device-side failure path, exercised without a fault: a kernel's bounded wait runs out on
an mbarrier that nothing arrives on, the kernel records the timeout in the workspace status word
and returns, the host reads ADAHOP_ERR_TIMEOUT, and the context keeps working afterwards."""
import time

import numpy as np
import pytest
import torch

import oracle as O
from synthetic import bf16_bits, normal_bf16
from tests.gpu_util import dev_bf16_from_bits, to_host_u8

pytestmark = pytest.mark.gpu

ADAHOP_ERR_TIMEOUT = 5
WAIT_LIMIT_S = 2.0          # the library's bounded-wait limit


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as lib
    return lib


def test_bounded_wait_runs_out_reports_timeout_and_leaves_the_context_usable(q):
    ws = q.new_workspace(256)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    q.adahop_check_bounded_wait(ws)
    assert q.adahop_get_device_status(ws) == ADAHOP_ERR_TIMEOUT
    waited = time.perf_counter() - t0
    assert WAIT_LIMIT_S * 0.95 <= waited < WAIT_LIMIT_S + 10.0
    assert q.adahop_get_device_status(ws) == 0           # reading the word cleared it

    # the same workspace and context afterwards: a quantisation is still bit-exact
    T = bf16_bits(normal_bf16(128, 256, 1.0, 3))
    codes = torch.zeros(128 * 256 // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(128 * 256 // 32, dtype=torch.uint8, device="cuda")
    q.adahop_quantize_mxfp4(dev_bf16_from_bits(T), 1, 1, None, None, codes, scales, 0)
    assert q.adahop_get_device_status(ws) == 0
    wc, wsc = O.quantize_operand(T, True)
    assert np.array_equal(to_host_u8(codes).reshape(128, -1), wc)
    assert np.array_equal(to_host_u8(scales).reshape(128, -1), wsc)


def test_bounded_wait_probe_rejects_bad_workspaces(q):
    small = q.new_workspace(256)[:128]
    with pytest.raises(q.AdahopError) as e:
        q.adahop_check_bounded_wait(small)
    assert e.value.status == 7                             # ADAHOP_ERR_WORKSPACE
    misaligned = q.new_workspace(1024)[16:16 + 512]
    with pytest.raises(q.AdahopError) as e:
        q.adahop_check_bounded_wait(misaligned)
    assert e.value.status == 3                             # ADAHOP_ERR_ALIGN
    assert q.adahop_get_device_status(q.new_workspace(256)) == 0

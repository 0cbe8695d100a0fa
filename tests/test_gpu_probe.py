"""K8 peak probes on the GPU: the tensor-pipe rate probe runs every MMA kind to completion with no
device-side error and reports plausible per-CTA cycle counts; the copy probe copies exactly."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_gemm_foid_gb300 as q
    return q


@pytest.mark.parametrize("kind,sf_copies,n", [(0, 0, 256), (1, 0, 256), (1, 1, 256), (2, 0, 256), (2, 1, 256),
                                              (3, 0, 256), (0, 0, 128), (1, 1, 128)])
def test_mma_rate_probe(q, kind, sf_copies, n):
    ctas = q.adahop_probe_ctas()
    assert ctas > 0
    out = torch.zeros(3 * ctas, dtype=torch.int64, device="cuda")
    ws = q.new_workspace(256)
    iters = 2000
    q.adahop_probe_mma_rate(kind, sf_copies, iters, out, ws, n=n)
    assert q.adahop_get_device_status(ws) == 0
    rec = out.view(ctas, 3).cpu()
    cycles = rec[:, 0].double()
    assert bool((cycles > 0).all())
    assert bool((rec[:, 2] > rec[:, 1]).all())
    flop = 4 * 2 * 128 * n * q.MMA_K_PER_INSTR[kind] * iters
    per_clk = flop / cycles
    # the dense tensor pipe of one SM does between 2^11 and 2^17 FLOP per clock for these kinds;
    # anything outside means the probe did not run the MMAs it claims
    assert float(per_clk.min()) > 2048 and float(per_clk.max()) < 131072


def test_mma_rate_probe_rejects_bad_arguments(q):
    ws = q.new_workspace(256)
    out = torch.zeros(3 * q.adahop_probe_ctas(), dtype=torch.int64, device="cuda")
    with pytest.raises(q.AdahopError):
        q.adahop_probe_mma_rate(4, 0, 10, out, ws)
    with pytest.raises(q.AdahopError):
        q.adahop_probe_mma_rate(1, 0, 0, out, ws)
    with pytest.raises(q.AdahopError):
        q.adahop_probe_mma_rate(1, 0, 10, out[:3], ws)
    with pytest.raises(q.AdahopError):
        q.adahop_probe_mma_rate(1, 0, 10, out, ws, n=64)


def test_copy_probe(q):
    n = (64 << 20) + 48                       # 64 MiB and a tail of three 16-byte words
    src = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda")
    dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
    q.adahop_probe_copy(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)


def test_fill_probe(q):
    """src None: the write-only stream sets every bf16 of dst to 1.0 (bit pattern 0x3F80)."""
    n = (32 << 20) + 24                       # 64 MiB of bf16 and a tail of three 16-byte words
    dst = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    q.adahop_probe_copy(None, dst)
    torch.cuda.synchronize()
    assert bool((dst == 1.0).all())

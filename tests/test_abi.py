"""Host-only checks of the C ABI: the library loads, exports every function declared in
include/adahop.h, and rejects bad arguments before touching a device (no kernel launches)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "adahop.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(adahop_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from quantized_gemm_foid_gb300.build import build
    build()
    import quantized_gemm_foid_gb300 as q
    return q


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = _declared_functions()
    assert len(names) >= 15
    raw = C.CDLL(lib.LIB._name)
    for n in names:
        assert hasattr(raw, n), n
        assert n in lib.PROTOTYPES, f"{n} missing from the binding"
    assert set(lib.PROTOTYPES) == set(names)


def test_status_strings(lib):
    for st in range(8):
        assert lib.LIB.adahop_status_string(st)
    assert lib.LIB.adahop_status_string(99) == b"unknown status"


def test_default_options(lib):
    o = lib.adahop_default_options()
    assert (o.tau, o.probe_len, o.oe_rank) == (8.0, 64, 64)


def test_workspace_size_validation(lib):
    plan = lib.make_plan(oe_rank=64)
    n = lib.adahop_workspace_size(plan, 4096, 2048, 8192)
    assert n > 4096 * 8192 // 2
    bad = C.c_size_t(0)
    assert lib.LIB.adahop_workspace_size(C.byref(plan), 4096, 2048, 100, C.byref(bad)) == 2   # SHAPE
    plan.fwd = 9
    assert lib.LIB.adahop_workspace_size(C.byref(plan), 4096, 2048, 8192, C.byref(bad)) == 1  # INVALID
    plan.fwd = 0
    plan.oe_rank = 300
    assert lib.LIB.adahop_workspace_size(C.byref(plan), 4096, 2048, 8192, C.byref(bad)) == 2
    plan.oe_rank = 12        # any rank 0 .. 256 is accepted
    assert lib.LIB.adahop_workspace_size(C.byref(plan), 4096, 2048, 8192, C.byref(bad)) == 0
    plan.oe_rank = -1
    assert lib.LIB.adahop_workspace_size(C.byref(plan), 4096, 2048, 8192, C.byref(bad)) == 2


def test_argument_errors_return_before_any_launch(lib):
    L = lib.LIB
    plan = lib.make_plan()
    # null tensors
    assert L.adahop_linear_fwd(C.byref(plan), None, None, 128, 128, 128, None, 0, None, 0, None) == 1
    # misaligned pointers are rejected before the device is queried
    assert L.adahop_linear_fwd(C.byref(plan), 0x1001, 0x2000, 128, 128, 128, 0x3000, 0, 0x4000, 1 << 20, None) == 3
    # bad output dtype
    assert L.adahop_linear_fwd(C.byref(plan), 0x1000, 0x2000, 128, 128, 128, 0x3000, 7, 0x4000, 1 << 20, None) == 1
    # bad shapes and a too-small workspace are caught before any device query
    assert L.adahop_linear_fwd(C.byref(plan), 0x1000, 0x2000, 100, 128, 128, 0x3000, 0, 0x4000, 1 << 20, None) == 2
    assert L.adahop_linear_fwd(C.byref(plan), 0x1000, 0x2000, 128, 128, 128, 0x3000, 0, 0x4000, 16, None) == 7
    assert L.adahop_linear_bwd(C.byref(plan), 0x1000, 0x2000, 0x3000, 128, 128, 128, None, None, 0, 0x4000, 0,
                               None) == 1
    assert L.adahop_quantize_mxfp4(0x1000, 100, 128, 1, 1, None, None, 0x2000, 0x3000, 0, None) == 2
    assert L.adahop_quantize_mxfp4(0x1000, 128, 128, 2, 1, None, None, 0x2000, 0x3000, 0, None) == 1
    assert L.adahop_foid(0x1000, 128, 128, 0, 300, 0x2000, None, 0x3000, 1 << 20, None) == 2
    assert L.adahop_gemm_bf16(0x1000, 1, 0x2000, 1, 128, 100, 128, 0x3000, 1, 1, None, 0x4000, 4096, None) == 2
    assert L.adahop_gemm_mxfp4(0x1000, 0x1000, 0x1000, 0x1000, 128, 128, 128, None, None, 16, 0x2000, 1, 0x3000,
                               4096, None) == 2
    assert L.adahop_scatter_add(None, 1, 1, 0, None, 1, None, 0, 0, None) == 1
    assert L.adahop_calibrate(None, None, None, 128, 128, 128, None, None, None, 0, None) == 1
    # the failure-path probe checks its workspace on the host (7 = workspace, 3 = alignment)
    assert L.adahop_check_bounded_wait(None, 256, None) == 7
    assert L.adahop_check_bounded_wait(0x1010, 256, None) == 3
    assert L.adahop_check_bounded_wait(0x1000, 128, None) == 7


def test_python_binding_names_match_c(lib):
    import quantized_gemm_foid_gb300.binding as b
    for name in lib.PROTOTYPES:
        if name in ("adahop_status_string", "adahop_last_cuda_error"):
            continue
        assert callable(getattr(b, name)), name


def test_saved_size_layout(lib):
    q = lib
    IHT, BF16 = 0, 3
    M, N, K = 512, 256, 384
    a = lambda v: (v + 255) // 256 * 256
    full = a(K * M // 2) + a(K * M // 32) + a(K * N // 2) + a(K * N // 32)
    assert q.adahop_saved_size(q.make_plan(fwd=IHT, dgrad=IHT, wgrad=IHT), M, N, K) == full
    assert q.adahop_saved_size(q.make_plan(dgrad=BF16, wgrad=IHT), M, N, K) == a(K * M // 2) + a(K * M // 32)
    assert q.adahop_saved_size(q.make_plan(dgrad=BF16, wgrad=BF16), M, N, K) == 0
    # compression of the saved activation against its bf16 copy: 2 / (1/2 + 1/32) bytes per element
    x_part = a(K * M // 2) + a(K * M // 32)
    assert 2 * M * K / x_part == pytest.approx(2 / (0.5 + 1 / 32), rel=1e-3)


def test_product_package_never_touches_the_oracle():
    """The oracle is test infrastructure: nothing in the product package or its CUDA sources
    imports, includes or names it, so no product call can route through it."""
    pkg = os.path.join(ROOT, "quantized_gemm_foid_gb300")
    offenders = []
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath or "__pycache__" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                if re.search(r"^\s*(import|from)\s+oracle\b|#\s*include\s*[<\"][^>\"]*oracle", text, flags=re.M):
                    offenders.append(os.path.join(dirpath, f))
    assert not offenders, offenders


def test_missing_library_raises_instead_of_falling_back(lib, tmp_path):
    from quantized_gemm_foid_gb300 import _lib
    with pytest.raises(ImportError):
        _lib.load_library(str(tmp_path / "libadahop.so"))

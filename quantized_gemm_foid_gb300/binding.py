"""Thin Python binding of the C ABI in include/adahop.h.

Every function has the name of the C entry point it calls and only marshals arguments: shapes
from the tensors, raw device pointers, the current CUDA stream.  All arithmetic runs in
libadahop.so's sm_103a kernels.  Tensors are torch tensors on the CUDA device (bf16 tensors are
passed as their 16-bit patterns); the library allocates nothing, so callers pass outputs and a
workspace (see ``new_workspace``).
"""
from __future__ import annotations

import ctypes as C

import torch

from ._lib import LIB, AdahopOptions, AdahopPlan

PAT_NONE, PAT_ROW, PAT_COL = 0, 1, 2
IHT, OE_LEFT, OE_RIGHT, BF16, MXFP4 = 0, 1, 2, 3, 4
OUT_BF16, OUT_FP32 = 0, 1
STRATEGY_NAMES = {IHT: "IHT", OE_LEFT: "OE-Left", OE_RIGHT: "OE-Right", BF16: "BF16", MXFP4: "MXFP4"}
PATTERN_NAMES = {PAT_NONE: "None", PAT_ROW: "Row-wise", PAT_COL: "Column-wise"}


class AdahopError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = LIB.adahop_status_string(status).decode()
        detail = LIB.adahop_last_cuda_error().decode()
        super().__init__(f"{what}: {msg}" + (f" ({detail})" if status == 4 and detail else ""))
        self.status = status


def _check(status: int, what: str) -> None:
    if status != 0:
        raise AdahopError(status, what)


def _p(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _out_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return OUT_BF16
    if t.dtype == torch.float32:
        return OUT_FP32
    raise TypeError("outputs must be bfloat16 or float32")


def _cuda(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}")
    return t


def make_plan(x=PAT_NONE, w=PAT_NONE, gy=PAT_NONE, fwd=IHT, dgrad=IHT, wgrad=IHT, oe_rank=64) -> AdahopPlan:
    p = AdahopPlan()
    p.x, p.w, p.gy, p.fwd, p.dgrad, p.wgrad, p.oe_rank = x, w, gy, fwd, dgrad, wgrad, oe_rank
    return p


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed uint8 device buffer (the status word must start at zero)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def adahop_default_options() -> AdahopOptions:
    o = AdahopOptions()
    LIB.adahop_default_options(C.byref(o))
    return o


def adahop_workspace_size(plan: AdahopPlan, M: int, N: int, K: int) -> int:
    n = C.c_size_t(0)
    _check(LIB.adahop_workspace_size(C.byref(plan), M, N, K, C.byref(n)), "adahop_workspace_size")
    return n.value


def adahop_calibrate(X, W, GY, workspace, opts: AdahopOptions | None = None, stream=None) -> AdahopPlan:
    _cuda(X, "X", torch.bfloat16)
    _cuda(W, "W", torch.bfloat16)
    if GY is not None:
        _cuda(GY, "GY", torch.bfloat16)
    M, K = X.shape
    N = W.shape[0]
    plan = AdahopPlan()
    _check(LIB.adahop_calibrate(_p(X), _p(W), _p(GY), M, N, K,
                                C.byref(opts) if opts is not None else None, C.byref(plan),
                                _p(workspace), workspace.numel(), _stream(stream)), "adahop_calibrate")
    return plan


def adahop_linear_fwd(plan: AdahopPlan, X, W, Y, workspace, stream=None) -> None:
    _cuda(X, "X", torch.bfloat16)
    _cuda(W, "W", torch.bfloat16)
    _cuda(Y, "Y")
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(Y.shape) != (M, N):
        raise ValueError("shape mismatch: X (M,K), W (N,K), Y (M,N)")
    _check(LIB.adahop_linear_fwd(C.byref(plan), _p(X), _p(W), M, N, K, _p(Y), _out_dtype(Y),
                                 _p(workspace), workspace.numel(), _stream(stream)), "adahop_linear_fwd")


def adahop_saved_size(plan: AdahopPlan, M: int, N: int, K: int) -> int:
    out = C.c_size_t(0)
    _check(LIB.adahop_saved_size(C.byref(plan), M, N, K, C.byref(out)), "adahop_saved_size")
    return out.value


def new_saved(plan: AdahopPlan, M: int, N: int, K: int, device="cuda") -> torch.Tensor:
    """A device buffer of adahop_saved_size bytes (uint8) for one layer's saved context."""
    return torch.empty(max(adahop_saved_size(plan, M, N, K), 256), dtype=torch.uint8, device=device)


def adahop_linear_fwd_save(plan: AdahopPlan, X, W, Y, saved, workspace, stream=None) -> None:
    _cuda(X, "X", torch.bfloat16)
    _cuda(W, "W", torch.bfloat16)
    _cuda(Y, "Y")
    _cuda(saved, "saved", torch.uint8)
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(Y.shape) != (M, N):
        raise ValueError("shape mismatch: X (M,K), W (N,K), Y (M,N)")
    _check(LIB.adahop_linear_fwd_save(C.byref(plan), _p(X), _p(W), M, N, K, _p(Y), _out_dtype(Y), _p(saved),
                                      saved.numel(), _p(workspace), workspace.numel(), _stream(stream)),
           "adahop_linear_fwd_save")


def _bwd_outputs(GY, X, W, dX, dW):
    _cuda(GY, "GY", torch.bfloat16)
    _cuda(X, "X", torch.bfloat16)
    _cuda(W, "W", torch.bfloat16)
    M, K = X.shape
    N = W.shape[0]
    if tuple(GY.shape) != (M, N):
        raise ValueError("GY must be M x N")
    outs = [t for t in (dX, dW) if t is not None]
    if not outs:
        raise ValueError("at least one of dX, dW")
    dt = _out_dtype(outs[0])
    if any(_out_dtype(t) != dt for t in outs):
        raise TypeError("dX and dW must share a dtype")
    if dX is not None and tuple(dX.shape) != (M, K):
        raise ValueError("dX must be M x K")
    if dW is not None and tuple(dW.shape) != (N, K):
        raise ValueError("dW must be N x K")
    return M, N, K, dt


def adahop_linear_bwd_saved(plan: AdahopPlan, GY, X, W, saved, dX, dW, workspace, stream=None) -> None:
    _cuda(saved, "saved", torch.uint8)
    M, N, K, dt = _bwd_outputs(GY, X, W, dX, dW)
    _check(LIB.adahop_linear_bwd_saved(C.byref(plan), _p(GY), _p(X), _p(W), _p(saved), saved.numel(), M, N, K,
                                       _p(dX), _p(dW), dt, _p(workspace), workspace.numel(), _stream(stream)),
           "adahop_linear_bwd_saved")


def adahop_linear_bwd(plan: AdahopPlan, GY, X, W, dX, dW, workspace, stream=None) -> None:
    _cuda(GY, "GY", torch.bfloat16)
    _cuda(X, "X", torch.bfloat16)
    _cuda(W, "W", torch.bfloat16)
    M, K = X.shape
    N = W.shape[0]
    if tuple(GY.shape) != (M, N):
        raise ValueError("GY must be M x N")
    outs = [t for t in (dX, dW) if t is not None]
    if not outs:
        raise ValueError("at least one of dX, dW")
    dt = _out_dtype(outs[0])
    if any(_out_dtype(t) != dt for t in outs):
        raise TypeError("dX and dW must share a dtype")
    if dX is not None and tuple(dX.shape) != (M, K):
        raise ValueError("dX must be M x K")
    if dW is not None and tuple(dW.shape) != (N, K):
        raise ValueError("dW must be N x K")
    _check(LIB.adahop_linear_bwd(C.byref(plan), _p(GY), _p(X), _p(W), M, N, K, _p(dX), _p(dW), dt,
                                 _p(workspace), workspace.numel(), _stream(stream)), "adahop_linear_bwd")


def adahop_get_device_status(workspace, stream=None) -> int:
    return LIB.adahop_get_device_status(_p(workspace), _stream(stream))


def adahop_check_bounded_wait(workspace, stream=None) -> None:
    """Launches the failure-path probe: a later adahop_get_device_status(workspace) returns
    ADAHOP_ERR_TIMEOUT once its bounded wait (2 s) has run out."""
    _check(LIB.adahop_check_bounded_wait(_p(workspace), workspace.numel(), _stream(stream)),
           "adahop_check_bounded_wait")


def adahop_foid_workspace_size(lines: int, r: int) -> int:
    return LIB.adahop_foid_workspace_size(lines, r)


def adahop_foid(T, axis: int, r: int, idx_out, mask_out, workspace, stream=None) -> None:
    _cuda(T, "T", torch.bfloat16)
    rows, cols = T.shape
    _check(LIB.adahop_foid(_p(T), rows, cols, axis, r, _p(idx_out), _p(mask_out), _p(workspace),
                           workspace.numel(), _stream(stream)), "adahop_foid")


def adahop_foid_noalloc(T, axis: int, r: int, idx_out, mask_out, stream=None) -> None:
    """FOID for callers that cannot allocate: the library keeps the scratch in a fixed device
    array (up to ceil(lines / 2048) * r = 8192 candidates); concurrent calls race on it."""
    _cuda(T, "T", torch.bfloat16)
    rows, cols = T.shape
    _check(LIB.adahop_foid_noalloc(_p(T), rows, cols, axis, r, _p(idx_out), _p(mask_out), _stream(stream)),
           "adahop_foid_noalloc")


def adahop_quantize_mxfp4(T, inner_axis: int, hadamard: int, zero_rows_mask, zero_cols_mask, codes,
                          scales, scale_layout: int = 0, stream=None) -> None:
    _cuda(T, "T", torch.bfloat16)
    rows, cols = T.shape
    _check(LIB.adahop_quantize_mxfp4(_p(T), rows, cols, inner_axis, hadamard, _p(zero_rows_mask),
                                     _p(zero_cols_mask), _p(codes), _p(scales), scale_layout,
                                     _stream(stream)), "adahop_quantize_mxfp4")


def adahop_quantize_mxfp4_dual(T, hadamard: int, zero_rows_mask, zero_cols_mask, codes_rows, scales_rows,
                               codes_cols, scales_cols, scale_layout: int = 0, stream=None) -> None:
    _cuda(T, "T", torch.bfloat16)
    rows, cols = T.shape
    _check(LIB.adahop_quantize_mxfp4_dual(_p(T), rows, cols, hadamard, _p(zero_rows_mask), _p(zero_cols_mask),
                                          _p(codes_rows), _p(scales_rows), _p(codes_cols), _p(scales_cols),
                                          scale_layout, _stream(stream)), "adahop_quantize_mxfp4_dual")


def adahop_gather(T, idx, r: int, mode: int, out, stream=None) -> None:
    _cuda(T, "T", torch.bfloat16)
    rows, cols = T.shape
    _check(LIB.adahop_gather(_p(T), rows, cols, _p(idx), r, mode, _p(out), _stream(stream)), "adahop_gather")


def adahop_gemm_mxfp4(a_codes, a_scales, b_codes, b_scales, P: int, Q: int, J: int, A_o, B_o, r: int, C_out,
                      workspace, stream=None) -> None:
    _check(LIB.adahop_gemm_mxfp4(_p(a_codes), _p(a_scales), _p(b_codes), _p(b_scales), P, Q, J, _p(A_o),
                                 _p(B_o), r, _p(C_out), _out_dtype(C_out), _p(workspace), workspace.numel(),
                                 _stream(stream)), "adahop_gemm_mxfp4")


def adahop_gemm_mxfp4_workspace_size() -> int:
    return int(LIB.adahop_gemm_mxfp4_workspace_size())


def adahop_gemm_bf16(A, a_kmajor: int, B, b_kmajor: int, P: int, Q: int, J: int, C_out, workspace,
                     splits: int = 1, c_partial=None, out_dtype: int | None = None, stream=None) -> None:
    od = _out_dtype(C_out) if C_out is not None else (OUT_FP32 if out_dtype is None else out_dtype)
    _check(LIB.adahop_gemm_bf16(_p(A), a_kmajor, _p(B), b_kmajor, P, Q, J, _p(C_out), od, splits,
                                _p(c_partial), _p(workspace), workspace.numel(), _stream(stream)),
           "adahop_gemm_bf16")


def adahop_gemm_bf16_scatter_add(A, a_kmajor: int, B, b_kmajor: int, P: int, Q: int, J: int, C_out, idx,
                                 r: int, axis: int, workspace, stream=None) -> None:
    c_rows, c_cols = C_out.shape
    _check(LIB.adahop_gemm_bf16_scatter_add(_p(A), a_kmajor, _p(B), b_kmajor, P, Q, J, _p(C_out), c_rows, c_cols,
                                            _out_dtype(C_out), _p(idx), r, axis, _p(workspace), workspace.numel(),
                                            _stream(stream)), "adahop_gemm_bf16_scatter_add")


def adahop_scatter_add(C_out, partial, splits: int, idx, r: int, axis: int, stream=None) -> None:
    P, Q = C_out.shape
    _check(LIB.adahop_scatter_add(_p(C_out), P, Q, _out_dtype(C_out), _p(partial), splits, _p(idx), r, axis,
                                  _stream(stream)), "adahop_scatter_add")


def adahop_calibration_stats(T, row_ms, col_ms, stream=None) -> None:
    _cuda(T, "T", torch.bfloat16)
    rows, cols = T.shape
    _check(LIB.adahop_calibration_stats(_p(T), rows, cols, _p(row_ms), _p(col_ms), _stream(stream)),
           "adahop_calibration_stats")


# ------------------------------------------------------------------------------- peak probes (K8)
MMA_KIND_NAMES = {0: "kind::f16", 1: "kind::mxf4 (2X)", 2: "kind::mxf4nvf4 (2X)", 3: "kind::mxf4nvf4 (4X)"}
MMA_K_PER_INSTR = {0: 16, 1: 64, 2: 64, 3: 64}


def adahop_probe_ctas() -> int:
    return int(LIB.adahop_probe_ctas())


def adahop_probe_mma_rate(kind: int, sf_copies: int, iters: int, out, ws, stream=None, n: int = 256) -> None:
    """Launches the tensor-pipe rate probe (MMA width n = 128 or 256); `out` is a uint64 (int64)
    device tensor of at least 3 * adahop_probe_ctas() entries (per CTA: loop cycles, start ns, end ns)."""
    _cuda(out, "out")
    _check(LIB.adahop_probe_mma_rate(int(kind), int(sf_copies), int(n), int(iters), _p(out),
                                     out.numel() * out.element_size(), _p(ws), ws.numel(), _stream(stream)),
           "adahop_probe_mma_rate")


def adahop_probe_copy(src, dst, stream=None) -> None:
    """src None: the write-only fill of all of dst."""
    _cuda(dst, "dst")
    if src is None:
        nbytes = dst.numel() * dst.element_size()
    else:
        _cuda(src, "src")
        nbytes = src.numel() * src.element_size()
        if dst.numel() * dst.element_size() < nbytes:
            raise ValueError("dst is smaller than src")
    _check(LIB.adahop_probe_copy(_p(src), _p(dst), nbytes, _stream(stream)), "adahop_probe_copy")

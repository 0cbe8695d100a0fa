"""ctypes loader for libadahop.so and the prototypes of every entry point in include/adahop.h.

Importing this module fails loudly if the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

from .build import LIB_PATH

c_int64, c_int, c_size_t, c_void_p = C.c_int64, C.c_int, C.c_size_t, C.c_void_p


class AdahopOptions(C.Structure):
    _fields_ = [("tau", C.c_double), ("probe_len", c_int), ("oe_rank", c_int)]


class AdahopPlan(C.Structure):
    _fields_ = [("x", C.c_int32), ("w", C.c_int32), ("gy", C.c_int32),
                ("fwd", C.c_int32), ("dgrad", C.c_int32), ("wgrad", C.c_int32),
                ("oe_rank", C.c_int32), ("reserved", C.c_int32), ("rho", C.c_double * 6)]

    def as_dict(self) -> dict:
        return {"x": self.x, "w": self.w, "gy": self.gy, "fwd": self.fwd, "dgrad": self.dgrad,
                "wgrad": self.wgrad, "oe_rank": self.oe_rank, "rho": list(self.rho)}


# name -> (restype, argtypes); the single source of the binding's view of the C ABI
PROTOTYPES = {
    "adahop_default_options": (None, [C.POINTER(AdahopOptions)]),
    "adahop_status_string": (C.c_char_p, [c_int]),
    "adahop_last_cuda_error": (C.c_char_p, []),
    "adahop_workspace_size": (c_int, [C.POINTER(AdahopPlan), c_int64, c_int64, c_int64,
                                      C.POINTER(c_size_t)]),
    "adahop_calibrate": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64,
                                 C.POINTER(AdahopOptions), C.POINTER(AdahopPlan), c_void_p,
                                 c_size_t, c_void_p]),
    "adahop_linear_fwd": (c_int, [C.POINTER(AdahopPlan), c_void_p, c_void_p, c_int64, c_int64,
                                  c_int64, c_void_p, c_int, c_void_p, c_size_t, c_void_p]),
    "adahop_linear_bwd": (c_int, [C.POINTER(AdahopPlan), c_void_p, c_void_p, c_void_p, c_int64,
                                  c_int64, c_int64, c_void_p, c_void_p, c_int, c_void_p, c_size_t,
                                  c_void_p]),
    "adahop_saved_size": (c_int, [C.POINTER(AdahopPlan), c_int64, c_int64, c_int64,
                                  C.POINTER(c_size_t)]),
    "adahop_linear_fwd_save": (c_int, [C.POINTER(AdahopPlan), c_void_p, c_void_p, c_int64, c_int64,
                                       c_int64, c_void_p, c_int, c_void_p, c_size_t, c_void_p,
                                       c_size_t, c_void_p]),
    "adahop_linear_bwd_saved": (c_int, [C.POINTER(AdahopPlan), c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_size_t, c_int64, c_int64, c_int64, c_void_p,
                                        c_void_p, c_int, c_void_p, c_size_t, c_void_p]),
    "adahop_get_device_status": (c_int, [c_void_p, c_void_p]),
    "adahop_check_bounded_wait": (c_int, [c_void_p, c_size_t, c_void_p]),
    "adahop_foid": (c_int, [c_void_p, c_int64, c_int64, c_int, c_int, c_void_p, c_void_p,
                            c_void_p, c_size_t, c_void_p]),
    "adahop_foid_workspace_size": (c_size_t, [c_int64, c_int]),
    "adahop_foid_noalloc": (c_int, [c_void_p, c_int64, c_int64, c_int, c_int, c_void_p, c_void_p,
                                    c_void_p]),
    "adahop_quantize_mxfp4": (c_int, [c_void_p, c_int64, c_int64, c_int, c_int, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "adahop_quantize_mxfp4_dual": (c_int, [c_void_p, c_int64, c_int64, c_int, c_void_p, c_void_p,
                                           c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "adahop_gather": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_int, c_int, c_void_p,
                              c_void_p]),
    "adahop_gemm_mxfp4": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64,
                                  c_int64, c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p,
                                  c_size_t, c_void_p]),
    "adahop_gemm_mxfp4_workspace_size": (c_size_t, []),
    "adahop_gemm_bf16": (c_int, [c_void_p, c_int, c_void_p, c_int, c_int64, c_int64, c_int64,
                                 c_void_p, c_int, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "adahop_gemm_bf16_scatter_add": (c_int, [c_void_p, c_int, c_void_p, c_int, c_int64, c_int64, c_int64,
                                             c_void_p, c_int64, c_int64, c_int, c_void_p, c_int, c_int,
                                             c_void_p, c_size_t, c_void_p]),
    "adahop_scatter_add": (c_int, [c_void_p, c_int64, c_int64, c_int, c_void_p, c_int, c_void_p,
                                   c_int, c_int, c_void_p]),
    "adahop_calibration_stats": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_void_p,
                                         c_void_p]),
    "adahop_probe_ctas": (c_int, []),
    "adahop_probe_mma_rate": (c_int, [c_int, c_int, c_int, c_int64, c_void_p, c_size_t, c_void_p, c_size_t,
                                      c_void_p]),
    "adahop_probe_copy": (c_int, [c_void_p, c_void_p, c_size_t, c_void_p]),
}


def load_library(path: str = LIB_PATH) -> C.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -m quantized_gemm_foid_gb300.build, or __graft_entry__.build())")
    lib = C.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(lib, name)          # AttributeError if the library lacks an entry point
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = load_library()

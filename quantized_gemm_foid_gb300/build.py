"""Builds the sm_103a shared library (libadahop.so) in-tree with nvcc.

Each CUDA translation unit is compiled in parallel, then linked into one shared object with a
C ABI (include/adahop.h).  No PyTorch headers are involved: the library is plain CUDA C++.

    python -m quantized_gemm_foid_gb300.build        # or build() from Python
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libadahop.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)

SOURCES = ["adahop.cu", "quant.cu", "foid.cu", "misc.cu", "gemm.cu", "probe.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libadahop.so")


def _compile(nvcc: str, src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH_FLAGS, *COMMON_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    return obj


def _up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    deps = [os.path.join(CSRC, s) for s in SOURCES]
    deps += [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith(".cuh")]
    deps.append(os.path.join(ROOT, "include", "adahop.h"))
    lib_mtime = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) < lib_mtime for d in deps)


def build(verbose: bool = False, extra_flags: list[str] | None = None, force: bool = False) -> str:
    """Compile every kernel for sm_103a and link libadahop.so; returns the library path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and not extra_flags and _up_to_date():
        return LIB_PATH
    nvcc = nvcc_path()
    extra = list(extra_flags or [])
    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, extra), SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(f"built {LIB_PATH}")
    return LIB_PATH


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv)

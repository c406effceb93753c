"""Build the in-tree C-ABI library ``_build/libvaedec.so`` with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel, then linked into one shared
library (CUDA runtime linked statically; the driver API entry point for tensor
maps is resolved at run time).  Run ``python -m row_band_layerwise_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libvaedec.so"
SOURCES = ["api.cu", "conv_tc.cu", "conv_halo.cu", "conv_halo_t.cu", "conv_narrow.cu", "conv_simple.cu", "norm.cu", "attn.cu", "attn_flash.cu", "gemm_cm.cu", "gn_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def lib_path() -> str:
    return os.path.join(OUT_DIR, LIB_NAME)


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
           "--expt-relaxed-constexpr", "-I", os.path.join(HERE, "..", "include"), "-I", CSRC,
           *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile every source and link the shared library; returns its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    extra = list(extra or [])
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = lib_path() + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path())
    if verbose:
        print("built", lib_path())
    return lib_path()


if __name__ == "__main__":
    build(verbose=True, extra=sys.argv[1:])

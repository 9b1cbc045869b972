"""Build the native library libcac.so in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel into _build/, then one link step
writes cache_aware_conformer_gb300/libcac.so.  No cmake, no torch extension
machinery; the CUDA runtime is linked statically so the library loads in any
process that has the NVIDIA driver.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libcac.so")
SOURCES = ["gemm_tc.cu", "gemm_tc_persist.cu", "gemm_simt.cu", "kernels.cu", "attn_mma.cu", "engine.cu", "decode.cu", "frontend.cu", "beam.cu", "gemm_palette.cu", "chain.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")


def _compile(src: str, extra: list[str], objdir: str = BUILD) -> str:
    obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


LIB_CHECKED = os.path.join(PKG, "libcac_checked.so")


def build(extra: list[str] | None = None, verbose: bool = False, checked: bool = False) -> str:
    """checked=True: the CAC_CHECKED variant (index checks in the step's
    kernels) as libcac_checked.so, selected at run time with CAC_LIB=checked."""
    objdir = os.path.join(BUILD, "checked") if checked else BUILD
    lib = LIB_CHECKED if checked else LIB
    os.makedirs(objdir, exist_ok=True)
    extra = list(extra or []) + (["-DCAC_CHECKED"] if checked else [])
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, objdir), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print("built", lib)
    return lib


if __name__ == "__main__":
    args = sys.argv[1:]
    build([a for a in args if a != "--checked"], verbose=True, checked="--checked" in args)

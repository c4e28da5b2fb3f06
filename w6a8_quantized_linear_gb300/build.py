"""Build libqlin.so (sm_103a) in-tree with nvcc.

One translation unit, one -gencode, shared CUDA runtime (so the library and
PyTorch share one runtime and one notion of the current device).  The output
goes to ``w6a8_quantized_linear_gb300/_build/libqlin.so`` (git-ignored).
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libqlin.so")
SOURCES = [os.path.join(CSRC, f) for f in ("qlin_api.cu", "qlin_forward.cuh", "qlin_repack.cuh", "qlin_layout.h", "qlin_ptx.cuh")] + [
    os.path.join(INCLUDE, "qlin.h")]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    for cand in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in SOURCES)


def build_library(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = nvcc_path()
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared", "-Xlinker", f"-rpath,{cuda_lib}",
           "-I", INCLUDE, os.path.join(CSRC, "qlin_api.cu"), "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    if verbose:
        print(r.stdout + r.stderr)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))

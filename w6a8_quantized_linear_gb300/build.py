"""Build libqlin.so (sm_103a) in-tree with nvcc.

Eight translation units compiled in parallel (the host API with the repack
kernels, and seven sets of forward-kernel variants), one
-gencode, shared CUDA runtime (so the library and PyTorch share one runtime
and one notion of the current device).  The output goes to
``w6a8_quantized_linear_gb300/_build/libqlin.so`` (git-ignored).
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
UNITS = ["qlin_api.cu", "qlin_kernels_w4.cu", "qlin_kernels_w6.cu", "qlin_kernels_codebook.cu",
         "qlin_kernels_moe_w4.cu", "qlin_kernels_moe_w6.cu", "qlin_kernels_export_w4.cu", "qlin_kernels_export_w6.cu",
         "qlin_kernels_tc.cu", "qlin_kernels_tc_export.cu", "qlin_kernels_w4_one_row.cu", "qlin_kernels_w6_one_row.cu",
         "qlin_kernels_moe_one_row.cu", "qlin_kernels_codebook_one_row.cu"]
SOURCES = [os.path.join(CSRC, f) for f in UNITS + ["qlin_forward.cuh", "qlin_forward_tc.cuh", "qlin_repack.cuh", "qlin_layout.h",
                                                   "qlin_ptx.cuh", "qlin_instances.h"]] + [
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
    tag = f".tmp{os.getpid()}"
    # kernels are instantiated in one unit and launched from another, so their
    # host stubs need external linkage
    common = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-static-global-template-stub=false", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    if verbose:
        common.insert(1, "-Xptxas=-v")
    objs, procs = [], []
    try:
        return _compile_and_link(nvcc, cuda_lib, common, tag, verbose)
    finally:
        for f in os.listdir(BUILD):  # objects of this build, also after a failure
            if f.endswith(tag + ".o"):
                os.remove(os.path.join(BUILD, f))


def _compile_and_link(nvcc, cuda_lib, common, tag, verbose):
    objs, procs = [], []
    for u in UNITS:
        obj = os.path.join(BUILD, u.replace(".cu", tag + ".o"))
        cmd = common + ["-c", os.path.join(CSRC, u), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    logs = []
    for cmd, pr in procs:
        out, _ = pr.communicate()
        logs.append(out)
        if pr.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + out)
    tmp = LIB + tag
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-cudart", "shared", "-Xlinker",
           f"-rpath,{cuda_lib}"] + objs + ["-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    if verbose:
        print("".join(logs) + r.stdout + r.stderr)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))

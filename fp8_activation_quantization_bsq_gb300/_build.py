"""Compile libbsq (the CUDA kernels + C ABI) in-tree for sm_103a with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_DIR, "include")
LIB_DIR = os.path.join(PKG_DIR, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libbsq.so")

SOURCES = ["bsq.cu"]
HEADERS = ["device_common.cuh", "box_quant.cuh", "dense_quant.cuh", "grouped_quant.cuh", "interleave.cuh",
           "tensor_scale.cuh", "block_scaled_dot.cuh", "cluster.cuh", "gemm_quant.cuh", "grouped_token.cuh"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libbsq")


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS]
            + [os.path.join(INCLUDE, "bsq.h"), os.path.abspath(__file__)])


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Build ``_lib/libbsq.so`` (skipped when up to date); returns its path."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc_path(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
           "-std=c++17", "-Werror", "all-warnings", "-shared", "-cudart", "shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
           "-Xlinker", "-rpath,/usr/local/cuda/lib64", "-I", INCLUDE, "-o", tmp]
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        print(" ".join(cmd))
        print(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError("libbsq build failed:\n" + res.stderr[-4000:])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

"""Build the C-ABI library (libhs.so) in-tree with nvcc for sm_103a.

Each translation unit is compiled (one -gencode) in its own nvcc process, all at once, then linked against the
shared CUDA runtime so that the process shares one runtime with PyTorch. The output goes to
hierarchical_sparse_attention_hs_gb300/_build/ (git-ignored).
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SOURCES = [os.path.join(HERE, "csrc", "hs_resolve.cu"), os.path.join(HERE, "csrc", "hs_attention.cu")]
HEADERS = [os.path.join(ROOT, "include", "hs.h"), os.path.join(HERE, "csrc", "hs_block.cuh"),
           os.path.join(HERE, "csrc", "hs_pool.hpp")]
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libhs.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libhs.so")


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS + [os.path.abspath(__file__)])


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = nvcc_path()
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + f".{os.getpid()}.o")
        cmd = [nvcc, *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    failed = [p.args for p in procs if p.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        subprocess.check_call([nvcc, *ARCH_FLAGS, "-shared", "-cudart", "shared", f"-Xlinker=-rpath={cuda_lib}",
                               "-o", tmp, *objs])
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

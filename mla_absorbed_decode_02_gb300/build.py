"""Build step for libmla_decode.so (nvcc, sm_103a only, in-tree)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "mla_decode.cu")
LIB = os.path.join(PKG, "libmla_decode.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc")


def _sources():
    d = os.path.join(PKG, "csrc")
    return [os.path.join(d, f) for f in os.listdir(d)] + [os.path.join(ROOT, "include", "mla_decode.h")]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library if any source is newer than the .so; returns its path."""
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in _sources())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
           "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-o", tmp, SRC]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

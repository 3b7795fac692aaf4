"""Build the CUDA library ``libnomas.so`` in-tree with nvcc for sm_103a.

Usage: ``python segment_causal_kv_int8_b300/_build.py [-v]`` (run by path, so
that building never imports the package, which loads the library).  The library
links the CUDA runtime statically and resolves the driver's tensor-map encoder
at run time, so loading it needs no GPU driver.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libnomas.so")
SOURCES = ["nomas_abi.cu", "rope3d.cu", "kvcache_append.cu", "segment_attn.cu", "sparse_select.cu", "camera_attn.cu", "selftest.cu"]
HEADERS = ["kernels.h", "sm100.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "nomas.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra=None) -> str:
    if not force and up_to_date():
        return LIB
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-cudart", "static", "-I", os.path.join(ROOT, "include"),
           "-Xptxas", "-v" if verbose else "-O3", *(extra or []),
           *[os.path.join(CSRC, f) for f in SOURCES], "-o", LIB + ".tmp"]
    res = subprocess.run(cmd, cwd=CSRC, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)

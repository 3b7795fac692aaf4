"""Build the CUDA libraries in-tree with nvcc for sm_103a.

``libnomas.so`` is the library; ``libnomas_checked.so`` is the same sources
compiled with ``-DNOMAS_BOUNDS_CHECK``, where every computed global-memory index
is range-checked and a bad one is recorded in the device error word
(NOMAS_ERR_INVALID_ARG) and its access skipped.  The package loads the checked
one when ``NOMAS_LIBRARY=checked`` is set in the environment.

Usage: ``python segment_causal_kv_int8_b300/_build.py [-v]`` (run by path, so
that building never imports the package, which loads the library).  The
libraries link the CUDA runtime statically and resolve the driver's tensor-map
encoder at run time, so loading them needs no GPU driver.
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
LIB_CHECKED = os.path.join(PKG, "libnomas_checked.so")
SOURCES = ["nomas_abi.cu", "rope3d.cu", "kvcache_append.cu", "segment_attn.cu", "sparse_select.cu",
           "camera_attn.cu", "selftest.cu"]
HEADERS = ["kernels.h", "sm100.cuh", "checks.cuh", "rope_math.cuh", "attn_common.cuh"]
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


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(lib: str, verbose: bool, extra) -> None:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-cudart", "static", "-I", os.path.join(ROOT, "include"),
           "-Xptxas", "-v" if verbose else "-O3", *(extra or []),
           *[os.path.join(CSRC, f) for f in SOURCES], "-o", lib + ".tmp"]
    res = subprocess.run(cmd, cwd=CSRC, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(lib + ".tmp", lib)


def build(force: bool = False, verbose: bool = False, extra=None, checked: bool = True) -> str:
    """Build libnomas.so (and, with ``checked``, libnomas_checked.so) unless up to date."""
    if force or not up_to_date(LIB):
        _compile(LIB, verbose, extra)
    if checked and (force or not up_to_date(LIB_CHECKED)):
        _compile(LIB_CHECKED, False, list(extra or []) + ["-DNOMAS_BOUNDS_CHECK"])
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)
    print(LIB_CHECKED)

"""Build the in-tree CUDA library libgemm_tn.so for sm_103a with nvcc.

One translation unit (csrc/gemm_tn.cu plus its headers), one -gencode,
static CUDA runtime; the driver API is reached through the runtime's entry
point query, so nothing links against libcuda.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libgemm_tn.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(ROOT, "include", "*.h")))


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libgemm_tn.so")


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile libgemm_tn.so in-tree if missing or older than its sources."""
    if not force and not is_stale():
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), "-O3", "-std=c++17", ARCH, "-lineinfo",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           "-shared", "-I", os.path.join(ROOT, "include"),
           os.path.join(CSRC, "gemm_tn.cu"), "-o", tmp]
    if ptxas_info:
        cmd.insert(1, "-Xptxas=-v")
    if verbose:
        print(" ".join(cmd))
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose or ptxas_info:
        print(r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv))

"""Build ``libbeamboundary.so`` in-tree with nvcc for sm_103a (no GPU needed).

The library links the CUDA runtime dynamically so that it shares the runtime
(current device, primary context) of the process that loads it, e.g. PyTorch.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libbeamboundary.so")
SOURCES = [os.path.join(CSRC, "beam_boundary.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + [
    os.path.join(INCLUDE, "beam_boundary.h")]

ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libbeamboundary")
    return p


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")


def flags(verbose: bool = False) -> list[str]:
    f = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-prec-div=true", "-prec-sqrt=true",
         "-ftz=false", f"-I{INCLUDE}", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-shared",
         "-cudart", "shared", f"-Xlinker=-rpath,{cuda_lib_dir()}"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    tmp = f"{LIB}.{os.getpid()}.tmp"
    cmd = [nvcc()] + flags(verbose) + SOURCES + ["-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed building libbeamboundary.so")
    if verbose:
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

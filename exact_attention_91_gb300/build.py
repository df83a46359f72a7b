"""Builds libfa.so in-tree with nvcc for sm_103a.

The library is one translation unit (``csrc/fa_api.cu``) that includes the
kernels; it links the CUDA runtime statically and resolves the driver's
tensor-map encoder at run time, so it needs no libcuda at link time.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libfa.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or cand)


def sources() -> list[str]:
    out = []
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh")):
            out.append(os.path.join(CSRC, name))
    out.append(os.path.join(INCLUDE, "fa.h"))
    return out


def nvcc_cmd(out_path: str, extra: list[str] | None = None) -> list[str]:
    return [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
            "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE, "-I", CSRC,
            *(extra or []), os.path.join(CSRC, "fa_api.cu"), "-o", out_path]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile libfa.so if any source is newer than it. Returns its path."""
    if not force and not extra and up_to_date():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = nvcc_cmd(tmp, (["-Xptxas", "-v"] if verbose else []) + (extra or []))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":  # pragma: no cover
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

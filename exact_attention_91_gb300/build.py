"""Builds libfa.so in-tree with nvcc for sm_103a.

The library is one translation unit (``csrc/fa_api.cu``) that includes the
kernels; it links the CUDA runtime statically and resolves the driver's
tensor-map encoder at run time, so it needs no libcuda at link time.
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys

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


# Kernels that split registers between warpgroups with setmaxnreg: the split
# in the source assumes this many registers per thread at launch (384 threads
# x 168). A different count would make setmaxnreg.inc wait for registers that
# never come, so the build refuses it.
LAUNCH_REGS = {"fa_fwd_kernel": 168}


def check_ptxas_report(report: str) -> dict[str, int]:
    """Parses `ptxas -v` output into {kernel: registers} and enforces LAUNCH_REGS."""
    regs, current = {}, None
    for line in report.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            regs[current] = int(m.group(1))
            current = None
    for name in LAUNCH_REGS:
        if not any(name in mangled for mangled in regs):
            raise RuntimeError(f"ptxas report lists no register count for {name}")
    for mangled, n in regs.items():
        for name, want in LAUNCH_REGS.items():
            if name in mangled and n != want:
                raise RuntimeError(f"{mangled}: ptxas allocated {n} registers per thread, the register "
                                   f"split assumes {want}")
    return regs


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile libfa.so if any source is newer than it. Returns its path."""
    if not force and not extra and up_to_date():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = nvcc_cmd(tmp, ["-Xptxas", "-v"] + (extra or []))
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise subprocess.CalledProcessError(res.returncode, cmd)
    try:
        check_ptxas_report(res.stdout + res.stderr)
    except RuntimeError:
        os.remove(tmp)
        raise
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

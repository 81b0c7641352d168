"""Build libsla.so (the C-ABI CUDA library) in place with nvcc for sm_103a.

    python -m sparse_iterative_linear_csr_b300.build [--verbose-ptxas]

The library is one translation unit (csrc/sla.cu) with the CUDA runtime
linked statically, so it loads next to PyTorch without sharing its runtime.
SLA_NVCC_EXTRA adds nvcc flags for tuning runs.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC_DIR = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libsla.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-shared", "--cudart", "static",
         "-I" + INCLUDE]


def sources() -> list[str]:
    return sorted(os.path.join(SRC_DIR, f) for f in os.listdir(SRC_DIR) if f.endswith((".cu", ".cuh")))


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + [os.path.join(INCLUDE, "sla.h")]
    return any(os.path.getmtime(s) > t for s in deps)


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    extra = os.environ.get("SLA_NVCC_EXTRA", "").split()
    cmd = [nvcc()] + ARCH + FLAGS + extra + (["-Xptxas", "-v"] if ptxas_verbose else []) + \
        ["-o", LIB + ".tmp", os.path.join(SRC_DIR, "sla.cu")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if ptxas_verbose:
        sys.stderr.write(res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, ptxas_verbose="--verbose-ptxas" in sys.argv))

"""Build the CUDA library ``_build/libtl_gemm.so`` for sm_103a with nvcc.

One translation unit (the host shim includes the kernel header), compiled with
``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``.  The library links the
CUDA runtime statically and reaches cuTensorMapEncodeTiled through the runtime's
driver entry-point query, so it needs no link against the driver library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libtl_gemm.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
SOURCES = ["tl_gemm.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build tl_gemm")
    return cand


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, d) for d in os.listdir(CSRC) if d.endswith((".cu", ".cuh"))] + [os.path.join(ROOT, "include", "tl_gemm.h"),
                                                     os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if any source is newer than it; return its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-I", os.path.join(ROOT, "include"), "-Xptxas", "-v",
           *[os.path.join(CSRC, s) for s in SOURCES], "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(BUILD_DIR, "ptxas.log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed building {LIB_NAME} (log: {log})")
    if verbose:
        sys.stdout.write(res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

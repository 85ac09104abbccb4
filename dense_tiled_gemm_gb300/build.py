"""Build the library in-tree: one nvcc invocation producing libdtgemm.so.

sm_103a only (``-gencode arch=compute_103a,code=sm_103a``). The CUDA runtime
is linked statically, so the .so needs only the NVIDIA driver at run time.
ptxas resource usage (registers, spills, shared memory) is written to
``_build/ptxas.log`` next to this file.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB_PATH = os.path.join(HERE, "libdtgemm.so")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = [os.path.join(HERE, "csrc", "gemm.cu"), os.path.join(HERE, "csrc", "attention.cu")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdtgemm.so")


def _inputs() -> list[str]:
    return (glob.glob(os.path.join(HERE, "csrc", "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    build_dir = os.path.join(HERE, "_build")
    os.makedirs(build_dir, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [_nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", "-cudart", "static", "-I", INCLUDE, "-o", tmp] + SOURCES
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(build_dir, "ptxas.log"), "w") as fh:
        fh.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stderr[-6000:]}")
    if verbose:
        print(res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

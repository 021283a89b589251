"""Builds libspecverify.so in-tree with nvcc for sm_103a (GB300)."""

from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
INCLUDE = os.path.join(ROOT, "include")
SOURCES = [os.path.join(PKG_DIR, "csrc", "specverify.cu")]
HEADERS = [os.path.join(INCLUDE, "specverify.h")]
LIB_PATH = os.path.join(PKG_DIR, "libspecverify.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile the CUDA library if a source or header is newer than it."""
    if not force and not _stale(LIB_PATH, SOURCES + HEADERS):
        return LIB_PATH
    nvcc = nvcc_path()
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE,
           "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
           "-Xlinker", f"-rpath,{cuda_lib}", *extra_flags, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

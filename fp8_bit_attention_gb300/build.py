"""Build libovc (the C ABI in include/ovc.h) in-tree for sm_103a with nvcc."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "ovc.cu")
HEADERS = [os.path.join(PKG, "csrc", f) for f in ("ptx.cuh", "prepare.cuh", "attention.cuh", "repair.cuh", "group.cuh",
                                                          "host_stream.cuh")]
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD_DIR, "libovc.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_command(out: str) -> list[str]:
    return ["nvcc", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
            "-I" + INCLUDE, "-o", out, SRC]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [SRC, os.path.join(INCLUDE, "ovc.h"), *HEADERS]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libovc.so (skipped when up to date) and return its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and not _stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp)
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

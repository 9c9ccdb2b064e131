"""Build ``_lib/libgdnspec.so`` in-tree with nvcc for sm_103a.

One translation unit, one ``-gencode``; the host code links the shared CUDA
runtime so the library and PyTorch share one runtime instance.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
SOURCES = [PKG / "csrc" / "gdn_spec.cu"]
HEADERS = [ROOT / "include" / "gdnspec.h"]
LIB = PKG / "_lib" / "libgdnspec.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-shared", "-cudart", "shared",
    "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", str(ROOT / "include"),
]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdnspec")
    return exe


def stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > t for p in SOURCES + HEADERS)


def build(force: bool = False, extra_flags: list[str] | None = None) -> Path:
    """Compile the library if it is missing or older than its sources."""
    if not force and not stale():
        return LIB
    LIB.parent.mkdir(parents=True, exist_ok=True)
    tmp = LIB.with_suffix(f".so.{os.getpid()}")
    cmd = [nvcc(), *NVCC_FLAGS, *(extra_flags or []), *map(str, SOURCES), "-o", str(tmp)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))

"""Build ``_lib/libgdnspec.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles to an object in parallel (one ``-gencode``),
then one link; the host code links the shared CUDA runtime so the library
and PyTorch share one runtime instance.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
SOURCES = [PKG / "csrc" / "gdn_spec.cu", PKG / "csrc" / "gdn_accept.cu"]
HEADERS = [ROOT / "include" / "gdnspec.h"]
LIB = PKG / "_lib" / "libgdnspec.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", str(ROOT / "include"),
]
LINK_FLAGS = ARCH + ["-shared", "-cudart", "shared"]


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
    objs = [LIB.parent / f"{src.stem}.{os.getpid()}.o" for src in SOURCES]
    procs = [subprocess.Popen([nvcc(), *COMPILE_FLAGS, *(extra_flags or []), "-c", str(src), "-o", str(obj)])
             for src, obj in zip(SOURCES, objs)]
    failed = [p.wait() for p in procs]
    try:
        if any(failed):
            raise subprocess.CalledProcessError(max(failed), "nvcc -c")
        tmp = LIB.with_suffix(f".so.{os.getpid()}")
        subprocess.run([nvcc(), *LINK_FLAGS, *map(str, objs), "-o", str(tmp)], check=True)
        os.replace(tmp, LIB)
    finally:
        for obj in objs:
            obj.unlink(missing_ok=True)
    return LIB


if __name__ == "__main__":
    print(build(force=True))

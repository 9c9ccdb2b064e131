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
# test-only variant: the verify/commit kernels with GDN_TEST_HOOKS (a state copy
# that can be declared and never issued) and a 2 ms staging-wait limit, for the
# test that makes the bounded wait run out; never loaded by the package
TEST_HOOKS_LIB = PKG / "_lib" / "libgdnspec_testhooks.so"
TEST_HOOKS_FLAGS = ["-DGDN_TEST_HOOKS", "-DGDN_WAIT_LIMIT_NS=2000000ull"]
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


def stale(lib: Path = LIB, sources: list[Path] = SOURCES) -> bool:
    if not lib.exists():
        return True
    t = lib.stat().st_mtime
    return any(p.stat().st_mtime > t for p in sources + HEADERS + [Path(__file__)])


def _compile(lib: Path, sources: list[Path], extra_flags: list[str]) -> Path:
    lib.parent.mkdir(parents=True, exist_ok=True)
    objs = [lib.parent / f"{src.stem}.{lib.stem}.{os.getpid()}.o" for src in sources]
    procs = [subprocess.Popen([nvcc(), *COMPILE_FLAGS, *extra_flags, "-c", str(src), "-o", str(obj)])
             for src, obj in zip(sources, objs)]
    failed = [p.wait() for p in procs]
    try:
        if any(failed):
            raise subprocess.CalledProcessError(max(failed), "nvcc -c")
        tmp = lib.with_suffix(f".so.{os.getpid()}")
        subprocess.run([nvcc(), *LINK_FLAGS, *map(str, objs), "-o", str(tmp)], check=True)
        os.replace(tmp, lib)
    finally:
        for obj in objs:
            obj.unlink(missing_ok=True)
    return lib


def build(force: bool = False, extra_flags: list[str] | None = None) -> Path:
    """Compile the library if it is missing or older than its sources."""
    if not force and not stale():
        return LIB
    return _compile(LIB, SOURCES, extra_flags or [])


def build_test_hooks(force: bool = False) -> Path:
    """Compile the test-only variant (verify/commit kernels only) if it is
    missing or older than its sources."""
    src = [PKG / "csrc" / "gdn_spec.cu"]
    if not force and not stale(TEST_HOOKS_LIB, src):
        return TEST_HOOKS_LIB
    return _compile(TEST_HOOKS_LIB, src, TEST_HOOKS_FLAGS)


if __name__ == "__main__":
    print(build(force=True))

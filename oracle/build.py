"""Compile the C oracle into ``oracle/_lib/libgdn_oracle.so`` with gcc.

Plain ISO C, no fused multiply-add contraction, no fast-math, no
machine-specific flags: the same source gives the same fp64 results on x86
and on Arm.
"""
from __future__ import annotations

import os
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
SRC = HERE / "gdn_oracle.c"
LIB = HERE / "_lib" / "libgdn_oracle.so"
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> Path:
    if not force and LIB.exists() and LIB.stat().st_mtime >= SRC.stat().st_mtime:
        return LIB
    LIB.parent.mkdir(parents=True, exist_ok=True)
    tmp = LIB.with_suffix(f".so.{os.getpid()}")
    subprocess.run(["gcc", *CFLAGS, str(SRC), "-o", str(tmp), "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))

"""Compiles the C oracle (test infrastructure) with gcc: IEEE arithmetic,
no contraction of multiply-adds, OpenMP for the O(n^3) GEMM reference."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "liboracle_fp8.so")


def build_oracle(force: bool = False) -> str:
    out = library_path()
    src = os.path.join(_HERE, "fp8_oracle.c")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fopenmp", "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out

"""Builds the C oracle (``gemm_oracle.c``) into ``oracle/_lib/liboracle.so``.

This is test infrastructure.  ``__graft_entry__.build()`` calls it so that
the checker exists on every machine where the tests run.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def build(verbose: bool = False) -> str:
    out_dir = os.path.join(_HERE, "_lib")
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(_HERE, "gemm_oracle.c")
    out = os.path.join(out_dir, "liboracle.so")
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))

"""Compiles the CUDA library in-tree for sm_103a.

Every ``csrc/*.cu`` file is compiled in parallel with one ``-gencode``
(``arch=compute_103a,code=sm_103a``) into ``_lib/``, then linked into
``_lib/libgemm_preshuffle.so`` with the CUDA runtime linked statically.  The
library therefore loads without a GPU or a driver, and it needs libcuda only
on its first CUDA call.  ``rates/mma_rate.cu``, the tensor-pipe rate probe the
benchmark runs for its FP8 and MXFP4 roofline denominators, is built beside
it as the executable ``_lib/mma_rate``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libgemm_preshuffle.so")
RATES_SRC = os.path.join(HERE, "rates", "mma_rate.cu")
RATES_BIN = os.path.join(OUT_DIR, "mma_rate")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--use_fast_math",
         "-Xptxas", "-warn-spills"]
# Files whose arithmetic decides integer codes build with IEEE semantics
# (no approximate division, no flush of denormals to zero).
IEEE_SOURCES = {"quant.cu"}


def _nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(HERE, "..", "include", "*.h")) + [RATES_SRC])


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(RATES_BIN):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(RATES_BIN))
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(verbose: bool = False, force: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
        flags = [f for f in FLAGS if not (os.path.basename(src) in IEEE_SOURCES and f == "--use_fast_math")]
        cmd = [nvcc, *ARCH, *flags, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    def compile_rates():
        tmp_bin = RATES_BIN + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-O3", "-std=c++17", RATES_SRC, "-o", tmp_bin]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {RATES_SRC}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp_bin, RATES_BIN)

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs) + 1)) as ex:
        rates = ex.submit(compile_rates)
        objs = list(ex.map(compile_one, srcs))
        rates.result()
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose=True, force="--force" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else []))

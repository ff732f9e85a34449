"""Seeded synthetic inputs for the preshuffle GEMM workloads.

This module only draws random numbers and turns them into the operand
encodings the GEMM consumes (E4M3 codes + fp32 row scales, INT8, BF16 bits,
packed E2M1 codes + UE8M0 block exponents).  It holds none of the GEMM's own
arithmetic (no products, sums, scaling of results or B packing), so both the
CUDA path and the CPU oracle can consume the very same bytes.

Recipes (the workloads' stated distributions):

* E4M3, per-row scaled: x ~ N(0,1) fp32; per row s = amax(|x|)/448 (fp32);
  q = E4M3FN(x / s), round-to-nearest-even, via torch's float8_e4m3fn cast
  (saturating values in [448, 480) to 448; |x/s| <= 448*(1+2^-24) here).
  A row whose amax is 0 gets s = 1.
* INT8: integers uniform in [-127, 127].
* W4A8: A as INT8; B integers uniform in [-8, 7] (int4), two per byte in
  two's complement, even k in the low nibble.
* BF16: x = N(0,1)/sqrt(K) in fp32, rounded to bf16 (torch cast, RNE).
* FP16: the same draws rounded to IEEE binary16 (torch cast, RNE).
* MXFP4: x ~ N(0,1) fp32; per (row, 32-element K block) the shared exponent
  e is the smallest integer with amax <= 6 * 2^e (i.e. ceil(log2(amax/6))
  evaluated exactly), clamped to [-127, 127], stored biased (e + 127) as
  UE8M0; q = E2M1(x * 2^-e) with round-to-nearest-even on the grid
  {0, .5, 1, 1.5, 2, 3, 4, 6}; two codes per byte, low nibble = even k.
  An all-zero block gets e = 0.

Generators are torch CPU ``Generator`` objects seeded with 20261202 + the
workload's index; A is drawn before B.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

SEED_BASE = 20261202

# dtype names used across the package, the binding and the tests
BF16, E4M3, INT8, E2M1, FP16, W4A8 = "bf16", "e4m3", "int8", "e2m1", "fp16", "w4a8"


@dataclass
class Workload:
    """One GEMM problem C[M,N] = A[M,K] . B[N,K]^T with its input recipe."""
    name: str
    dtype: str
    M: int
    N: int
    K: int
    index: int  # seed offset

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index


# The five workloads, in order (index = seed offset).
WORKLOADS = {
    "fp8_128x256x512": Workload("fp8_128x256x512", E4M3, 128, 256, 512, 0),
    "int8_16x7168x4096": Workload("int8_16x7168x4096", INT8, 16, 7168, 4096, 1),
    "bf16_512x4096x4096": Workload("bf16_512x4096x4096", BF16, 512, 4096, 4096, 2),
    "fp8_8192x8192x8192": Workload("fp8_8192x8192x8192", E4M3, 8192, 8192, 8192, 3),
    "mxfp4_4096x8192x8192": Workload("mxfp4_4096x8192x8192", E2M1, 4096, 8192, 8192, 4),
}

# Further shapes, timed beside the five: the GEMM Optimization Guide's
# worked example (section 14: 5120 x 5120 x 8320 FP8 with per-token scales),
# and FP16 operands at the BF16 shape.
EXTRA_WORKLOADS = {
    "fp8_5120x5120x8320": Workload("fp8_5120x5120x8320", E4M3, 5120, 5120, 8320, 5),
    "fp16_512x4096x4096": Workload("fp16_512x4096x4096", FP16, 512, 4096, 4096, 6),
    "w4a8_16x7168x4096": Workload("w4a8_16x7168x4096", W4A8, 16, 7168, 4096, 7),
}
ALL_WORKLOADS = {**WORKLOADS, **EXTRA_WORKLOADS}


@dataclass
class Operands:
    """Encoded operands.  Arrays are host numpy arrays, row-major.

    a, b       : codes.  uint8 [rows, K] for e4m3 / int8 (int8 viewed as
                 int8), uint16 [rows, K] bf16 or fp16 bits, uint8 [rows, K/2]
                 for e2m1.
    scale_a/b  : float32 [rows] (e4m3) or uint8 [rows, K/32] UE8M0 (e2m1),
                 None otherwise.
    """
    dtype: str
    M: int
    N: int
    K: int
    a: np.ndarray
    b: np.ndarray
    scale_a: Optional[np.ndarray] = None
    scale_b: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def e4m3_rows(rows: int, K: int, g: torch.Generator, chunk: int = 1024):
    """Per-row amax/448 scaled E4M3 codes (uint8 [rows,K]) and fp32 scales."""
    codes = np.empty((rows, K), dtype=np.uint8)
    scales = np.empty((rows,), dtype=np.float32)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        x = torch.randn((r1 - r0, K), generator=g, dtype=torch.float32)
        amax = x.abs().amax(dim=1)
        s = amax / 448.0
        s = torch.where(amax > 0, s, torch.ones_like(s))
        q = (x / s[:, None]).to(torch.float8_e4m3fn)
        codes[r0:r1] = q.view(torch.uint8).numpy()
        scales[r0:r1] = s.numpy()
    return codes, scales


def int8_rows(rows: int, K: int, g: torch.Generator):
    """Integers uniform in [-127, 127] as int8 [rows, K]."""
    x = torch.randint(-127, 128, (rows, K), generator=g, dtype=torch.int16)
    return x.to(torch.int8).numpy()


def int4_rows(rows: int, K: int, g: torch.Generator):
    """Integers uniform in [-8, 7], packed two per byte (two's complement
    nibbles, even k low): uint8 [rows, K/2]."""
    x = torch.randint(-8, 8, (rows, K), generator=g, dtype=torch.int16).numpy()
    nib = (x & 0xF).astype(np.uint8)
    return nib[:, 0::2] | (nib[:, 1::2] << 4)


def bf16_rows(rows: int, K: int, g: torch.Generator, chunk: int = 2048):
    """N(0,1)/sqrt(K) rounded to bf16; returned as uint16 bit patterns."""
    out = np.empty((rows, K), dtype=np.uint16)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        x = torch.randn((r1 - r0, K), generator=g, dtype=torch.float32) / math.sqrt(K)
        out[r0:r1] = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out


def fp16_rows(rows: int, K: int, g: torch.Generator, chunk: int = 2048):
    """N(0,1)/sqrt(K) rounded to IEEE binary16; returned as uint16 bit patterns."""
    out = np.empty((rows, K), dtype=np.uint16)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        x = torch.randn((r1 - r0, K), generator=g, dtype=torch.float32) / math.sqrt(K)
        out[r0:r1] = x.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    return out


# Midpoints between consecutive E2M1 magnitudes {0,.5,1,1.5,2,3,4,6}.
_E2M1_MID = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round values with |v| <= 6 to E2M1 codes (RNE), uint8 in [0,16)."""
    y = np.abs(v).astype(np.float64)
    mid = _E2M1_MID.astype(np.float64)
    i = np.searchsorted(mid, y, side="left")  # number of midpoints < y
    tie = (i < 7) & (y == mid[np.minimum(i, 6)])
    code = i + (tie & (i % 2 == 1))  # a tie goes to the even code
    code = np.minimum(code, 7).astype(np.uint8)
    return code | (np.signbit(v).astype(np.uint8) << 3)


def ue8m0_block_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with amax <= 6*2^e (amax > 0), 0 for amax == 0,
    clamped to [-127, 127].  Evaluated exactly in float64 (6*2^e is exact)."""
    a = amax.astype(np.float64)
    pos = a > 0
    safe = np.where(pos, a, 6.0)
    _, ex = np.frexp(safe / 6.0)           # estimate of ceil(log2(amax/6))
    e = ex.astype(np.int64)
    for _ in range(3):                      # exact correction both ways
        too_small = safe > 6.0 * np.ldexp(1.0, e)
        e = np.where(too_small, e + 1, e)
        too_big = safe <= 6.0 * np.ldexp(1.0, e - 1)
        e = np.where(too_big, e - 1, e)
    e = np.where(pos, e, 0)
    return np.clip(e, -127, 127)


def mxfp4_rows(rows: int, K: int, g: torch.Generator, chunk: int = 512):
    """MXFP4 operand: packed E2M1 codes uint8 [rows, K/2] and UE8M0 uint8 [rows, K/32]."""
    assert K % 32 == 0
    codes = np.empty((rows, K // 2), dtype=np.uint8)
    exps = np.empty((rows, K // 32), dtype=np.uint8)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        x = torch.randn((r1 - r0, K), generator=g, dtype=torch.float32).numpy()
        xb = x.reshape(r1 - r0, K // 32, 32)
        e = ue8m0_block_exponent(np.abs(xb).max(axis=2))
        # power-of-two scaling: exact in float64
        y = (xb.astype(np.float64) * np.ldexp(1.0, -e)[:, :, None]).reshape(r1 - r0, K)
        c = e2m1_encode(y)
        codes[r0:r1] = c[:, 0::2] | (c[:, 1::2] << 4)
        exps[r0:r1] = (e + 127).astype(np.uint8)
    return codes, exps


def make_operands(dtype: str, M: int, N: int, K: int, seed: int) -> Operands:
    """Draw A [M,K] then B [N,K] with the recipe of ``dtype``."""
    g = _gen(seed)
    if dtype == E4M3:
        a, sa = e4m3_rows(M, K, g)
        b, sb = e4m3_rows(N, K, g)
        return Operands(dtype, M, N, K, a, b, sa, sb)
    if dtype == INT8:
        return Operands(dtype, M, N, K, int8_rows(M, K, g), int8_rows(N, K, g))
    if dtype == W4A8:
        return Operands(dtype, M, N, K, int8_rows(M, K, g), int4_rows(N, K, g))
    if dtype == BF16:
        return Operands(dtype, M, N, K, bf16_rows(M, K, g), bf16_rows(N, K, g))
    if dtype == FP16:
        return Operands(dtype, M, N, K, fp16_rows(M, K, g), fp16_rows(N, K, g))
    if dtype == E2M1:
        a, ea = mxfp4_rows(M, K, g)
        b, eb = mxfp4_rows(N, K, g)
        return Operands(dtype, M, N, K, a, b, ea, eb)
    raise ValueError(f"unknown dtype {dtype!r}")


def workload_operands(name: str) -> Operands:
    w = ALL_WORKLOADS[name]
    return make_operands(w.dtype, w.M, w.N, w.K, w.seed)

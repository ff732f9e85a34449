"""CPU oracle for the preshuffle GEMM  C[M,N] = A[M,K] . B[N,K]^T.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s ``cpu_baseline`` leg may import this package.  It shares no
code with the CUDA path and imports nothing from it.  The two meet only in
the seeded input generator (``dense_gemm_preshuffle_gb300.inputs``), which
holds no GEMM arithmetic.

Contents:

* Codecs written from the format definitions:
  - E4M3FN (OCP 8-bit floating point spec: bias 7, no infinities, S.1111.111
    is NaN)
  - E2M1 and UE8M0 (OCP Microscaling formats v1.0)
  - BF16 (the upper half of an IEEE binary32)
  - FP16 (IEEE 754 binary16: bias 15, 10 fraction bits, subnormals)
* GEMMs in fp64 / int64.  The triple loops live in ``gemm_oracle.c``, built
  by ``oracle/build.py``:
  - INT8: C = sum_k a*b, exact in int64.
  - W4A8 (int4 weights B, int8 activations A; "GEMM Optimization Guide"
    section 8.2 counts N*K//2 bytes for such a B): C = sum_k a*b, exact in
    int64.
  - BF16 and FP16: C = sum_k a*b, fp64.
  - E4M3 with per-row/per-column fp32 scales: C = (sum_k qa*qb) * sa[m] * sb[n].
    "GEMM Optimization Guide", section 7.1 (direct store): the epilogue forms
    acc * scale_a * scale_b.  Every E4M3 product is a multiple of 2^-18 and
    |sum| < K*448^2 < 2^31, so the fp64 sum is exact.
  - MXFP4: C = sum_j 2^(ea[m,j]-127) 2^(eb[n,j]-127) sum_{k in block j} qa*qb.
    Same guide, section 8.2: one UE8M0 byte per 32 K-elements of each
    operand.
* The packed-B layout model used to check the device packer byte by byte.
  The layout is this library's own, not the one the guide prints.
* Tile bookkeeping from the guide: section 1.2 (derived tile parameters),
  section 1.5 (MFMA count per tile), sections 8.1-8.2 (flops, bytes moved) and
  section 14 (worked example).
* The fused epilogues the guide names for the preshuffle GEMM ("Kernel
  Tuning Guide", section 6, Epilogue Strategies: "none", "bias",
  "bias_relu", "bias_silu", "bias_gelu"), in fp64: the bias (one value per
  output column) is added to the scaled product, then the activation.
  ReLU max(x, 0); SiLU x / (1 + e^-x); GELU 0.5 x (1 + erf(x / sqrt 2)),
  the exact (erf) form.  The guide names the epilogues without formulas;
  these are the standard definitions.
* The activation quantisers in front of the GEMM (the workloads' operand
  recipes: per-token E4M3 with s = amax/448; MXFP4 with one UE8M0 exponent
  per 32 K-elements, "GEMM Optimization Guide" section 8.2).  Encoders
  written from the format definitions, round to nearest even, saturating.
  The float steps that decide a code are taken in fp32 as the kernel takes
  them: s = fp32(amax / 448) and x / s are IEEE fp32 divisions.
* The float parity metric max |C - C_ref| / (|C_ref| + 1e-2).
* ``gemm_dequantized``: the same plain definition for whole products at the
  workloads' full sizes, dq(A) . dq(B)^T with numpy's fp64 matmul forming
  the sum (the loops above would stream B once per output row).

Parity pins (tests/test_oracle.py): brute force in exact rational arithmetic,
identity and permutation operands, library decodes (torch float8/bfloat16),
the guide's printed worked numbers (tests/golden/), the byte counts of
section 8.2 against the sizes of the arrays they count, and round trips of
the pack model.  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import time
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "liboracle.so")
_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        from . import build as _b
        _b.build()
    lib = ctypes.CDLL(_LIB_PATH)
    i64 = ctypes.c_int64
    vp = ctypes.c_void_p
    lib.oracle_gemm_i8_i64.argtypes = [vp, vp, i64, i64, i64, vp]
    lib.oracle_gemm_f64.argtypes = [vp, vp, i64, i64, i64, vp]
    lib.oracle_gemm_block_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.oracle_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------
# Codecs (decode only; the oracle never needs to encode)
# ----------------------------------------------------------------------------

def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """E4M3FN code -> value (fp64).  Layout s.eeee.mmm, exponent bias 7.

    e == 0  : subnormal, (-1)^s * 2^-6 * m/8
    e  > 0  : normal,    (-1)^s * 2^(e-7) * (1 + m/8)
    e == 15 and m == 7 : NaN (E4M3FN has no infinities).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where(s == 1, -mag, mag)
    return np.where((e == 15) & (m == 7), np.nan, val)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """E2M1 code (low 4 bits) -> value (fp64).  Layout s.ee.m, exponent bias 1.

    e == 0 : subnormal, (-1)^s * 0.5 * m
    e  > 0 : normal,    (-1)^s * 2^(e-1) * (1 + m/2)
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 0xF
    s = (c >> 3) & 1
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + m / 2.0, e - 1))
    return np.where(s == 1, -mag, mag)


def decode_ue8m0(codes: np.ndarray) -> np.ndarray:
    """UE8M0 scale byte -> 2^(code - 127) (fp64); 0xFF is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """BF16 bit pattern -> value (fp64): the upper 16 bits of a binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def decode_fp16(bits: np.ndarray) -> np.ndarray:
    """IEEE 754 binary16 bit pattern -> value (fp64): sign, 5 exponent bits
    (bias 15), 10 fraction bits; exponent 0 is subnormal (2^-14 * f/1024),
    exponent 31 is infinity (f = 0) or NaN."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    normal = sign * (1.0 + f / 1024.0) * np.exp2(e.astype(np.float64) - 15.0)
    sub = sign * (f / 1024.0) * 2.0 ** -14
    special = np.where(f == 0, sign * np.inf, np.nan)
    return np.where(e == 0, sub, np.where(e == 31, special, normal))


def unpack_e2m1_rows(packed: np.ndarray, K: int) -> np.ndarray:
    """[rows, K/2] bytes (low nibble = even k) -> [rows, K] codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], K), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


# ----------------------------------------------------------------------------
# GEMMs.  All return the exact (unrounded) fp64 result, or int64 for INT8.
# ----------------------------------------------------------------------------

def gemm_int8(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """C = A . B^T for int8 A [M,K], B [N,K]; int64 result."""
    a = np.ascontiguousarray(a, dtype=np.int8)
    b = np.ascontiguousarray(b, dtype=np.int8)
    M, K = a.shape
    N = b.shape[0]
    c = np.empty((M, N), dtype=np.int64)
    _load().oracle_gemm_i8_i64(_p(a), _p(b), M, N, K, _p(c))
    return c


def unpack_int4_rows(packed: np.ndarray, K: int) -> np.ndarray:
    """int4 B [rows, K/2] bytes (two's complement nibbles, even k in the low
    nibble) -> int8 [rows, K] values in [-8, 7]."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], K), dtype=np.int16)
    lo = (p & 0xF).astype(np.int16)
    hi = (p >> 4).astype(np.int16)
    out[:, 0::2] = np.where(lo >= 8, lo - 16, lo)
    out[:, 1::2] = np.where(hi >= 8, hi - 16, hi)
    return out.astype(np.int8)


def gemm_w4a8(a: np.ndarray, b_packed: np.ndarray, K: int) -> np.ndarray:
    """C = A . B^T for int8 A [M, K] and int4 B (packed [N, K/2]); int64."""
    return gemm_int8(a, unpack_int4_rows(b_packed, K))


def gemm_f64(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """C = A . B^T for already-decoded fp64 A [M,K], B [N,K]."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    M, K = a.shape
    N = b.shape[0]
    c = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_f64(_p(a), _p(b), M, N, K, _p(c))
    return c


def gemm_bf16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return gemm_f64(decode_bf16(a_bits), decode_bf16(b_bits))


def gemm_fp16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return gemm_f64(decode_fp16(a_bits), decode_fp16(b_bits))


def gemm_e4m3_rowcol(qa: np.ndarray, qb: np.ndarray, sa: np.ndarray, sb: np.ndarray) -> np.ndarray:
    """C[m,n] = (sum_k qa[m,k] qb[n,k]) * sa[m] * sb[n]: the accumulator is
    scaled by the row scale of A and the column scale (row of B).  Missing
    scales (None) mean an unscaled product."""
    acc = gemm_f64(decode_e4m3(qa), decode_e4m3(qb))
    if sa is not None:
        acc = acc * np.asarray(sa, np.float64)[:, None]
    if sb is not None:
        acc = acc * np.asarray(sb, np.float64)[None, :]
    return acc


def gemm_mxfp4(pa: np.ndarray, pb: np.ndarray, ea: np.ndarray, eb: np.ndarray, K: int) -> np.ndarray:
    """MXFP4 product: packed E2M1 [rows, K/2] with UE8M0 [rows, K/32]."""
    a = np.ascontiguousarray(decode_e2m1(unpack_e2m1_rows(pa, K)))
    b = np.ascontiguousarray(decode_e2m1(unpack_e2m1_rows(pb, K)))
    sa = np.ascontiguousarray(decode_ue8m0(ea))
    sb = np.ascontiguousarray(decode_ue8m0(eb))
    M, N = a.shape[0], b.shape[0]
    c = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_block_f64(_p(a), _p(b), _p(sa), _p(sb), M, N, K, 32, _p(c))
    return c


def gemm_operands(ops, rows: Optional[np.ndarray] = None, cols: Optional[np.ndarray] = None) -> np.ndarray:
    """Reference C for an ``Operands`` bundle, optionally restricted to the
    given output rows (of A) and columns (rows of B)."""
    a, b, sa, sb = ops.a, ops.b, ops.scale_a, ops.scale_b
    if rows is not None:
        a = a[rows]
        sa = None if sa is None else sa[rows]
    if cols is not None:
        b = b[cols]
        sb = None if sb is None else sb[cols]
    if ops.dtype == "int8":
        return gemm_int8(a, b)
    if ops.dtype == "w4a8":
        return gemm_w4a8(a, b, ops.K)
    if ops.dtype == "bf16":
        return gemm_bf16(a, b)
    if ops.dtype == "fp16":
        return gemm_fp16(a, b)
    if ops.dtype == "e4m3":
        return gemm_e4m3_rowcol(a, b, sa, sb)
    if ops.dtype == "e2m1":
        return gemm_mxfp4(a, b, sa, sb, ops.K)
    raise ValueError(ops.dtype)


def expand_block_scales(e: np.ndarray, K: int, blk: int = 32) -> np.ndarray:
    """UE8M0 block exponents [rows, K/blk] -> per-element scales [rows, K]
    (fp64): element k takes the scale of block k // blk."""
    return np.repeat(decode_ue8m0(e), blk, axis=1)[:, :K]


def _mx_sum_is_exact(ea: np.ndarray, eb: np.ndarray, K: int) -> bool:
    """True when every sum over k of dq(A)[m,k] dq(B)[n,k] is exact in fp64.

    E2M1 values are multiples of 1/2 with |v| <= 6, so a product is a multiple
    of 2^(ea + eb - 254 - 2) with magnitude at most 36 * 2^(ea + eb - 254).
    Over all (m, n) the exponent sums lie in [lo, hi]; a sum of K products
    then needs fewer than log2(K * 36) + (hi - lo) + 2 bits, which must stay
    within fp64's 53."""
    if ea.size == 0 or eb.size == 0:
        return True
    if (ea == 255).any() or (eb == 255).any():
        return False  # NaN scales
    lo = int(ea.min()) + int(eb.min())
    hi = int(ea.max()) + int(eb.max())
    return np.log2(max(K, 1) * 36.0) + (hi - lo) + 2 < 53


def gemm_dequantized(ops, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Reference C of a whole large product, from the plain definition
    C[m,n] = sum_k dq(A)[m,k] dq(B)[n,k] with numpy's fp64 matmul (a library
    routine) forming the sum over k.  At the full workload sizes the loops of
    ``gemm_operands`` stream B from memory once per output row and take hours;
    this takes seconds and reaches the same values:

    * E4M3: the sum of the decoded codes is exact in fp64 in any order (every
      product is a multiple of 2^-18 and |sum| < K 448^2), then it is scaled
      by sa[m] and sb[n] exactly as ``gemm_e4m3_rowcol`` does, so the result
      is bit-identical to it.
    * MXFP4 ("GEMM Optimization Guide" section 8.2: one UE8M0 scale per 32
      K-elements of each operand): dq(x)[k] = e2m1(x[k]) * 2^(e[k//32]-127).
      Summing dq(A) dq(B) over k regroups the block-scaled sum of
      ``gemm_mxfp4`` term by term; where ``_mx_sum_is_exact`` holds both are
      the exact value, hence identical.  Otherwise the block loops are used.
    * BF16 / FP16: the decoded operands summed in fp64; the order differs from
      the loops, each within K 2^-53 sum |a b|.
    * INT8 / W4A8: the exact int64 product of ``gemm_operands``.
    """
    a, b, sa, sb = ops.a, ops.b, ops.scale_a, ops.scale_b
    if rows is not None:
        a = a[rows]
        sa = None if sa is None else sa[rows]
    if ops.dtype in ("int8", "w4a8"):
        return gemm_operands(ops, rows=rows)
    if ops.dtype == "bf16":
        return decode_bf16(a) @ decode_bf16(b).T
    if ops.dtype == "fp16":
        return decode_fp16(a) @ decode_fp16(b).T
    if ops.dtype == "e4m3":
        acc = decode_e4m3(a) @ decode_e4m3(b).T
        if sa is not None:
            acc = acc * np.asarray(sa, np.float64)[:, None]
        if sb is not None:
            acc = acc * np.asarray(sb, np.float64)[None, :]
        return acc
    if ops.dtype == "e2m1":
        K = ops.K
        if not _mx_sum_is_exact(sa, sb, K):
            return gemm_operands(ops, rows=rows)
        da = decode_e2m1(unpack_e2m1_rows(a, K)) * expand_block_scales(sa, K)
        db = decode_e2m1(unpack_e2m1_rows(b, K)) * expand_block_scales(sb, K)
        return da @ db.T
    raise ValueError(ops.dtype)


def gemm_abs_operands(ops, rows: Optional[np.ndarray] = None, cols: Optional[np.ndarray] = None) -> np.ndarray:
    """S[m,n] = sum_k |dq(A)[m,k]| |dq(B)[n,k]|, the magnitude that the
    accumulation runs through: the denominator of the error diagnostic
    max |C - C_ref| / S, in which bf16 output rounding contributes at most
    2^-9 and an fp32 accumulation at most about K 2^-24 (the dequantised
    operands are the same as in ``gemm_operands``; scales are positive)."""
    a, b, sa, sb = ops.a, ops.b, ops.scale_a, ops.scale_b
    if rows is not None:
        a = a[rows]
        sa = None if sa is None else sa[rows]
    if cols is not None:
        b = b[cols]
        sb = None if sb is None else sb[cols]
    if ops.dtype == "int8":
        return gemm_f64(np.abs(a.astype(np.float64)), np.abs(b.astype(np.float64)))
    if ops.dtype == "w4a8":
        return gemm_f64(np.abs(a.astype(np.float64)), np.abs(unpack_int4_rows(b, ops.K).astype(np.float64)))
    if ops.dtype == "bf16":
        return gemm_f64(np.abs(decode_bf16(a)), np.abs(decode_bf16(b)))
    if ops.dtype == "fp16":
        return gemm_f64(np.abs(decode_fp16(a)), np.abs(decode_fp16(b)))
    if ops.dtype == "e4m3":
        acc = gemm_f64(np.abs(decode_e4m3(a)), np.abs(decode_e4m3(b)))
        if sa is not None:
            acc = acc * np.abs(np.asarray(sa, np.float64))[:, None]
        if sb is not None:
            acc = acc * np.abs(np.asarray(sb, np.float64))[None, :]
        return acc
    if ops.dtype == "e2m1":
        K = ops.K
        av = np.ascontiguousarray(np.abs(decode_e2m1(unpack_e2m1_rows(a, K))))
        bv = np.ascontiguousarray(np.abs(decode_e2m1(unpack_e2m1_rows(b, K))))
        M, N = av.shape[0], bv.shape[0]
        c = np.empty((M, N), dtype=np.float64)
        _load().oracle_gemm_block_f64(_p(av), _p(bv), _p(np.ascontiguousarray(decode_ue8m0(sa))),
                                      _p(np.ascontiguousarray(decode_ue8m0(sb))), M, N, K, 32, _p(c))
        return c
    raise ValueError(ops.dtype)


def max_err_over_abs(c: np.ndarray, c_ref: np.ndarray, s: np.ndarray) -> float:
    """max |C - C_ref| / S with S from ``gemm_abs_operands`` (entries with
    S = 0 must match exactly and count as 0)."""
    c = np.asarray(c, np.float64)
    r = np.asarray(c_ref, np.float64)
    s = np.asarray(s, np.float64)
    if c.size == 0:
        return 0.0
    d = np.abs(c - r)
    if np.any((s == 0) & (d != 0)):
        return float("inf")
    return float(np.max(np.where(s > 0, d / np.where(s > 0, s, 1.0), 0.0)))


# ----------------------------------------------------------------------------
# Output rounding model and the parity metric
# ----------------------------------------------------------------------------

# ----------------------------------------------------------------------------
# Activation quantisers (encoders from the OCP format definitions)
# ----------------------------------------------------------------------------

def encode_e4m3(v: np.ndarray) -> np.ndarray:
    """Values -> E4M3FN codes, round to nearest even, saturating at +-448
    (no infinities; 448 is S.1111.110).  NaN -> 0x7F."""
    v = np.asarray(v, dtype=np.float64)
    a = np.where(np.isnan(v), 0.0, np.abs(v))           # NaN is coded separately below
    sign = np.signbit(v).astype(np.uint8) << 7
    f, ex = np.frexp(np.where(a > 0, a, 1.0))          # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, -6)         # floor(log2 a), subnormals below 2^-6
    quantum = np.ldexp(1.0, e - 3)                       # 3 fraction bits
    n = np.rint(a / quantum).astype(np.int64)            # exact quotient, ties to even
    carry = n >= 16                                      # rounded up to the next binade
    e = np.where(carry, e + 1, e)
    n = np.where(carry, n // 2, n)
    normal = n >= 8
    code = np.where(normal, ((e + 7) << 3) | (n - 8), n)
    code = np.where(a == 0, 0, code)
    code = np.where((code > 0x7E) | (a >= 448.0), 0x7E, code)  # satfinite
    code = code.astype(np.uint8) | sign
    return np.where(np.isnan(v), np.uint8(0x7F), code)


def encode_e2m1(v: np.ndarray) -> np.ndarray:
    """Values -> E2M1 codes (4-bit, uint8), round to nearest even on the grid
    {0, .5, 1, 1.5, 2, 3, 4, 6}, saturating at +-6."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = np.signbit(v).astype(np.uint8) << 3
    # spacing 0.5 below 2, 1 in [2, 4), 2 from 4
    quantum = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    n = np.rint(a / quantum).astype(np.int64)
    val = np.minimum(n * quantum, 6.0)                   # a tie that crosses a binade edge lands on it
    code = np.select([val < 2.0, val < 4.0], [(val * 2).astype(np.int64), (val + 2).astype(np.int64)],
                     (val / 2 + 4).astype(np.int64))
    return code.astype(np.uint8) | sign


def quantize_e4m3_rows(x: np.ndarray):
    """Per-row (per-token) E4M3 quantisation of fp32 x [M, K]:
    s = fp32(amax / 448) (1 where amax = 0), q = E4M3(fp32(x / s)).
    Returns (codes uint8 [M, K], s fp32 [M])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    return encode_e4m3((x / s[:, None]).astype(np.float64)), s


def mx_block_exponent(amax: np.ndarray) -> np.ndarray:
    """The smallest integer e with amax <= 6 * 2^e (0 for amax = 0), clamped
    to [-127, 127].  With amax = f * 2^x (f in [0.5, 1)): 6 * 2^e = 0.75 *
    2^(e + 3), so e = x - 3 when f <= 0.75, else x - 2.  Exact."""
    a = np.asarray(amax, dtype=np.float64)
    f, x = np.frexp(a)
    e = np.where(f <= 0.75, x - 3, x - 2).astype(np.int64)
    return np.clip(np.where(a > 0, e, 0), -127, 127)


def quantize_mxfp4_rows(x: np.ndarray):
    """MXFP4 quantisation of fp32 x [M, K] in blocks of 32 along K: e from
    the block's amax, q = E2M1(x * 2^-e).  Returns (packed codes uint8
    [M, K/2], even k in the low nibble; UE8M0 exponents e + 127, uint8
    [M, K/32])."""
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    xb = x.reshape(M, K // 32, 32).astype(np.float64)
    e = mx_block_exponent(np.abs(xb).max(axis=2))
    c = encode_e2m1((xb * np.ldexp(1.0, -e)[:, :, None]).reshape(M, K))
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8), (e + 127).astype(np.uint8)


EPILOGUES = ("none", "bias", "bias_relu", "bias_silu", "bias_gelu")


def apply_epilogue(c: np.ndarray, epilogue: str, bias: Optional[np.ndarray] = None) -> np.ndarray:
    """The named epilogue applied to an fp64 product C [M, N]: C + bias[n],
    then the activation ("Kernel Tuning Guide", section 6)."""
    if epilogue not in EPILOGUES:
        raise ValueError(f"unknown epilogue {epilogue!r}")
    x = np.asarray(c, dtype=np.float64)
    if epilogue == "none":
        return x.copy()
    x = x + np.asarray(bias, dtype=np.float64)[None, :]
    if epilogue == "bias":
        return x
    if epilogue == "bias_relu":
        return np.maximum(x, 0.0)
    if epilogue == "bias_silu":
        with np.errstate(over="ignore"):
            return x / (1.0 + np.exp(-x))
    from scipy.special import erf
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def max_rel_err(c: np.ndarray, c_ref: np.ndarray) -> float:
    """max over all elements of |C - C_ref| / (|C_ref| + 1e-2)."""
    c = np.asarray(c, np.float64)
    r = np.asarray(c_ref, np.float64)
    if c.size == 0:
        return 0.0
    return float(np.max(np.abs(c - r) / (np.abs(r) + 1e-2)))


FLOAT_TOL = 8e-3


# ----------------------------------------------------------------------------
# Packed-B layout model (this library's own layout)
#
# B is a byte matrix [N, Kb] (Kb = K * element bytes; E2M1 packs two per
# byte).  It is cut into tiles of R rows x 128 bytes, where the band height R
# is 128 for BF16, E4M3 and E2M1 (the tcgen05 tiles) and 8 for INT8 (the
# weight-streaming kernel, whose per-SM strips are whole 8-row units).
# Tile (tn, tk) is stored at tile index tn * (Kb/128) + tk, i.e. all K tiles
# of one R-row band are contiguous.  Inside a tile, row r occupies 128 bytes
# at r*128 and its eight 16-byte chunks are permuted: chunk c of the row is
# stored at chunk position c XOR (r mod 8).  INT8 bytes are stored in offset
# binary (b XOR 0x80 = b + 128 unsigned), the form its kernel feeds the MMA.
# ----------------------------------------------------------------------------

TILE_ROWS = 128
TILE_BYTES = 128


def elem_bits(dtype: str) -> int:
    return {"bf16": 16, "fp16": 16, "e4m3": 8, "int8": 8, "e2m1": 4, "w4a8": 4}[dtype]


def band_rows(dtype: str) -> int:
    """Rows per packed tile: 8 for INT8 and W4A8, 128 for the tcgen05 element types."""
    return 8 if dtype in ("int8", "w4a8") else TILE_ROWS


def packed_offset(n: np.ndarray, kb: np.ndarray, Kb: int, rows: int = TILE_ROWS, w4: bool = False) -> np.ndarray:
    """Byte offset in the packed buffer of byte (n, kb) of B, for tiles of `rows` rows.

    The 16-byte chunk c of row r sits at slot c XOR (r mod 8).  W4A8's
    layout also flips slot bit 2 on odd rows (c XOR (r mod 8) XOR 4 (r mod 2)):
    its kernel reads four consecutive chunks of rows 2i and 2i + 1 together,
    and the flip puts the two rows in different halves of the banks."""
    n = np.asarray(n, np.int64)
    kb = np.asarray(kb, np.int64)
    tiles_k = Kb // TILE_BYTES
    tn, r = n // rows, n % rows
    tk, col = kb // TILE_BYTES, kb % TILE_BYTES
    chunk, byte = col // 16, col % 16
    tile_index = tn * tiles_k + tk
    mask = (r % 8) ^ (4 * (r % 2)) if w4 else r % 8
    return tile_index * (rows * TILE_BYTES) + r * TILE_BYTES + ((chunk ^ mask) * 16) + byte


def pack_b_bytes(b_bytes: np.ndarray, rows: int = TILE_ROWS, w4: bool = False) -> np.ndarray:
    """Scatter every byte of B [N, Kb] to its packed offset."""
    b = np.ascontiguousarray(b_bytes).view(np.uint8)
    N, Kb = b.shape
    nn, kk = np.meshgrid(np.arange(N), np.arange(Kb), indexing="ij")
    out = np.zeros(N * Kb, dtype=np.uint8)
    out[packed_offset(nn, kk, Kb, rows, w4).ravel()] = b.ravel()
    return out


def unpack_b_bytes(packed: np.ndarray, N: int, Kb: int, rows: int = TILE_ROWS, w4: bool = False) -> np.ndarray:
    """Gather B [N, Kb] back from the packed buffer."""
    nn, kk = np.meshgrid(np.arange(N), np.arange(Kb), indexing="ij")
    return np.asarray(packed, np.uint8)[packed_offset(nn, kk, Kb, rows, w4)]


# Block scales of an MXFP4 B ([N, K/32] UE8M0) are packed per (128-row band,
# 128-byte K tile) = 128 rows x 8 scale bytes, in two 512-byte groups of four
# K-blocks.  Inside a group, the byte of (row r, block j) is at
# (r % 32) * 16 + (r // 32) * 4 + (j % 4).  The scale region follows the data
# region in the same buffer.

def packed_scale_offset(n: np.ndarray, j: np.ndarray, nblk: int) -> np.ndarray:
    """Offset (within the scale region) of the scale of (row n, K block j)."""
    n = np.asarray(n, np.int64)
    j = np.asarray(j, np.int64)
    tiles_k = nblk // 8            # 8 scale blocks per 128-byte K tile of E2M1
    tn, r = n // TILE_ROWS, n % TILE_ROWS
    tk, jj = j // 8, j % 8
    group = tn * (tiles_k * 2) + tk * 2 + jj // 4
    return group * 512 + (r % 32) * 16 + (r // 32) * 4 + (jj % 4)


def pack_b_scales(scales: np.ndarray) -> np.ndarray:
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    N, nblk = s.shape
    nn, jj = np.meshgrid(np.arange(N), np.arange(nblk), indexing="ij")
    out = np.zeros(N * nblk, dtype=np.uint8)
    out[packed_scale_offset(nn, jj, nblk).ravel()] = s.ravel()
    return out


def unpack_b_scales(packed: np.ndarray, N: int, nblk: int) -> np.ndarray:
    nn, jj = np.meshgrid(np.arange(N), np.arange(nblk), indexing="ij")
    return np.asarray(packed, np.uint8)[packed_scale_offset(nn, jj, nblk)]


def byte_bias(dtype: str) -> int:
    """XOR applied to every packed data byte: INT8 is stored in offset binary
    (b + 128 as an unsigned byte), the other element types unchanged."""
    return 0x80 if dtype == "int8" else 0


# W4A8's int4 B: each 32-bit little-endian word of a row holds K values
# k0..k7 as offset-binary nibbles u = b + 8, k0..k7 at bits 0, 16, 4, 20, 8,
# 24, 12, 28, so that (word >> 4j) & 0x000F000F is the pair (k2j, k2j+1) as
# two fp16 bit patterns.
W4_NIBBLE_BITS = (0, 16, 4, 20, 8, 24, 12, 28)


def interleave_int4_words(b_packed: np.ndarray) -> np.ndarray:
    """int4 B bytes [N, K/2] (two's complement, even k low) -> the packed
    word order above, as bytes [N, K/2]."""
    p = np.ascontiguousarray(b_packed, dtype=np.uint8)
    N, Kb = p.shape
    nib = np.empty((N, Kb * 2), dtype=np.uint32)
    nib[:, 0::2] = p & 0xF
    nib[:, 1::2] = p >> 4
    u = nib ^ 0x8                                         # offset binary: b + 8
    u = u.reshape(N, Kb // 4, 8)
    words = np.zeros((N, Kb // 4), dtype=np.uint32)
    for k, bit in enumerate(W4_NIBBLE_BITS):
        words |= u[:, :, k] << np.uint32(bit)
    return words.astype("<u4").view(np.uint8).reshape(N, Kb)


def pack_b(b: np.ndarray, dtype: str, scales: Optional[np.ndarray] = None) -> np.ndarray:
    """Whole packed buffer for B (data region, then the scale region for E2M1)."""
    if dtype == "w4a8":
        return pack_b_bytes(interleave_int4_words(b), band_rows(dtype), w4=True)
    raw = np.ascontiguousarray(b).view(np.uint8).reshape(b.shape[0], -1) ^ np.uint8(byte_bias(dtype))
    data = pack_b_bytes(raw, band_rows(dtype))
    if dtype == "e2m1":
        return np.concatenate([data, pack_b_scales(scales)])
    return data


# ----------------------------------------------------------------------------
# Tile bookkeeping and byte/flop counts ("GEMM Optimization Guide")
# ----------------------------------------------------------------------------

def tile_params(tile_m: int, tile_n: int, tile_k: int, elem_bytes: float, a_elem_vec_pack: int = 1) -> dict:
    """Section 1.2: derived tile parameters of the 4-wave, 16x16-MFMA tiling."""
    tile_k_bytes = int(tile_k * elem_bytes)
    return {
        "m_repeat": tile_m // 16,
        "n_per_wave": tile_n // 4,
        "num_acc_n": (tile_n // 4) // 16,
        "k_unroll": tile_k_bytes // a_elem_vec_pack // 64,
    }


def mfma_per_tile(tile_m: int, tile_n: int, tile_k: int, elem_bytes: float) -> int:
    """Section 1.5: k_unroll * m_repeat * num_acc_n * 2 (two K32 per K64 step)."""
    p = tile_params(tile_m, tile_n, tile_k, elem_bytes)
    return p["k_unroll"] * p["m_repeat"] * p["num_acc_n"] * 2


def grid_blocks(M: int, N: int, tile_m: int, tile_n: int) -> int:
    """Section 1.1: one block per (M tile, N tile)."""
    return (M // tile_m) * (N // tile_n)


def mfma_per_block(K: int, tile_m: int, tile_n: int, tile_k: int, elem_bytes: float) -> int:
    """Section 14, step 2: MFMAs per tile times the number of K tiles."""
    return mfma_per_tile(tile_m, tile_n, tile_k, elem_bytes) * (K // tile_k)


def lds_bytes(tile_m: int, tile_k: int, elem_bytes: float, stages: int = 2) -> int:
    """Section 2.4: stages * tile_m * tile_k * elem_bytes."""
    return int(stages * tile_m * tile_k * elem_bytes)


def flops(M: int, N: int, K: int) -> int:
    """Section 8.1: 2*M*N*K."""
    return 2 * M * N * K


def bytes_moved(M: int, N: int, K: int, kind: str) -> int:
    """Section 8.2 byte counts.

    kind = "fp8" / "int8"  : M*K + N*K + 2*M*N + 4*(M+N)
    kind = "int4"          : M*K + N*K/2 + 2*M*N + 4*(M+N)
    kind = "mxfp4"         : M*K/2 + N*K/2 + 2*M*N + (M+N)*K/32
    """
    if kind in ("fp8", "int8"):
        return M * K + N * K + M * N * 2 + (M + N) * 4
    if kind == "int4":
        return M * K + (N * K) // 2 + M * N * 2 + (M + N) * 4
    if kind == "mxfp4":
        return (M * K) // 2 + (N * K) // 2 + M * N * 2 + (M + N) * (K // 32)
    raise ValueError(kind)


def tflops(M: int, N: int, K: int, us: float) -> float:
    """Section 8.1: flops / (us/1e6) / 1e12."""
    return flops(M, N, K) / (us / 1e6) / 1e12


# ----------------------------------------------------------------------------
# CPU baseline timing helper (used by bench.py's cpu_baseline leg only)
# ----------------------------------------------------------------------------

def time_gemm(ops, rows: np.ndarray, cols: Optional[np.ndarray] = None) -> float:
    """Wall-clock seconds for the reference C of the given output rows (and columns)."""
    t0 = time.perf_counter()
    gemm_operands(ops, rows=rows, cols=cols)
    return time.perf_counter() - t0

"""Seeded random shapes through the K-split paths, against the oracle.

* INT8 / W4A8 with a narrow N, where the library splits each strip's K
  stages over a 2-, 4- or 8-CTA cluster (or not at all, where the stages
  are too few): random M (1-48 rows, ragged row groups), N (multiples of
  128 up to 2048) and K (multiples of 128, or 256 for int4 weights, up to
  16384).  Bit-exact.
* The two-pair K split (GP_XPAIR=1 forces it wherever valid, in a child
  process): random M (129-1024), N (multiples of 256 up to 1536) and K
  (any number of 128-byte K tiles from 2 to 80), BF16 / FP16 / E4M3.
  Within the float bound.
* The library's own choice of float kernel (128 x 128 or 128 x 256 tiles,
  2-CTA pairs, split-K clusters, the two-pair K split): random M (1-1500),
  N (multiples of 128 up to 3072) and K (1-40 K tiles of 128 bytes),
  BF16 / FP16 / E4M3.  Within the float bound.
* MXFP4 (single-CTA 128 x 256 tiles for M <= 128, 2-CTA pairs above):
  random M (1-700), N (multiples of 256 up to 1536) and K (multiples of
  256 up to 6144).  Within the float bound.

The shapes come from a fixed seed, so every run checks the same ones.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import oracle
import dense_gemm_preshuffle_gb300 as gp
from dense_gemm_preshuffle_gb300 import inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def int_shapes(n=14):
    rng = np.random.default_rng(2026)
    out = []
    for i in range(n):
        dtype = "int8" if i % 2 == 0 else "w4a8"
        M = int(rng.integers(1, 49))
        N = 128 * int(rng.integers(1, 17))
        step = 256 if dtype == "w4a8" else 128
        K = step * int(rng.integers(1, 16384 // step + 1))
        out.append((dtype, M, N, K))
    return out


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_preshuffle_gb300 import build
    build.build()
    gp.load_library()


@pytest.mark.parametrize("case", int_shapes(), ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_integer_random_shapes(lib, case):
    dtype, M, N, K = case
    ops = inputs.make_operands(dtype, M, N, K, seed=150 + M + N // 128)
    A = torch.from_numpy(np.ascontiguousarray(ops.a)).cuda()
    Bp = gp.preshuffle_b(torch.from_numpy(np.ascontiguousarray(ops.b)).cuda(), dtype)
    out = torch.full((M, N), -2 ** 31, dtype=torch.int32, device="cuda")
    gp.matmul(A, Bp, dtype, N, K, out=out)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    c = out.cpu().numpy().astype(np.int64)
    ref = oracle.gemm_operands(ops)
    assert np.array_equal(c, ref), f"{int((c != ref).sum())} mismatching int32 outputs"


def float_shapes(n=10):
    rng = np.random.default_rng(4052)
    out = []
    for i in range(n):
        dtype = ("bf16", "fp16", "e4m3")[i % 3]
        M = int(rng.integers(129, 1025))
        N = 256 * int(rng.integers(1, 7))
        ktiles = int(rng.integers(2, 81))
        K = ktiles * (128 if dtype == "e4m3" else 64)
        out.append((dtype, M, N, K))
    return out


CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np, torch
    import dense_gemm_preshuffle_gb300 as gp
    from dense_gemm_preshuffle_gb300 import inputs
    gp.load_library()
    out = {{}}
    for i, (dtype, M, N, K) in enumerate({cases!r}):
        ops = inputs.make_operands(dtype, M, N, K, seed=170 + i)
        def t(x):
            if x is None:
                return None
            if x.dtype == np.uint16:
                x = x.view(np.int16)
            return torch.from_numpy(np.ascontiguousarray(x)).cuda()
        A, B, sa, sb = t(ops.a), t(ops.b), t(ops.scale_a), t(ops.scale_b)
        Bp = gp.preshuffle_b(B, dtype)
        C = torch.full((M, N), float("nan"), dtype=torch.float16 if dtype == "fp16" else torch.bfloat16,
                       device="cuda")
        gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb, out=C)
        torch.cuda.synchronize()
        assert gp.gemm_last_device_status() == 0
        out["c%d" % i] = C.view(torch.int16).cpu().numpy()
    np.savez({path!r}, **out)
""")


def test_two_pair_random_shapes(lib, tmp_path):
    cases = float_shapes()
    path = str(tmp_path / "sweep.npz")
    env = dict(os.environ, GP_XPAIR="1")
    for k in ("GP_TC_TILE", "GP_TC_PAIR", "GP_SPLITK", "GP_PAIR_KSPLIT"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, cases=cases, path=path)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    res = np.load(path)
    for i, (dtype, M, N, K) in enumerate(cases):
        ops = inputs.make_operands(dtype, M, N, K, seed=170 + i)
        ref = oracle.gemm_dequantized(ops)
        c = torch.from_numpy(res["c%d" % i]).view(torch.float16 if dtype == "fp16" else torch.bfloat16)
        c = c.float().numpy().astype(np.float64)
        assert not np.isnan(c).any(), f"{dtype} {M}x{N}x{K}: outputs left unwritten"
        err = oracle.max_rel_err(c, ref)
        assert err <= oracle.FLOAT_TOL, f"{dtype} {M}x{N}x{K}: max rel err {err:.3e}"


def _dev(x):
    if x is None:
        return None
    if x.dtype == np.uint16:
        x = x.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _float_result(c, dtype):
    return c.view(torch.float16 if dtype == "fp16" else torch.bfloat16).float().cpu().numpy().astype(np.float64)


def dispatch_shapes(n=12):
    rng = np.random.default_rng(6104)
    out = []
    for i in range(n):
        dtype = ("bf16", "e4m3", "fp16")[i % 3]
        M = int(rng.integers(1, 1501))
        N = 128 * int(rng.integers(1, 25))
        ktiles = int(rng.integers(1, 41))
        K = ktiles * (128 if dtype == "e4m3" else 64)
        out.append((dtype, M, N, K))
    return out


@pytest.mark.parametrize("case", dispatch_shapes(), ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_float_random_shapes_default_dispatch(lib, case):
    dtype, M, N, K = case
    ops = inputs.make_operands(dtype, M, N, K, seed=190 + M % 97)
    A, B, sa, sb = _dev(ops.a), _dev(ops.b), _dev(ops.scale_a), _dev(ops.scale_b)
    Bp = gp.preshuffle_b(B, dtype)
    C = torch.full((M, N), float("nan"), dtype=torch.float16 if dtype == "fp16" else torch.bfloat16, device="cuda")
    gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb, out=C)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    c = _float_result(C, dtype)
    assert not np.isnan(c).any(), "outputs left unwritten"
    err = oracle.max_rel_err(c, oracle.gemm_dequantized(ops))
    assert err <= oracle.FLOAT_TOL, f"max rel err {err:.3e}"


def mxfp4_shapes(n=10):
    rng = np.random.default_rng(7311)
    out = []
    for i in range(n):
        M = int(rng.integers(1, 129)) if i % 3 == 0 else int(rng.integers(129, 701))
        N = 256 * int(rng.integers(1, 7))
        K = 256 * int(rng.integers(1, 25))
        out.append(("e2m1", M, N, K))
    return out


@pytest.mark.parametrize("case", mxfp4_shapes(), ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_mxfp4_random_shapes(lib, case):
    dtype, M, N, K = case
    ops = inputs.make_operands(dtype, M, N, K, seed=230 + M % 89)
    A, B, ea, eb = _dev(ops.a), _dev(ops.b), _dev(ops.scale_a), _dev(ops.scale_b)
    Bp = gp.preshuffle_b(B, dtype, B_scales=eb)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    gp.matmul(A, Bp, dtype, N, K, scale_a=ea, out=C)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    c = _float_result(C, dtype)
    assert not np.isnan(c).any(), "outputs left unwritten"
    err = oracle.max_rel_err(c, oracle.gemm_dequantized(ops))
    assert err <= oracle.FLOAT_TOL, f"max rel err {err:.3e}"

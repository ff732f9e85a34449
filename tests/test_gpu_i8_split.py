"""INT8 / W4A8 split along K over a thread-block cluster.

The "GEMM Optimization Guide" (section 1.3) asks small batches to stream the
weights with a large K tile; with a narrow N the strips of B rows alone
leave SMs idle, so the weight-streaming kernel splits each strip's K stages
over 2, 4 or 8 CTAs of a cluster and sums their int32 partials exactly through
distributed shared memory.  Integer sums do not depend on the order, so
every split must give the same bits as the oracle's exact product.

In-process cases take the library's own choice (narrow N: a split of 2, 4
or 8; the shapes are chosen so that each split occurs, with ragged M, several
row groups, ranks with unequal stage counts, and a last stage with fewer
than 8 K tiles).  A child process per forced split (GP_I8_SPLITK, read once
per process) runs shared inputs, the 16 x 7168 x 4096 workload included,
and must match bit for bit.
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
INT32_SENTINEL = -2 ** 31


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_preshuffle_gb300 import build
    build.build()
    gp.load_library()


def run(ops):
    A = torch.from_numpy(np.ascontiguousarray(ops.a)).cuda()
    Bp = gp.preshuffle_b(torch.from_numpy(np.ascontiguousarray(ops.b)).cuda(), ops.dtype)
    out = torch.full((ops.M, ops.N), INT32_SENTINEL, dtype=torch.int32, device="cuda")
    C = gp.matmul(A, Bp, ops.dtype, ops.N, ops.K, out=out)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    return C.cpu().numpy().astype(np.int64)


# (dtype, M, N, K) and the split the library takes for it on 152 SMs
# (16-row strips; a split keeps the grid within 3 CTAs an SM and gives each
# rank >= 2 stages of 8 K tiles).
AUTO = [
    ("int8", 16, 1024, 16384),   # 64 strips: split 4, 4 stages a rank
    ("int8", 16, 2048, 8192),    # 128 strips: split 2
    ("int8", 5, 1152, 4736),     # ragged M, 72 strips, 37 K tiles: split 2, ranks of 2 and 3 stages
    ("int8", 16, 1024, 7808),    # 61 K tiles: split 4, the last rank's last stage has 5 K tiles
    ("int8", 32, 1024, 8192),    # two row groups, 128 CTAs: split 2
    ("w4a8", 16, 1024, 8192),    # int4 weights: split 4
    ("w4a8", 7, 1152, 4864),     # int4, ragged M, 38 K tiles: split 2, the last stage has 6 K tiles
    ("int8", 16, 512, 16384),    # 32 strips: split 8 (the portable cluster limit), 2 stages a rank
    ("w4a8", 16, 512, 16384),    # int4 weights: split 8
]


@pytest.mark.parametrize("case", AUTO, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_split_k_bit_exact(case):
    dtype, M, N, K = case
    ops = inputs.make_operands(dtype, M, N, K, seed=90 + M + N // 8)
    c = run(ops)
    ref = oracle.gemm_operands(ops)
    assert np.array_equal(c, ref), f"{int((c != ref).sum())} mismatching int32 outputs"


@pytest.mark.parametrize("dtype", ["int8", "w4a8"])
def test_split_k_extremes(dtype):
    """Extreme codes and cancellation with the K range split 4 ways: every
    rank's partial carries its own offset correction (128 or 8 times its
    row sums of A), and the sum of the partials is the exact product."""
    M, N, K = 16, 1024, 16384
    a = np.full((M, K), -128, np.int8)
    rng = np.random.default_rng(5)
    a[1] = 127
    a[2, ::2] = 127                       # alternating signs: cancellation across the ranks' ranges
    a[3, : K // 2] = 127                  # one sign per half of K: the ranks' partials cancel
    a[4:] = rng.choice(np.array([-128, 127, 0, -1], np.int8), size=(M - 4, K))
    if dtype == "int8":
        b = np.full((N, K), -128, np.int8)
        b[1] = 127
        b[2:] = rng.choice(np.array([-128, 127, 0, 1], np.int8), size=(N - 2, K))
    else:
        b = np.full((N, K // 2), 0x88, np.uint8)  # every nibble -8
        b[1] = 0x77                                # every nibble 7
        b[2:] = rng.integers(0, 256, size=(N - 2, K // 2), dtype=np.uint8)
    ops = inputs.Operands(dtype, M, N, K, a, b)
    c = run(ops)
    ref = oracle.gemm_operands(ops)
    assert ref[0, 0] == K * 128 * (128 if dtype == "int8" else 8)
    assert np.array_equal(c, ref), f"{int((c != ref).sum())} mismatching int32 outputs"


FORCED = [("int8", 16, 7168, 4096), ("int8", 5, 1152, 4736), ("int8", 16, 512, 2176), ("w4a8", 16, 7168, 4096),
          ("w4a8", 9, 1152, 4864), ("int8", 16, 1024, 8192)]

CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np, torch
    import dense_gemm_preshuffle_gb300 as gp
    from dense_gemm_preshuffle_gb300 import inputs
    gp.load_library()
    out = {{}}
    for i, (dtype, M, N, K) in enumerate({cases!r}):
        ops = inputs.make_operands(dtype, M, N, K, seed=60 + i)
        A = torch.from_numpy(np.ascontiguousarray(ops.a)).cuda()
        Bp = gp.preshuffle_b(torch.from_numpy(np.ascontiguousarray(ops.b)).cuda(), dtype)
        C = torch.full((M, N), -2 ** 31, dtype=torch.int32, device="cuda")
        gp.matmul(A, Bp, dtype, N, K, out=C)
        torch.cuda.synchronize()
        assert gp.gemm_last_device_status() == 0
        out["c%d" % i] = C.cpu().numpy()
    np.savez({path!r}, **out)
""")


def run_forced(split, path):
    env = dict(os.environ)
    env.pop("GP_I8_STRIP", None)
    env["GP_I8_SPLITK"] = str(split)
    code = CHILD.format(root=ROOT, cases=FORCED, path=path)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return np.load(path)


def test_forced_splits_bit_identical(tmp_path):
    """Splits 1, 2, 4 and 8 forced on the same inputs: identical bits, and
    the oracle's exact product.  A split runs only where every rank gets a
    stage and, for 8, the strip has 16 rows (otherwise the case runs
    unsplit): 17 K tiles (3 stages) admit a split of 2 only, and 16 x 1024 x
    8192 (8 stages) a split of 8 with one stage a rank."""
    results = {s: run_forced(s, str(tmp_path / f"split{s}.npz")) for s in (1, 2, 4, 8)}
    for i, (dtype, M, N, K) in enumerate(FORCED):
        key = "c%d" % i
        ref = oracle.gemm_operands(inputs.make_operands(dtype, M, N, K, seed=60 + i))
        for s, res in results.items():
            c = res[key].astype(np.int64)
            assert np.array_equal(c, ref), f"{dtype} {M}x{N}x{K} split {s}: {int((c != ref).sum())} mismatches"

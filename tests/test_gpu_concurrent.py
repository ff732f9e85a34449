"""Products on several streams at once give the bits they give alone.

The kernels that coordinate the CTAs of a thread-block cluster (the 2-CTA
pairs, the two-pair K split, split-K over a cluster, the INT8 K split)
and the single-CTA kernels are launched together on four streams, several
times over, so that their CTAs share the GPU in varying ways.  Each output
must equal, bit for bit, the output of the same call run alone (the
kernels' results do not depend on scheduling), and each alone-run output is
checked against the oracle once.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_preshuffle_gb300 as gp
from dense_gemm_preshuffle_gb300 import inputs

pytestmark = pytest.mark.gpu

# (dtype, M, N, K) and the path the library takes on 152 SMs: the two-pair
# K split (32 tiles of 256 x 256), split-K over 2-CTA clusters (48 tiles,
# too many for one wave of 4-CTA clusters), the persistent pair kernel (81
# tiles), the INT8 K split over 4-CTA clusters (narrow N), the INT8 stream
# (wide N), MXFP4 pairs, and single-CTA 128 x 128 tiles (N = 384).
CASES = [("bf16", 512, 4096, 4096), ("bf16", 768, 4096, 4096), ("e4m3", 2304, 2304, 2048),
         ("int8", 16, 1024, 16384), ("int8", 16, 7168, 4096), ("e2m1", 512, 2048, 2048),
         ("bf16", 200, 384, 320)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_preshuffle_gb300 import build
    build.build()
    gp.load_library()


def prepare(case, seed):
    dtype, M, N, K = case
    ops = inputs.make_operands(dtype, M, N, K, seed=seed)

    def t(x):
        if x is None:
            return None
        if x.dtype == np.uint16:
            x = x.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    A, B, sa, sb = t(ops.a), t(ops.b), t(ops.scale_a), t(ops.scale_b)
    if dtype == "e2m1":
        Bp = gp.preshuffle_b(B, dtype, B_scales=sb)
        sb = None
    else:
        Bp = gp.preshuffle_b(B, dtype)
    cdt = torch.int32 if dtype == "int8" else torch.bfloat16

    def run(stream):
        out = torch.full((M, N), -2 ** 31 if cdt == torch.int32 else float("nan"), dtype=cdt, device="cuda")
        with torch.cuda.stream(stream):
            gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb, out=out, stream=stream)
        return out
    return ops, run


def test_concurrent_streams_bit_identical():
    torch.cuda.synchronize()
    preps = [prepare(c, 130 + i) for i, c in enumerate(CASES)]
    main = torch.cuda.current_stream()
    alone = []
    for ops, run in preps:
        c = run(main)
        torch.cuda.synchronize()
        assert gp.gemm_last_device_status() == 0
        alone.append(c.clone())
    # each alone-run output against the oracle
    for (ops, _), c in zip(preps, alone):
        ref = oracle.gemm_operands(ops)
        if ops.dtype == "int8":
            assert np.array_equal(c.cpu().numpy().astype(np.int64), ref)
        else:
            err = oracle.max_rel_err(c.float().cpu().numpy().astype(np.float64), ref)
            assert err <= oracle.FLOAT_TOL, f"{ops.dtype} {ops.M}x{ops.N}x{ops.K}: max rel err {err:.3e}"
    streams = [torch.cuda.Stream() for _ in range(4)]
    for rep in range(6):
        outs = []
        for i, (_, run) in enumerate(preps):
            # rotate the stream assignment so different products meet each round
            outs.append(run(streams[(i + rep) % len(streams)]))
        torch.cuda.synchronize()
        assert gp.gemm_last_device_status() == 0
        for (ops, _), c, ref in zip(preps, outs, alone):
            diff = int((c.view(torch.int32 if c.dtype == torch.int32 else torch.int16)
                        != ref.view(torch.int32 if ref.dtype == torch.int32 else torch.int16)).sum())
            assert diff == 0, f"round {rep}: {ops.dtype} {ops.M}x{ops.N}x{ops.K}: {diff} outputs differ from the run alone"

"""Failure detection without a GPU fault: a host-selected injection makes
the producer of one GEMM skip a stage load (each kernel in turn).  The MMA warp's bounded
wait then runs out after a short limit.  The kernel drains, frees its tensor
memory and exits.  The host reads GP_ERR_DEVICE_TIMEOUT, and the next normal
call on the same context passes parity.  It runs in a child process so the
short wait limit (read once per process) applies to it alone."""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys, time
    sys.path.insert(0, {root!r})
    import numpy as np, torch
    import dense_gemm_preshuffle_gb300 as gp
    import oracle
    from dense_gemm_preshuffle_gb300 import inputs
    gp.load_library()
    dtype, M, N, K = {case!r}
    ops = inputs.make_operands(dtype, M, N, K, seed=3)
    def t(x):
        if x is None:
            return None
        if x.dtype == np.uint16:
            x = x.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    A, B, sa, sb = t(ops.a), t(ops.b), t(ops.scale_a), t(ops.scale_b)
    if dtype == "e2m1":
        Bp = gp.preshuffle_b(B, dtype, B_scales=sb)
        run = lambda: gp.matmul(A, Bp, dtype, N, K, scale_a=sa)
    else:
        Bp = gp.preshuffle_b(B, dtype)
        run = lambda: gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    gp.gemm_debug_skip_load(3)
    t0 = time.time()
    run()
    st = gp.gemm_last_device_status()
    dt = time.time() - t0
    assert st == 6, f"expected GP_ERR_DEVICE_TIMEOUT, got {{st}}"
    assert dt < 20, dt
    C = run()
    assert gp.gemm_last_device_status() == 0
    rows = np.arange(min(M, 64))
    ref = oracle.gemm_operands(ops, rows=rows)
    if C.dtype == torch.int32:
        assert np.array_equal(C.cpu().numpy().astype(np.int64)[rows], ref)
        err = 0.0
    else:
        err = oracle.max_rel_err(C.float().cpu().numpy().astype(np.float64)[rows], ref)
        assert err <= oracle.FLOAT_TOL, err
    print(f"timeout reported after {{dt:.2f}} s; next call ok (max rel err {{err:.2e}})")
""")


# One case per kernel: the tcgen05 tile kernel (128 x 128 tiles), its 2-CTA
# pair form (256 x 256 tiles: both CTAs of every pair skip the stage), the
# INT8 weight-streaming kernel (its B producer skips the stage), the MXFP4
# kernel (M = 128) and its pair form (M = 200), the split-K cluster kernel
# (every CTA of every cluster skips the stage), and the INT8 kernel split
# along K over 4-CTA clusters (narrow N: every rank skips its stage, and all
# of them still meet at the cluster barriers of the reduction), and the
# K split over two pairs of CTAs (512 x 4096 x 4096: both pairs of every
# cluster skip the stage; the exchange and both cluster barriers still end).
CASES = [("e4m3", 256, 512, 1024), ("e4m3", 2048, 4096, 1024), ("int8", 16, 7168, 4096), ("e2m1", 128, 512, 2048),
         ("e2m1", 200, 512, 2048), ("bf16", 400, 4096, 8192), ("int8", 16, 1024, 16384), ("bf16", 512, 4096, 4096)]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_bounded_wait_timeout_reported_and_context_survives(case):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_preshuffle_gb300 import build
    build.build()
    env = dict(os.environ, GP_WAIT_LIMIT_MS="200")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, case=case)], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "next call ok" in r.stdout

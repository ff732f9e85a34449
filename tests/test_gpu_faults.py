"""Failure detection without a GPU fault: a host-selected injection makes
the producer of one tcgen05 GEMM skip a stage load.  The MMA warp's bounded
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
    ops = inputs.make_operands("e4m3", 256, 512, 1024, seed=3)
    A = torch.from_numpy(ops.a).cuda(); B = torch.from_numpy(ops.b).cuda()
    sa = torch.from_numpy(ops.scale_a).cuda(); sb = torch.from_numpy(ops.scale_b).cuda()
    Bp = gp.preshuffle_b(B, "e4m3")
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    gp.gemm_debug_skip_load(3)
    t0 = time.time()
    gp.matmul(A, Bp, "e4m3", ops.N, ops.K, sa, sb)
    st = gp.gemm_last_device_status()
    dt = time.time() - t0
    assert st == 6, f"expected GP_ERR_DEVICE_TIMEOUT, got {{st}}"
    assert dt < 20, dt
    C = gp.matmul(A, Bp, "e4m3", ops.N, ops.K, sa, sb)
    assert gp.gemm_last_device_status() == 0
    err = oracle.max_rel_err(C.float().cpu().numpy().astype(np.float64), oracle.gemm_operands(ops))
    assert err <= oracle.FLOAT_TOL, err
    print(f"timeout reported after {{dt:.2f}} s; next call ok (max rel err {{err:.2e}})")
""")


@pytest.mark.gpu
def test_bounded_wait_timeout_reported_and_context_survives():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_preshuffle_gb300 import build
    build.build()
    env = dict(os.environ, GP_WAIT_LIMIT_MS="200")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "next call ok" in r.stdout

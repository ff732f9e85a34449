"""K split over two pairs of CTAs (a 4-CTA cluster per 256 x 256 tile).

Each pair accumulates one half of K; the halves are summed in fp32 through
distributed shared memory before the epilogue.  The sum of two partial
chains rounds differently from one chain, so the results are compared with
the oracle at the float bound (not bit for bit with the other kernels), and
repeated launches must give identical bits (the exchange has a fixed
order: a + b rounds the same either way).

The library takes this kernel by default for few tiles and a long K (the
BF16 / FP16 512 x 4096 x 4096 workloads, whose every output the parity
tests in test_gpu_gemm.py compare).  Here GP_XPAIR=1 forces it, in a child
process (the switch is read once per process), on ragged M, an odd number
of K tiles (the halves differ by one and a stage straddles the split),
E4M3 with row / column scales, FP16, fused epilogues, more clusters than
fit at once, and K ranges of one or two K tiles a half.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

# (dtype, M, N, K, epilogue)
CASES = [("bf16", 512, 4096, 4096, "none"), ("bf16", 300, 512, 1088, "none"), ("e4m3", 200, 768, 2176, "none"),
         ("fp16", 129, 512, 960, "none"), ("bf16", 257, 512, 1024, "bias_gelu"), ("e4m3", 384, 1024, 4224, "bias"),
         ("bf16", 2000, 4096, 1088, "none"), ("fp16", 512, 1024, 8192, "bias_silu"),
         # the shortest K ranges: one K tile a half (2 tiles), one and two (3)
         ("bf16", 256, 256, 128, "none"), ("e4m3", 512, 512, 384, "bias_relu")]

CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np, torch
    import dense_gemm_preshuffle_gb300 as gp
    from dense_gemm_preshuffle_gb300 import inputs
    gp.load_library()
    out = {{}}
    for i, (dtype, M, N, K, epi) in enumerate({cases!r}):
        ops = inputs.make_operands(dtype, M, N, K, seed=70 + i)
        def t(x):
            if x is None:
                return None
            if x.dtype == np.uint16:
                x = x.view(np.int16)
            return torch.from_numpy(np.ascontiguousarray(x)).cuda()
        A, B, sa, sb = t(ops.a), t(ops.b), t(ops.scale_a), t(ops.scale_b)
        bias = None
        if epi != "none":
            bias = torch.from_numpy(np.linspace(-2.0, 2.0, N, dtype=np.float32)).cuda()
        Bp = gp.preshuffle_b(B, dtype)
        fdt = torch.float16 if dtype == "fp16" else torch.bfloat16
        runs = []
        for r in range(3):
            C = torch.full((M, N), float("nan"), dtype=fdt, device="cuda")
            gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb, epilogue=epi, bias=bias, out=C)
            torch.cuda.synchronize()
            assert gp.gemm_last_device_status() == 0
            runs.append(C.view(torch.int16).cpu().numpy())
        for r in range(1, 3):
            assert np.array_equal(runs[r], runs[0]), f"case {{i}}: run {{r}} differs from run 0"
        out["c%d" % i] = runs[0]
    np.savez({path!r}, **out)
""")


def test_two_pair_k_split_parity(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from dense_gemm_preshuffle_gb300 import build, inputs
    build.build()
    path = str(tmp_path / "xpair.npz")
    env = dict(os.environ, GP_XPAIR="1")
    for k in ("GP_TC_TILE", "GP_TC_PAIR", "GP_SPLITK", "GP_PAIR_KSPLIT"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, cases=CASES, path=path)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    res = np.load(path)
    for i, (dtype, M, N, K, epi) in enumerate(CASES):
        ops = inputs.make_operands(dtype, M, N, K, seed=70 + i)
        bias = np.linspace(-2.0, 2.0, N, dtype=np.float32).astype(np.float64)
        ref = oracle.apply_epilogue(oracle.gemm_operands(ops), epi, bias)
        raw = res["c%d" % i]
        c = torch.from_numpy(raw).view(torch.float16 if dtype == "fp16" else torch.bfloat16).float().numpy()
        assert not np.isnan(c).any(), f"{dtype} {M}x{N}x{K} {epi}: outputs left unwritten"
        err = oracle.max_rel_err(c.astype(np.float64), ref)
        assert err <= oracle.FLOAT_TOL, f"{dtype} {M}x{N}x{K} {epi}: max rel err {err:.3e}"

"""Tile shapes reorder the work, not the arithmetic.

The tile kernel can cover C with 256x256, 128x256 or 128x128 tiles.  The
128x128 shape stages two K tiles per ring slot.  Where a tile has more than
128 rows, the 256x256 shape runs as pairs of CTAs (one tcgen05 MMA over both
CTAs' halves), and so does the 128x128 shape, on 256x128 tiles, with
GP_TC_PAIR=1; GP_TC_PAIR=0 keeps the single-CTA kernel.  The MXFP4 kernel
runs 256x256 pairs, or 128x256 single-CTA tiles with GP_TC_PAIR=0 (the
"... single" runs).  Each output element still takes the same K steps,
in the same order, into the same fp32 accumulator.  The epilogue is per
element.  So, as the "GEMM Optimization Guide" asks of reorder-only changes,
every shape must give the same bits.

Each shape runs in its own child process, because the GP_TC_TILE and
GP_TC_PAIR overrides are read once per process.  The same seeded inputs are used each time, and
the outputs are compared bit for bit.  Each output is also checked against
the oracle.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (dtype, M, N, K, epilogue): ragged M, K tiles that leave a partial
# two-tile stage, and N a multiple of 256 so that every shape applies.
CASES = [("bf16", 300, 512, 1088, "none"), ("e4m3", 200, 768, 2176, "none"), ("fp16", 129, 512, 960, "none"),
         ("bf16", 257, 512, 1024, "bias_gelu"),
         # more 128x128 tiles than SMs: each persistent CTA (or pair) takes
         # several tiles and reuses both accumulator buffers; 17 K tiles
         ("bf16", 2000, 4096, 1088, "none"),
         # MXFP4 has one tile shape: 256x256 pairs, or 128x256 single-CTA
         # tiles with GP_TC_PAIR=0; more tiles than SMs, ragged M
         ("e2m1", 2500, 4096, 1024, "none"), ("e2m1", 300, 512, 2048, "bias_relu")]

CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np, torch
    import dense_gemm_preshuffle_gb300 as gp
    from dense_gemm_preshuffle_gb300 import inputs
    gp.load_library()
    out = {{}}
    for i, (dtype, M, N, K, epi) in enumerate({cases!r}):
        ops = inputs.make_operands(dtype, M, N, K, seed=40 + i)
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
        if dtype == "e2m1":  # B's block scales travel inside the packed B
            Bp = gp.preshuffle_b(B, dtype, B_scales=sb)
            C = gp.matmul(A, Bp, dtype, N, K, scale_a=sa, epilogue=epi, bias=bias)
        else:
            Bp = gp.preshuffle_b(B, dtype)
            C = gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb, epilogue=epi, bias=bias)
        torch.cuda.synchronize()
        assert gp.gemm_last_device_status() == 0
        out["c%d" % i] = C.view(torch.int16).cpu().numpy()
    np.savez({path!r}, **out)
""")


def run_shape(tile, path):
    env = dict(os.environ)
    env.pop("GP_TC_TILE", None)
    env.pop("GP_TC_PAIR", None)
    env.pop("GP_SPLITK", None)
    if tile is not None and tile.endswith(" single"):  # the single-CTA kernel, pairs off
        env["GP_TC_TILE"] = tile.split()[0]
        env["GP_TC_PAIR"] = "0"
    elif tile is not None and tile.endswith(" pair"):  # 2-CTA pairs for this shape too
        env["GP_TC_TILE"] = tile.split()[0]
        env["GP_TC_PAIR"] = "1"
    elif tile is not None:
        env["GP_TC_TILE"] = tile
    code = CHILD.format(root=ROOT, cases=CASES, path=path)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return np.load(path)


@pytest.mark.gpu
def test_tile_shapes_are_bit_identical(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from dense_gemm_preshuffle_gb300 import build, inputs
    build.build()
    results = {tile: run_shape(tile, str(tmp_path / f"{tile}.npz"))
               for tile in (None, "256x256", "128x256", "128x128", "256x256 single", "128x128 pair")}
    base = results[None]
    for i, (dtype, M, N, K, epi) in enumerate(CASES):
        key = "c%d" % i
        for tile, res in results.items():
            diff = int((res[key] != base[key]).sum())
            assert diff == 0, f"{dtype} {M}x{N}x{K} {epi}: {diff} outputs differ between {tile} and the default tile"
        # and the common result passes parity against the oracle
        ops = inputs.make_operands(dtype, M, N, K, seed=40 + i)
        bias = np.linspace(-2.0, 2.0, N, dtype=np.float32).astype(np.float64)
        ref = oracle.apply_epilogue(oracle.gemm_operands(ops), epi, bias)
        raw = base[key]
        c = torch.from_numpy(raw).view(torch.float16 if dtype == "fp16" else torch.bfloat16).float().numpy()
        err = oracle.max_rel_err(c.astype(np.float64), ref)
        assert err <= oracle.FLOAT_TOL, f"{dtype} {M}x{N}x{K} {epi}: max rel err {err:.3e}"

"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

The tolerance metric is max |C - C_ref| / (|C_ref| + 1e-2) <= 8e-3 for bf16
outputs, and INT8 must be bit-exact.  Inputs come from the seeded generator
shared with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_preshuffle_gb300 as gp
from dense_gemm_preshuffle_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 8e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_preshuffle_gb300 import build
    build.build()
    gp.load_library()


def dev(ops):
    """Device tensors of an Operands bundle (raw bytes / codes)."""
    def t(x):
        if x is None:
            return None
        if x.dtype == np.uint16:
            x = x.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t(ops.a), t(ops.b), t(ops.scale_a), t(ops.scale_b)


# Sentinels an output buffer is filled with before every GPU call, so that an
# output the kernel never writes fails the comparison: NaN for float outputs,
# and INT32_MIN for int32 ones (no exact INT8/W4A8 result the library accepts
# reaches -2^31: |C| <= K * 128 * 128 < 2^31 for K <= 130944).
INT32_SENTINEL = -2 ** 31


def sentinel_out(M, N, dtype):
    if dtype in ("int8", "w4a8"):
        return torch.full((M, N), INT32_SENTINEL, dtype=torch.int32, device="cuda")
    fdt = torch.float16 if dtype == "fp16" else torch.bfloat16  # the default output of each type
    return torch.full((M, N), float("nan"), dtype=fdt, device="cuda")


def gpu_gemm(ops, out=None):
    if out is None:
        out = sentinel_out(ops.M, ops.N, ops.dtype)
    A, B, sa, sb = dev(ops)
    if ops.dtype == "e2m1":
        Bp = gp.preshuffle_b(B, "e2m1", B_scales=sb)
        C = gp.matmul(A, Bp, "e2m1", ops.N, ops.K, scale_a=sa, out=out)
    else:
        Bp = gp.preshuffle_b(B, ops.dtype)
        C = gp.matmul(A, Bp, ops.dtype, ops.N, ops.K, scale_a=sa, scale_b=sb, out=out)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    return C


def as_host(C):
    if C.dtype == torch.int32:
        return C.cpu().numpy().astype(np.int64)
    return C.float().cpu().numpy().astype(np.float64)


def reference(ops, rows=None):
    """The oracle's C: the plain loops for small products, the full-size
    dequantized matmul (same values, see oracle.gemm_dequantized) for large
    ones."""
    work = (len(rows) if rows is not None else ops.M) * ops.N * ops.K
    if work > (1 << 31) and ops.dtype not in ("int8", "w4a8"):
        return oracle.gemm_dequantized(ops, rows=rows)
    return oracle.gemm_operands(ops, rows=rows)


def check(ops, C, rows=None):
    c = as_host(C)
    ref = reference(ops, rows=rows)
    if rows is not None:
        c = c[rows]
    if ops.dtype in ("int8", "w4a8"):
        assert np.array_equal(c, ref), f"{int((c != ref).sum())} mismatching int32 outputs"
    else:
        err = oracle.max_rel_err(c, ref)
        assert err <= TOL, f"max rel err {err:.3e}"
        return err


def abs_sum_diagnostic(ops, C, rows=None):
    """max |C - C_ref| / sum_k |a||b| on the given rows, against its bound:
    output rounding (2^-9 bf16, 2^-11 fp16) plus K 2^-24 for an fp32
    accumulation and a few ulps of fp32 scaling."""
    c = as_host(C)
    if rows is not None:
        c = c[rows]
    d = oracle.max_err_over_abs(c, oracle.gemm_operands(ops, rows=rows), oracle.gemm_abs_operands(ops, rows=rows))
    out_ulp = 2.0 ** -11 if C.dtype == torch.float16 else 2.0 ** -9
    bound = out_ulp + ops.K * 2.0 ** -24 + 2.0 ** -21
    print(f"{ops.dtype} {ops.M}x{ops.N}x{ops.K}: max |C-C_ref| / sum|a||b| = {d:.3e} (bound {bound:.3e})")
    assert d <= bound
    return d


# ---------------------------------------------------------------- packing

@pytest.mark.parametrize("dtype,N,K", [("e4m3", 256, 512), ("int8", 384, 1024), ("bf16", 128, 192),
                                       ("e2m1", 256, 1024), ("int8", 7168, 4096), ("fp16", 256, 320),
                                       ("w4a8", 384, 1024), ("w4a8", 7168, 4096)])
def test_pack_matches_oracle_layout_and_roundtrips(dtype, N, K):
    ops = inputs.make_operands(dtype, 1, N, K, seed=123)
    _, B, _, sb = dev(ops)
    Bp = gp.preshuffle_b(B, dtype, B_scales=sb if dtype == "e2m1" else None)
    expect = oracle.pack_b(ops.b, dtype, scales=ops.scale_b)
    assert np.array_equal(Bp.cpu().numpy(), expect)
    back = torch.empty_like(B)
    back_s = torch.empty_like(sb) if dtype == "e2m1" else None
    gp.gemm_unpack_b(Bp, dtype, N, K, back, back_s)
    torch.cuda.synchronize()
    assert torch.equal(back, B)
    if dtype == "e2m1":
        assert torch.equal(back_s, sb)


# ---------------------------------------------------------------- small and ragged shapes

SMALL = [
    ("e4m3", 1, 128, 128), ("e4m3", 300, 512, 1024), ("e4m3", 129, 256, 256), ("e4m3", 17, 384, 640),
    ("e4m3", 1000, 1024, 512),
    ("bf16", 257, 384, 512), ("bf16", 128, 128, 64), ("bf16", 64, 256, 4096), ("bf16", 700, 640, 320),
    ("int8", 1, 128, 128), ("int8", 37, 256, 384), ("int8", 16, 384, 256), ("int8", 100, 1152, 1280),
    ("int8", 16, 7168, 4096),
    ("e2m1", 1, 256, 256), ("e2m1", 200, 512, 512), ("e2m1", 129, 256, 1024), ("e2m1", 300, 768, 2048),
    ("fp16", 1, 128, 64), ("fp16", 257, 384, 512), ("fp16", 64, 256, 4096), ("fp16", 700, 640, 320),
    ("w4a8", 1, 128, 256), ("w4a8", 37, 256, 512), ("w4a8", 16, 384, 256), ("w4a8", 100, 1152, 1280),
    ("w4a8", 16, 7168, 4096),
]


@pytest.mark.parametrize("dtype,M,N,K", SMALL, ids=lambda v: str(v))
def test_small_and_ragged(dtype, M, N, K):
    ops = inputs.make_operands(dtype, M, N, K, seed=1000 + M + N + K)
    check(ops, gpu_gemm(ops))


def test_mxfp4_single_hot_scale_blocks():
    """Every element 1.0 and every scale 2^-127 except one (row, block) per
    probe: C shows exactly which output row and K block each A scale reaches."""
    M, N, K = 128, 256, 512
    a = np.full((M, K // 2), 0x22, np.uint8)   # E2M1 1.0 in both nibbles
    b = np.full((N, K // 2), 0x22, np.uint8)
    rng = np.random.default_rng(4)
    ea = np.zeros((M, K // 32), np.uint8)
    eb = np.full((N, K // 32), 127, np.uint8)
    for m in range(M):
        ea[m, rng.integers(0, K // 32)] = 127 + (m % 5)
    ops = inputs.Operands("e2m1", M, N, K, a, b, ea, eb)
    check(ops, gpu_gemm(ops))
    ea2 = np.full((M, K // 32), 127, np.uint8)
    eb2 = np.zeros((N, K // 32), np.uint8)
    for n in range(N):
        eb2[n, rng.integers(0, K // 32)] = 126 + (n % 7)
    ops2 = inputs.Operands("e2m1", M, N, K, a, b, ea2, eb2)
    check(ops2, gpu_gemm(ops2))


def test_e4m3_without_scales():
    ops = inputs.make_operands("e4m3", 200, 256, 384, seed=5)
    ops.scale_a = ops.scale_b = None
    check(ops, gpu_gemm(ops))


# ---------------------------------------------------------------- the five workloads

def sample_rows(M, n=32, seed=0):
    rng = np.random.default_rng(seed)
    r = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    r.update({0, M - 1})
    return np.array(sorted(r))


@pytest.mark.parametrize("name", ["fp8_128x256x512", "int8_16x7168x4096", "bf16_512x4096x4096",
                                  "w4a8_16x7168x4096"])
def test_workload_full_compare(name):
    ops = inputs.workload_operands(name)
    C = gpu_gemm(ops)
    check(ops, C)
    if ops.dtype not in ("int8", "w4a8"):
        abs_sum_diagnostic(ops, C, rows=sample_rows(ops.M, 64, seed=2))


@pytest.mark.parametrize("name", ["fp8_8192x8192x8192", "mxfp4_4096x8192x8192", "fp8_5120x5120x8320",
                                  "fp16_512x4096x4096"])
def test_workload_full_compare_large(name):
    """Every output of the large products against the oracle at the G10
    bound (the output starts as NaN, so a tile never written fails)."""
    ops = inputs.workload_operands(name)
    C = gpu_gemm(ops)
    check(ops, C)
    abs_sum_diagnostic(ops, C, rows=sample_rows(ops.M, 24, seed=1))


@pytest.mark.parametrize("dtype", ["e4m3", "bf16", "fp16"])
def test_tile256_path_ragged(dtype):
    # enough 256 x 256 tiles (17 x 38 >= 4 per SM) to take the 256-row tile
    # path, with a ragged last row band
    ops = inputs.make_operands(dtype, 4173, 9728, 256, seed=31)
    C = gpu_gemm(ops)
    check(ops, C)


@pytest.mark.parametrize("dtype,M,N,K", [("bf16", 400, 4096, 8192), ("e4m3", 300, 8192, 8192),
                                         ("fp16", 400, 4096, 8192)])
def test_split_k_cluster_path_ragged(dtype, M, N, K):
    # few 256 x 256 tiles and a long K: K is split across a 4- (bf16) or
    # 2-CTA (e4m3) cluster and reduced over distributed shared memory
    ops = inputs.make_operands(dtype, M, N, K, seed=37)
    C = gpu_gemm(ops)
    check(ops, C)


def test_split_k_exchange_repeatable():
    """The split-K reduce-scatter hands blocks between CTAs through staging
    buffers that are reused once the owner acknowledges them.  A buffer
    reused too early would hand a peer a wrong partial in some runs only;
    50 runs into NaN-filled outputs must all be bit-identical to the first,
    which matches the oracle on every output."""
    ops = inputs.make_operands("bf16", 400, 4096, 8192, seed=41)
    A, B, _, _ = dev(ops)
    Bp = gp.preshuffle_b(B, "bf16")
    outs = []
    for i in range(50):
        C = sentinel_out(ops.M, ops.N, "bf16")
        gp.matmul(A, Bp, "bf16", ops.N, ops.K, out=C, b_constant=(i % 2 == 1))
        outs.append(C)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    first = outs[0].view(torch.int16)
    for i, C in enumerate(outs[1:]):
        assert torch.equal(C.view(torch.int16), first), f"run {i + 1} differs"
    check(ops, outs[0])


# ---------------------------------------------------------------- edge cases

def test_int8_extremes_bit_exact():
    M, N, K = 16, 256, 4096
    a = np.full((M, K), -128, np.int8)
    b = np.full((N, K), -128, np.int8)
    a[1] = 127
    b[1] = 127
    a[2, ::2] = 127          # alternating signs: large cancellation
    b[2, 1::2] = -127
    rng = np.random.default_rng(0)
    a[3:] = rng.choice(np.array([-128, 127, 0, 1, -1], np.int8), size=(M - 3, K))
    ops = inputs.Operands("int8", M, N, K, a, b)
    check(ops, gpu_gemm(ops))


@pytest.mark.parametrize("dtype,K", [("int8", 130944), ("w4a8", 2096896)])
def test_integer_extremes_at_the_k_limit(dtype, K):
    """The largest K the ABI accepts: all -128 (x -128 or x -8) sums to just
    below 2^31, and the exact int32 result survives every partial sum."""
    M, N = 16, 256
    a = np.full((M, K), -128, np.int8)
    rng = np.random.default_rng(1)
    a[1] = 127
    a[2:] = rng.choice(np.array([-128, 127, 0, -1], np.int8), size=(M - 2, K))
    if dtype == "int8":
        b = np.full((N, K), -128, np.int8)
        b[1] = 127
    else:
        b = np.full((N, K // 2), 0x88, np.uint8)  # every nibble -8
        b[1] = 0x77                                # every nibble 7
    ops = inputs.Operands(dtype, M, N, K, a, b)
    C = gpu_gemm(ops)
    rows = np.arange(M)
    ref = oracle.gemm_operands(ops, rows=rows)
    assert ref[0, 0] == K * 128 * (128 if dtype == "int8" else 8) and ref[0, 0] < 2**31
    check(ops, C)


def test_int8_more_row_groups_than_one_grid():
    """M past 65535 groups of 16 rows: the launcher splits the row groups
    over launches; rows on both sides of the split are checked."""
    M, N, K = 16 * 65537, 128, 256
    ops = inputs.make_operands("int8", M, N, K, seed=77)
    C = gpu_gemm(ops)
    split = 16 * 65535
    rows = np.unique(np.concatenate([np.arange(16), np.arange(split - 16, split + 32), [M - 1],
                                     np.random.default_rng(3).choice(M, 64, replace=False)]))
    check(ops, C, rows=rows)


def test_w4a8_extremes_bit_exact():
    M, N, K = 16, 256, 4096
    a = np.full((M, K), -128, np.int8)
    b = np.full((N, K), -8, np.int8)
    a[1] = 127
    b[1] = 7
    a[2, ::2] = 127                       # alternating signs: large cancellation
    b[2, 1::2] = -7
    rng = np.random.default_rng(1)
    a[3:] = rng.choice(np.array([-128, 127, 0, 1, -1], np.int8), size=(M - 3, K))
    b[3:] = rng.choice(np.array([-8, 7, 0, 1, -1], np.int8), size=(N - 3, K))
    nib = (b.astype(np.int16) & 0xF).astype(np.uint8)
    bp = nib[:, 0::2] | (nib[:, 1::2] << 4)
    ops = inputs.Operands("w4a8", M, N, K, a, bp)
    check(ops, gpu_gemm(ops))


def test_k_zero_gives_zeros():
    C = torch.full((5, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    gp.gemm_run(dummy, dummy, "bf16", 5, 128, 0, "none", None, None, C, "bf16")
    torch.cuda.synchronize()
    assert (C == 0).all()


def test_guard_bands_untouched():
    ops = inputs.make_operands("e4m3", 77, 256, 512, seed=9)
    M, N = ops.M, ops.N
    guard = 4096
    buf = torch.full((M * N + 2 * guard,), -3.0, dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + M * N].view(M, N)
    gpu_gemm(ops, out=C)
    assert (buf[:guard] == -3.0).all() and (buf[guard + M * N:] == -3.0).all()
    check(ops, C)
    ops8 = inputs.make_operands("int8", 19, 384, 256, seed=9)
    buf8 = torch.full((19 * 384 + 2 * guard,), -7, dtype=torch.int32, device="cuda")
    C8 = buf8[guard:guard + 19 * 384].view(19, 384)
    gpu_gemm(ops8, out=C8)
    assert (buf8[:guard] == -7).all() and (buf8[guard + 19 * 384:] == -7).all()
    check(ops8, C8)


def test_int8_partial_last_strip_guard_bands():
    # 7168 rows of B split into 48-row strips leave a 16-row last strip
    ops = inputs.make_operands("int8", 16, 7168, 1024, seed=21)
    M, N = ops.M, ops.N
    guard = 8192
    buf = torch.full((M * N + 2 * guard,), -5, dtype=torch.int32, device="cuda")
    C = buf[guard:guard + M * N].view(M, N)
    gpu_gemm(ops, out=C)
    assert (buf[:guard] == -5).all() and (buf[guard + M * N:] == -5).all()
    check(ops, C)


def test_repeatable_bitwise():
    ops = inputs.make_operands("e4m3", 512, 1024, 1024, seed=2)
    A, B, sa, sb = dev(ops)
    Bp = gp.preshuffle_b(B, "e4m3")
    first = gp.matmul(A, Bp, "e4m3", ops.N, ops.K, sa, sb)
    for _ in range(20):
        again = gp.matmul(A, Bp, "e4m3", ops.N, ops.K, sa, sb)
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    ops8 = inputs.make_operands("int8", 16, 7168, 4096, seed=3)
    A8, B8, _, _ = dev(ops8)
    Bp8 = gp.preshuffle_b(B8, "int8")
    f8 = gp.matmul(A8, Bp8, "int8", ops8.N, ops8.K)
    for _ in range(20):
        assert torch.equal(gp.matmul(A8, Bp8, "int8", ops8.N, ops8.K), f8)


# ---------------------------------------------------------------- constant-weight scheduling flag

@pytest.mark.parametrize("dtype,M,N,K", [
    ("int8", 16, 7168, 4096), ("int8", 37, 256, 384), ("int8", 16, 384, 128),
    ("w4a8", 16, 7168, 4096), ("w4a8", 37, 256, 512),
    ("e4m3", 300, 512, 1024), ("e4m3", 17, 384, 256), ("bf16", 257, 384, 512),
    ("e2m1", 200, 512, 512), ("e2m1", 129, 256, 256),
    ("bf16", 400, 4096, 8192),   # split-K cluster path
    ("e4m3", 4173, 9728, 256),   # 256-row tile path
], ids=lambda v: str(v))
def test_b_constant_flag_matches_oracle_and_default(dtype, M, N, K):
    """GP_RUN_B_CONSTANT only moves the first B requests before the wait on
    the previous kernel: the result is bit-identical to the default call."""
    ops = inputs.make_operands(dtype, M, N, K, seed=4000 + M + N + K)
    A, B, sa, sb = dev(ops)
    if dtype == "e2m1":
        Bp = gp.preshuffle_b(B, "e2m1", B_scales=sb)
        sa_, sb_ = sa, None
    else:
        Bp = gp.preshuffle_b(B, dtype)
        sa_, sb_ = sa, sb
    torch.cuda.synchronize()   # the weights are complete before any flagged call
    ref = gp.matmul(A, Bp, dtype, N, K, scale_a=sa_, scale_b=sb_)
    for _ in range(3):
        C = gp.matmul(A, Bp, dtype, N, K, scale_a=sa_, scale_b=sb_, b_constant=True)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    if C.dtype == torch.int32:
        assert torch.equal(C, ref)
    else:
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    check(ops, C)


@pytest.mark.parametrize("M,N1,K1,N2", [(2048, 2048, 4096, 384), (400, 8192, 2048, 4096)])
def test_b_constant_reads_a_only_after_previous_kernel(M, N1, K1, N2):
    """Chain C2 = (A.B1^T).B2^T with the second call flagged: its A is the
    first call's output, so an early read of A would see the fill value."""
    ops1 = inputs.make_operands("bf16", M, N1, K1, seed=77)
    ops2 = inputs.make_operands("bf16", M, N2, N1, seed=78)
    A1, B1, _, _ = dev(ops1)
    _, B2, _, _ = dev(ops2)
    Bp1 = gp.preshuffle_b(B1, "bf16")
    Bp2 = gp.preshuffle_b(B2, "bf16")
    torch.cuda.synchronize()
    for trial in range(3):
        C1 = torch.full((M, N1), float("nan"), dtype=torch.bfloat16, device="cuda")
        gp.matmul(A1, Bp1, "bf16", N1, K1, out=C1)
        C2 = gp.matmul(C1, Bp2, "bf16", N2, N1, b_constant=True)
        torch.cuda.synchronize()
        assert torch.isfinite(C2.float()).all()
        again = gp.matmul(C1, Bp2, "bf16", N2, N1)  # C1 complete: the plain call
        torch.cuda.synchronize()
        assert torch.equal(C2.view(torch.int16), again.view(torch.int16))
    check(ops1, C1, rows=sample_rows(M, 16, seed=6))


# ---------------------------------------------------------------- independent-call scheduling flag

@pytest.mark.parametrize("dtype,M,N,K", [
    ("int8", 16, 7168, 4096), ("int8", 37, 256, 384), ("int8", 16, 384, 128),
    ("w4a8", 16, 7168, 4096), ("w4a8", 37, 256, 512),
    ("e4m3", 300, 512, 1024), ("bf16", 257, 384, 512),   # tcgen05 kernels: taken as B constant
], ids=lambda v: str(v))
def test_independent_run_matches_default(dtype, M, N, K):
    """A run of GP_RUN_INDEPENDENT calls on weights and outputs of their own
    overlaps the calls; every output is bit-identical to the plain call."""
    ops = inputs.make_operands(dtype, M, N, K, seed=4100 + M + N + K)
    A, B, sa, sb = dev(ops)
    Bp = gp.preshuffle_b(B, dtype)
    copies = [Bp] + [Bp.clone() for _ in range(3)]
    torch.cuda.synchronize()
    ref = gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb)
    torch.cuda.synchronize()
    for trial in range(2):
        outs = [gp.matmul(A, copies[i % 4], dtype, N, K, scale_a=sa, scale_b=sb, independent=True)
                for i in range(12)]
        torch.cuda.synchronize()
        assert gp.gemm_last_device_status() == 0
        for C in outs:
            if C.dtype == torch.int32:
                assert torch.equal(C, ref)
            else:
                assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    check(ops, outs[-1])


def test_independent_run_keeps_stream_order():
    """A long plain INT8 call writes C_a; three short independent calls
    follow; then a plain call reads C_a (its bytes as int8 activations).
    The independent calls wait for their predecessor before exiting, so the
    last call's wait on them also covers C_a."""
    Ma, Na, Ka = 16, 7168, 65536
    opsa = inputs.make_operands("int8", Ma, Na, Ka, seed=91)
    Aa, Ba, _, _ = dev(opsa)
    Bpa = gp.preshuffle_b(Ba, "int8")
    opsb = inputs.make_operands("int8", 16, 384, 256, seed=92)
    Ab, Bb, _, _ = dev(opsb)
    Bpb = gp.preshuffle_b(Bb, "int8")
    Kc, Nc = 4 * Na, 256
    opsc = inputs.make_operands("int8", Ma, Nc, Kc, seed=93)
    _, Bc, _, _ = dev(opsc)
    Bpc = gp.preshuffle_b(Bc, "int8")
    torch.cuda.synchronize()
    ref_b = gp.matmul(Ab, Bpb, "int8", 384, 256)
    for trial in range(3):
        Ca = torch.full((Ma, Na), 0x7F7F7F7F, dtype=torch.int32, device="cuda")
        gp.matmul(Aa, Bpa, "int8", Na, Ka, out=Ca, b_constant=True)
        outs_b = [gp.matmul(Ab, Bpb, "int8", 384, 256, independent=True) for _ in range(3)]
        Cc = gp.matmul(Ca.view(torch.int8), Bpc, "int8", Nc, Kc, b_constant=True)
        torch.cuda.synchronize()
        assert gp.gemm_last_device_status() == 0
        again = gp.matmul(Ca.view(torch.int8), Bpc, "int8", Nc, Kc)
        torch.cuda.synchronize()
        assert torch.equal(Cc, again)
        for C in outs_b:
            assert torch.equal(C, ref_b)
    # C_a itself, on a few columns, against the oracle
    cols = np.arange(0, Na, 997)
    want = (opsa.a.astype(np.int64) @ opsa.b[cols].astype(np.int64).T)
    assert np.array_equal(Ca.cpu().numpy()[:, cols].astype(np.int64), want)


# ---------------------------------------------------------------- fused epilogues

EPI_SHAPES = [("bf16", 257, 384, 512), ("e4m3", 300, 512, 1024), ("e2m1", 200, 512, 512), ("e4m3", 17, 256, 256),
              ("e4m3", 4173, 9728, 256),   # 256-row tile path
              ("bf16", 400, 4096, 8192)]   # split-K cluster path


@pytest.mark.parametrize("epilogue", ["bias", "bias_relu", "bias_silu", "bias_gelu"])
@pytest.mark.parametrize("dtype,M,N,K", EPI_SHAPES, ids=lambda v: str(v))
def test_fused_epilogue(dtype, M, N, K, epilogue):
    """C = act(A.B^T scaled + bias[n]) against the oracle's fp64 epilogue."""
    ops = inputs.make_operands(dtype, M, N, K, seed=5000 + M + N + K)
    plain = reference(ops)
    rng = np.random.default_rng(M + N)
    bias = (rng.standard_normal(N) * plain.std()).astype(np.float32)
    A, B, sa, sb = dev(ops)
    if dtype == "e2m1":
        Bp = gp.preshuffle_b(B, "e2m1", B_scales=sb)
        C = gp.matmul(A, Bp, "e2m1", N, K, scale_a=sa, epilogue=epilogue, bias=torch.from_numpy(bias).cuda(),
                      out=sentinel_out(M, N, dtype))
    else:
        Bp = gp.preshuffle_b(B, dtype)
        C = gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb, epilogue=epilogue,
                      bias=torch.from_numpy(bias).cuda(), out=sentinel_out(M, N, dtype))
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    c = as_host(C)
    ref = oracle.apply_epilogue(plain, epilogue, bias.astype(np.float64))
    err = oracle.max_rel_err(c, ref)
    assert err <= TOL, f"max rel err {err:.3e}"


@pytest.mark.parametrize("epilogue", ["bias", "bias_relu", "bias_silu", "bias_gelu"])
def test_fused_epilogue_empty_sum(epilogue):
    # K == 0: the product is zero, every row is act(bias)
    M, N = 5, 256
    bias = np.linspace(-6, 6, N).astype(np.float32)
    C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    gp.gemm_run_ex(dummy, dummy, "bf16", M, N, 0, "none", None, None, epilogue, torch.from_numpy(bias).cuda(), C,
                   "bf16")
    torch.cuda.synchronize()
    ref = oracle.apply_epilogue(np.zeros((M, N)), epilogue, bias.astype(np.float64))
    assert oracle.max_rel_err(as_host(C), ref) <= TOL



# ---------------------------------------------------------------- fp16 output

@pytest.mark.parametrize("dtype,M,N,K", [("fp16", 300, 512, 1024), ("bf16", 200, 384, 512), ("e4m3", 129, 256, 512),
                                         ("e2m1", 200, 512, 512), ("fp16", 4173, 9728, 256)])
def test_fp16_output(dtype, M, N, K):
    """IEEE fp16 output (RNE from fp32) from every float path."""
    ops = inputs.make_operands(dtype, M, N, K, seed=6000 + M + N + K)
    A, B, sa, sb = dev(ops)
    if dtype == "e2m1":
        Bp = gp.preshuffle_b(B, "e2m1", B_scales=sb)
        C = gp.matmul(A, Bp, "e2m1", N, K, scale_a=sa, out_dtype="fp16")
    else:
        Bp = gp.preshuffle_b(B, dtype)
        C = gp.matmul(A, Bp, dtype, N, K, scale_a=sa, scale_b=sb, out_dtype="fp16")
    torch.cuda.synchronize()
    assert C.dtype == torch.float16 and gp.gemm_last_device_status() == 0
    check(ops, C)


@pytest.mark.parametrize("epilogue", ["bias_gelu", "bias_silu"])
def test_fp16_output_with_epilogue(epilogue):
    ops = inputs.make_operands("fp16", 257, 384, 512, seed=71)
    plain = oracle.gemm_operands(ops)
    bias = (np.random.default_rng(3).standard_normal(384) * plain.std()).astype(np.float32)
    A, B, _, _ = dev(ops)
    Bp = gp.preshuffle_b(B, "fp16")
    C = gp.matmul(A, Bp, "fp16", 384, 512, epilogue=epilogue, bias=torch.from_numpy(bias).cuda())
    torch.cuda.synchronize()
    ref = oracle.apply_epilogue(plain, epilogue, bias.astype(np.float64))
    assert oracle.max_rel_err(as_host(C), ref) <= TOL
    # K = 0 broadcast into fp16
    Cz = torch.full((3, 384), 7.0, dtype=torch.float16, device="cuda")
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    gp.gemm_run_ex(dummy, dummy, "fp16", 3, 384, 0, "none", None, None, epilogue, torch.from_numpy(bias).cuda(), Cz,
                   "fp16")
    torch.cuda.synchronize()
    assert oracle.max_rel_err(as_host(Cz), oracle.apply_epilogue(np.zeros((3, 384)), epilogue,
                                                                 bias.astype(np.float64))) <= TOL

"""Pins of the CPU oracle against things other than itself.

- Codecs: torch's float8_e4m3fn / bfloat16 decodes (library routines) and the
  OCP E2M1 table (tests/golden/).
- GEMMs: brute force in exact rational arithmetic (fractions.Fraction) on tiny
  shapes, numpy's int64 matmul, identity and permutation operands, and the
  block-scaled form reducing to the plain one when every scale is 1.
- Bookkeeping: the numbers the "GEMM Optimization Guide" prints
  (tests/golden/).
- Pack model: round trips and layout invariants.

The last group plants mistakes in the oracle, on the CPU, and checks that
some pin fails for each one.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_preshuffle_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- codecs

def torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch_all_codes():
    ref = torch_e4m3_values()
    got = oracle.decode_e4m3(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def load_e2m1_golden():
    vals = {}
    for line in open(os.path.join(GOLDEN, "ocp_e2m1_values.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, v = line.split()
        vals[int(c)] = float(v)
    return vals


def test_e2m1_decode_matches_ocp_table():
    table = load_e2m1_golden()
    got = oracle.decode_e2m1(np.arange(16, dtype=np.uint8))
    for c in range(16):
        assert got[c] == table[c], c
        assert np.signbit(got[c]) == np.signbit(table[c]) or table[c] == 0.0


def test_ue8m0_decode():
    got = oracle.decode_ue8m0(np.arange(256, dtype=np.uint8))
    assert got[127] == 1.0 and got[128] == 2.0 and got[126] == 0.5
    assert got[0] == float.fromhex("0x1p-127") and got[254] == float.fromhex("0x1p+127")
    assert np.isnan(got[255])
    assert np.all(got[1:255] == 2.0 * got[0:254])


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=100000, dtype=np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode_bf16(bits)
    nan = np.isnan(t)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], t[~nan])


# ---------------------------------------------------------------- GEMMs

def frac_gemm(a_vals, b_vals):
    """Exact C[m][n] = sum_k a[m][k] * b[n][k] over Fractions (pure Python)."""
    M, K = len(a_vals), len(a_vals[0])
    N = len(b_vals)
    return [[sum((a_vals[m][k] * b_vals[n][k] for k in range(K)), Fraction(0)) for n in range(N)]
            for m in range(M)]


def to_frac(x):
    return [[Fraction(float(v)) for v in row] for row in np.asarray(x, np.float64)]


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (8, 8, 64), (2, 9, 33)])
def test_int8_bruteforce_and_numpy(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    a = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    b = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    got = oracle.gemm_int8(a, b)
    brute = [[sum(int(a[m, k]) * int(b[n, k]) for k in range(K)) for n in range(N)] for m in range(M)]
    assert got.tolist() == brute
    assert np.array_equal(got, a.astype(np.int64) @ b.astype(np.int64).T)


def test_int8_extremes_fit_int32():
    # max |C| for the small-batch workload's K=4096: 4096 * 128^2 < 2^31
    K = 4096
    a = np.full((2, K), -128, dtype=np.int8)
    b = np.full((3, K), -128, dtype=np.int8)
    b[1] = 127
    got = oracle.gemm_int8(a, b)
    assert got[0, 0] == K * 128 * 128 and got[0, 1] == -K * 128 * 127
    assert abs(int(got.max())) < 2 ** 31


@pytest.mark.parametrize("M,N,K", [(3, 4, 64), (8, 8, 64), (5, 3, 96)])
def test_e4m3_rowcol_vs_fraction(M, N, K):
    ops = inputs.make_operands("e4m3", M, N, K, seed=7 + M)
    vals = torch_e4m3_values()  # library decode
    qa = to_frac(vals[ops.a])
    qb = to_frac(vals[ops.b])
    acc = frac_gemm(qa, qb)
    got = oracle.gemm_operands(ops)
    for m in range(M):
        for n in range(N):
            exact = acc[m][n] * Fraction(float(ops.scale_a[m])) * Fraction(float(ops.scale_b[n]))
            # the unscaled sum is exact in fp64; two scalings each round once
            assert abs(Fraction(got[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 51)


@pytest.mark.parametrize("M,N,K", [(3, 4, 16), (4, 2, 40)])
def test_bf16_vs_fraction(M, N, K):
    ops = inputs.make_operands("bf16", M, N, K, seed=11)
    av = torch.from_numpy(ops.a.view(np.int16)).view(torch.bfloat16).double().numpy()
    bv = torch.from_numpy(ops.b.view(np.int16)).view(torch.bfloat16).double().numpy()
    exact = frac_gemm(to_frac(av), to_frac(bv))
    got = oracle.gemm_operands(ops)
    for m in range(M):
        for n in range(N):
            bound = sum(abs(Fraction(float(av[m, k])) * Fraction(float(bv[n, k]))) for k in range(K))
            assert abs(Fraction(got[m, n]) - exact[m][n]) <= bound * K * Fraction(1, 2 ** 52)


@pytest.mark.parametrize("M,N,K", [(2, 3, 64), (4, 4, 96)])
def test_mxfp4_vs_fraction(M, N, K):
    ops = inputs.make_operands("e2m1", M, N, K, seed=13)
    table = load_e2m1_golden()
    ca = oracle.unpack_e2m1_rows(ops.a, K)
    cb = oracle.unpack_e2m1_rows(ops.b, K)
    got = oracle.gemm_operands(ops)
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for j in range(K // 32):
                part = sum((Fraction(table[int(ca[m, k])]) * Fraction(table[int(cb[n, k])])
                            for k in range(32 * j, 32 * j + 32)), Fraction(0))
                tot += part * Fraction(2) ** (int(ops.scale_a[m, j]) - 127) * Fraction(2) ** (int(ops.scale_b[n, j]) - 127)
            assert Fraction(got[m, n]) == tot  # exact: power-of-two scales, short sums


@pytest.mark.parametrize("M,N,K", [(2, 3, 64), (4, 4, 96), (3, 2, 160)])
def test_dequantized_matmul_vs_fraction(M, N, K):
    """The full-size path (dq(A) . dq(B)^T through numpy's matmul) against
    exact rational brute force: bit-exact for E4M3 (before the two scalings)
    and MXFP4, within K 2^-52 sum|ab| for BF16."""
    table = load_e2m1_golden()
    ops = inputs.make_operands("e2m1", M, N, K, seed=17 + K)
    # non-uniform block exponents, so a wrong block mapping changes the sum
    rng = np.random.default_rng(K)
    ops.scale_a = rng.integers(120, 131, size=ops.scale_a.shape).astype(np.uint8)
    ops.scale_b = rng.integers(120, 131, size=ops.scale_b.shape).astype(np.uint8)
    ca = oracle.unpack_e2m1_rows(ops.a, K)
    cb = oracle.unpack_e2m1_rows(ops.b, K)
    got = oracle.gemm_dequantized(ops)
    for m in range(M):
        for n in range(N):
            tot = sum((Fraction(table[int(ca[m, k])]) * Fraction(table[int(cb[n, k])]) *
                       Fraction(2) ** (int(ops.scale_a[m, k // 32]) + int(ops.scale_b[n, k // 32]) - 254)
                       for k in range(K)), Fraction(0))
            assert Fraction(got[m, n]) == tot
    ops8 = inputs.make_operands("e4m3", M, N, K, seed=19 + K)
    vals = torch_e4m3_values()
    acc = frac_gemm(to_frac(vals[ops8.a]), to_frac(vals[ops8.b]))
    got8 = oracle.gemm_dequantized(ops8)
    for m in range(M):
        for n in range(N):
            want = float(acc[m][n]) * np.float64(ops8.scale_a[m]) * np.float64(ops8.scale_b[n])
            assert got8[m, n] == want  # exact sum, then the same two roundings
    opsb = inputs.make_operands("bf16", M, N, K, seed=23 + K)
    av = torch.from_numpy(opsb.a.view(np.int16)).view(torch.bfloat16).double().numpy()
    bv = torch.from_numpy(opsb.b.view(np.int16)).view(torch.bfloat16).double().numpy()
    exact = frac_gemm(to_frac(av), to_frac(bv))
    gotb = oracle.gemm_dequantized(opsb)
    for m in range(M):
        for n in range(N):
            bound = sum(abs(Fraction(float(av[m, k])) * Fraction(float(bv[n, k]))) for k in range(K))
            assert abs(Fraction(gotb[m, n]) - exact[m][n]) <= bound * K * Fraction(1, 2 ** 52)


@pytest.mark.parametrize("dtype,M,N,K", [("e4m3", 70, 384, 1024), ("e2m1", 65, 512, 2048)])
def test_dequantized_matmul_equals_the_loops(dtype, M, N, K):
    """Where the sums are exact, the matmul path and the plain loops agree bit
    for bit, on all rows and on a subset."""
    ops = inputs.make_operands(dtype, M, N, K, seed=29)
    assert np.array_equal(oracle.gemm_dequantized(ops), oracle.gemm_operands(ops))
    rows = np.array([0, 3, M - 1])
    assert np.array_equal(oracle.gemm_dequantized(ops, rows=rows), oracle.gemm_operands(ops, rows=rows))


def test_mx_exactness_guard():
    K = 8192
    ea = np.full((2, K // 32), 127, np.uint8)
    assert oracle._mx_sum_is_exact(ea, ea, K)
    wide = ea.copy()
    wide[0, 0], wide[1, 1] = 10, 240  # exponent sums spanning ~460 binades
    assert not oracle._mx_sum_is_exact(wide, ea, K)
    # with a span the fp64 sum could not hold, the block loops are used instead
    ops = inputs.make_operands("e2m1", 2, 256, K, seed=3)
    ops.scale_a = wide
    assert np.array_equal(oracle.gemm_dequantized(ops), oracle.gemm_operands(ops))


def test_planted_block_scale_mapping_is_caught(monkeypatch):
    # element k takes block (k mod K/32) instead of k // 32
    _pins_fail(monkeypatch, "expand_block_scales",
               lambda e, K, blk=32: np.tile(oracle.decode_ue8m0(e), (1, blk))[:, :K],
               lambda: test_dequantized_matmul_vs_fraction(2, 3, 64))


def test_block_scaled_reduces_to_plain_when_scales_are_one():
    rng = np.random.default_rng(3)
    M, N, K = 5, 6, 128
    pa = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    pb = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    one_a = np.full((M, K // 32), 127, np.uint8)
    one_b = np.full((N, K // 32), 127, np.uint8)
    got = oracle.gemm_mxfp4(pa, pb, one_a, one_b, K)
    plain = oracle.gemm_f64(oracle.decode_e2m1(oracle.unpack_e2m1_rows(pa, K)),
                            oracle.decode_e2m1(oracle.unpack_e2m1_rows(pb, K)))
    assert np.array_equal(got, plain)
    # numpy's BLAS on the same decoded values (a library routine)
    ref = oracle.decode_e2m1(oracle.unpack_e2m1_rows(pa, K)) @ oracle.decode_e2m1(oracle.unpack_e2m1_rows(pb, K)).T
    assert np.array_equal(got, ref)


def test_identity_and_permutation_operands():
    K = 64
    rng = np.random.default_rng(5)
    # bf16: A = I (0x3F80 is 1.0) -> C = B^T
    b = inputs.bf16_rows(48, K, inputs._gen(1))
    eye = np.where(np.eye(K, dtype=bool), np.uint16(0x3F80), np.uint16(0))
    c = oracle.gemm_bf16(eye, b)
    assert np.array_equal(c, oracle.decode_bf16(b).T)
    # A = permutation P -> C = P . B^T (rows of B^T permuted)
    perm = rng.permutation(K)
    pm = np.zeros((K, K), np.uint16)
    pm[np.arange(K), perm] = 0x3F80
    c = oracle.gemm_bf16(pm, b)
    assert np.array_equal(c, oracle.decode_bf16(b).T[perm])
    # e4m3 with unit scales: 0x38 is 1.0
    qb, _ = inputs.e4m3_rows(40, K, inputs._gen(2))
    eye8 = np.where(np.eye(K, dtype=bool), np.uint8(0x38), np.uint8(0))
    c = oracle.gemm_e4m3_rowcol(eye8, qb, np.ones(K, np.float32), np.ones(40, np.float32))
    assert np.array_equal(c, oracle.decode_e4m3(qb).T)
    # row and column scales act on rows and columns of C
    sa = np.arange(1, K + 1, dtype=np.float32)
    sb = np.full(40, 0.5, np.float32)
    c = oracle.gemm_e4m3_rowcol(eye8, qb, sa, sb)
    assert np.array_equal(c, oracle.decode_e4m3(qb).T * sa[:, None] * 0.5)
    # int8: diagonal A scales the rows of B^T
    d = np.diag(np.arange(-32, 32)).astype(np.int8)
    bi = rng.integers(-128, 128, size=(20, K)).astype(np.int8)
    c = oracle.gemm_int8(d, bi)
    assert np.array_equal(c, np.arange(-32, 32)[:, None] * bi.T.astype(np.int64))


def test_sampled_rows_cols_equal_full():
    ops = inputs.make_operands("e4m3", 40, 72, 128, seed=3)
    full = oracle.gemm_operands(ops)
    rows = np.array([0, 7, 39])
    cols = np.array([1, 64, 71, 5])
    part = oracle.gemm_operands(ops, rows=rows, cols=cols)
    assert np.array_equal(part, full[np.ix_(rows, cols)])


def test_parity_metric():
    r = np.array([[0.0, 1.0], [-100.0, 3.0]])
    assert oracle.max_rel_err(r, r) == 0.0
    c = r.copy()
    c[1, 0] *= 1 + 0.009       # 0.9 % off a large value -> above the bound
    assert oracle.max_rel_err(c, r) > oracle.FLOAT_TOL
    c = r.copy()
    c[0, 0] = 5e-5             # near zero: the +1e-2 floor governs
    assert oracle.max_rel_err(c, r) == pytest.approx(5e-3)


# ---------------------------------------------------------------- bookkeeping

def load_worked_numbers():
    rows = []
    for line in open(os.path.join(GOLDEN, "gemm_optimization_worked_numbers.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, args, val, how = [x.strip() for x in line.split("|")]
        rows.append((key, args.split(), float(val), how))
    return rows


def _eval(key, args):
    if key == "mfma_per_tile":
        m, n, k, eb = map(int, args)
        return oracle.mfma_per_tile(m, n, k, eb)
    if key in ("k_unroll", "m_repeat", "num_acc_n"):
        m, n, k, eb = map(int, args)
        return oracle.tile_params(m, n, k, eb)[key]
    if key == "lds_kb":
        m, k, eb = map(int, args)
        return oracle.lds_bytes(m, k, eb) / 1024
    if key == "grid_blocks":
        M, N, tm, tn = map(int, args)
        return oracle.grid_blocks(M, N, tm, tn)
    if key == "mfma_per_block":
        K, tm, tn, tk, eb = map(int, args)
        return oracle.mfma_per_block(K, tm, tn, tk, eb)
    if key == "gflop":
        M, N, K = map(int, args)
        return oracle.flops(M, N, K) / 1e9
    if key == "mbytes":
        M, N, K, kind = int(args[0]), int(args[1]), int(args[2]), args[3]
        return oracle.bytes_moved(M, N, K, kind) / 1e6
    if key == "gbps_at_ms":
        M, N, K, kind, ms = int(args[0]), int(args[1]), int(args[2]), args[3], float(args[4])
        return oracle.bytes_moved(M, N, K, kind) / (ms * 1e-3) / 1e9
    raise KeyError(key)


@pytest.mark.parametrize("row", load_worked_numbers(), ids=lambda r: r[0] + ":" + "x".join(r[1]))
def test_worked_numbers(row):
    key, args, printed, how = row
    got = _eval(key, args)
    if how == "exact":
        assert got == printed
    elif how.startswith("round:"):
        d = int(how.split(":")[1])
        assert round(got, d) == printed
    elif how.startswith("trunc:"):
        d = int(how.split(":")[1])
        assert int(got * 10 ** d) / 10 ** d == pytest.approx(printed)


@pytest.mark.parametrize("M,N,K", [(16, 7168, 4096), (128, 256, 512), (4096, 8192, 8192), (3, 128, 64)])
def test_bytes_moved_counts_the_operand_arrays(M, N, K):
    """Section 8.2's three byte counts against the sizes of the arrays they
    count, built independently: A and B as stored (int8 one byte per value;
    int4 and E2M1 two values per byte), a bf16 C [M, N], and the scales
    (fp32 per row of A and of B; one UE8M0 byte per 32 K-elements of each
    operand for MXFP4)."""
    a8 = np.zeros((M, K), np.int8)
    b8 = np.zeros((N, K), np.int8)
    b4 = np.zeros((N, K // 2), np.uint8)
    a_fp4 = np.zeros((M, K // 2), np.uint8)
    b_fp4 = np.zeros((N, K // 2), np.uint8)
    c = np.zeros((M, N), np.uint16)
    row_scales = np.zeros(M + N, np.float32)
    mx_scales = [np.zeros((M, K // 32), np.uint8), np.zeros((N, K // 32), np.uint8)]
    assert oracle.bytes_moved(M, N, K, "int8") == a8.nbytes + b8.nbytes + c.nbytes + row_scales.nbytes
    assert oracle.bytes_moved(M, N, K, "fp8") == a8.nbytes + b8.nbytes + c.nbytes + row_scales.nbytes
    assert oracle.bytes_moved(M, N, K, "int4") == a8.nbytes + b4.nbytes + c.nbytes + row_scales.nbytes
    assert oracle.bytes_moved(M, N, K, "mxfp4") == (a_fp4.nbytes + b_fp4.nbytes + c.nbytes +
                                                    sum(x.nbytes for x in mx_scales))


def test_bytes_moved_int4_and_mxfp4_by_hand():
    """Hand-worked from the section 8.2 counts for M = N = K = 1024 (MB =
    1e6 B): int4 = 1,048,576 (A) + 524,288 (B) + 2,097,152 (C) + 8,192
    (scales) = 3,678,208; MXFP4 = 524,288 + 524,288 + 2,097,152 + 65,536
    (2 x 1024 x 32 scale bytes) = 3,211,264."""
    assert oracle.bytes_moved(1024, 1024, 1024, "int4") == 3678208
    assert oracle.bytes_moved(1024, 1024, 1024, "mxfp4") == 3211264


def test_planted_mxfp4_scale_bytes_are_caught(monkeypatch):
    good = oracle.bytes_moved
    _pins_fail(monkeypatch, "bytes_moved",
               lambda M, N, K, kind: good(M, N, K, kind) - (M + N) * (K // 32) * (kind == "mxfp4"),
               lambda: test_bytes_moved_counts_the_operand_arrays(128, 256, 512))


def test_tflops_formula():
    # section 8.1: 2*M*N*K flops in `us` microseconds
    assert oracle.tflops(1000, 1000, 1000, 1.0) == pytest.approx(2000.0)


# ---------------------------------------------------------------- pack model

@pytest.mark.parametrize("rows", [128, 8])
@pytest.mark.parametrize("N,Kb", [(128, 128), (256, 512), (384, 256)])
def test_pack_roundtrip_and_permutation(N, Kb, rows):
    rng = np.random.default_rng(N + Kb)
    b = rng.integers(0, 256, size=(N, Kb), dtype=np.uint8)
    p = oracle.pack_b_bytes(b, rows)
    assert p.size == b.size
    assert np.array_equal(oracle.unpack_b_bytes(p, N, Kb, rows), b)
    offs = oracle.packed_offset(*np.meshgrid(np.arange(N), np.arange(Kb), indexing="ij"), Kb, rows)
    assert np.array_equal(np.sort(offs.ravel()), np.arange(N * Kb))  # a bijection


@pytest.mark.parametrize("rows", [128, 8])
def test_pack_layout_invariants(rows):
    check_pack_layout(rows)


def check_pack_layout(rows):
    N, Kb = 256, 384
    tile_bytes = rows * 128
    # index-encode: byte value identifies (row mod rows, 16-byte chunk) etc.
    n, k = np.meshgrid(np.arange(N), np.arange(Kb), indexing="ij")
    off = oracle.packed_offset(n, k, Kb, rows)
    tile = off // tile_bytes
    # each tile holds exactly one rows x 128-byte block of B, K tiles of a band adjacent
    assert np.all(tile == (n // rows) * (Kb // 128) + k // 128)
    # a 16-byte chunk of a row stays contiguous and in order
    assert np.all(off[:, 1:][k[:, 1:] % 16 != 0] == off[:, :-1][k[:, 1:] % 16 != 0] + 1)
    # rows sit at a 128-byte pitch inside their tile
    assert np.all((off % tile_bytes) // 128 == n % rows)
    # any 8 consecutive rows (aligned) reading the same logical chunk hit 8
    # distinct 16-byte positions: no shared-memory bank conflicts
    pos = (off % 128) // 16
    for c in range(8):
        for g in range(0, N, 8):
            assert len(set(pos[g:g + 8, c * 16].tolist())) == 8


def test_w4_layout_spreads_the_kernels_reads_over_all_banks():
    # The W4A8 kernel's lane (g, t) reads logical chunk c0 + t (c0 = 0 or 4)
    # of row g.  One 16-byte shared-memory load serves 8 lanes at a time:
    # rows 2i and 2i + 1, four chunks each.  Those 8 chunks must sit in 8
    # distinct 16-byte positions of the 128-byte bank window.
    N, Kb = 16, 256
    n, k = np.meshgrid(np.arange(N), np.arange(Kb), indexing="ij")
    pos = (oracle.packed_offset(n, k, Kb, 8, w4=True) % 128) // 16
    plain = (oracle.packed_offset(n, k, Kb, 8) % 128) // 16
    for c0 in (0, 4):
        for i in range(0, 8, 2):
            chunks = [(c0 + t) * 16 for t in range(4)]
            assert len({int(pos[r, c]) for r in (i, i + 1) for c in chunks}) == 8
            # the INT8 slot rule alone puts the two rows on the same 4 positions
            assert len({int(plain[r, c]) for r in (i, i + 1) for c in chunks}) == 4
    # a bijection, and every other layout property of the 8-row bands holds
    offs = oracle.packed_offset(n, k, Kb, 8, w4=True)
    assert np.array_equal(np.sort(offs.ravel()), np.arange(N * Kb))
    assert np.all(offs // 1024 == (n // 8) * (Kb // 128) + k // 128)
    assert np.all((offs % 1024) // 128 == n % 8)


def test_pack_band_rows_per_dtype():
    # INT8 packs 8-row bands: a band's K tiles are 1 KiB apart
    assert oracle.band_rows("int8") == 8
    assert all(oracle.band_rows(d) == 128 for d in ("bf16", "e4m3", "e2m1"))
    b = np.arange(16 * 256, dtype=np.int64).astype(np.uint8).reshape(16, 256)
    p = oracle.pack_b(b.view(np.int8), "int8") ^ np.uint8(0x80)  # undo the offset binary
    assert np.array_equal(p[:128], b[0, :128])            # row 0, K tile 0
    assert np.array_equal(p[1024:1024 + 128], b[0, 128:])  # row 0, K tile 1 follows the 8-row tile
    assert np.array_equal(p[2048:2048 + 16], b[8, 0:16])  # row 8 opens band 1
    # offset binary: -128 -> 0x00, 0 -> 0x80, 127 -> 0xff; other types untouched
    q = oracle.pack_b(np.array([[-128, 0, 127, -1] * 32] * 8, np.int8), "int8")
    assert q[0] == 0x00 and q[1] == 0x80 and q[2] == 0xFF and q[3] == 0x7F
    e = np.arange(128 * 128, dtype=np.int64).astype(np.uint8).reshape(128, 128)
    assert np.array_equal(oracle.pack_b(e, "e4m3"), oracle.pack_b_bytes(e))


def test_pack_scale_roundtrip():
    rng = np.random.default_rng(9)
    N, nblk = 256, 64
    s = rng.integers(0, 255, size=(N, nblk), dtype=np.uint8)
    p = oracle.pack_b_scales(s)
    assert np.array_equal(oracle.unpack_b_scales(p, N, nblk), s)
    offs = oracle.packed_scale_offset(*np.meshgrid(np.arange(N), np.arange(nblk), indexing="ij"), nblk)
    assert np.array_equal(np.sort(offs.ravel()), np.arange(N * nblk))


# ---------------------------------------------------------------- planted mistakes

def _pins_fail(monkeypatch, attr, mutant, check):
    monkeypatch.setattr(oracle, attr, mutant)
    with pytest.raises(AssertionError):
        check()


def test_planted_e4m3_subnormal_bug_is_caught(monkeypatch):
    good = oracle.decode_e4m3

    def bad(c):
        v = good(c)
        c = np.asarray(c, np.uint8)
        return np.where(((c >> 3) & 0xF) == 0, v * 2, v)  # wrong subnormal exponent
    _pins_fail(monkeypatch, "decode_e4m3", bad, test_e4m3_decode_matches_torch_all_codes)


def test_planted_e2m1_bias_bug_is_caught(monkeypatch):
    good = oracle.decode_e2m1
    _pins_fail(monkeypatch, "decode_e2m1", lambda c: good(c) * 2.0, test_e2m1_decode_matches_ocp_table)


def test_planted_transposed_operand_is_caught(monkeypatch):
    good = oracle.gemm_f64
    _pins_fail(monkeypatch, "gemm_f64", lambda a, b: good(a, np.ascontiguousarray(b[:, ::-1])),
               lambda: test_e4m3_rowcol_vs_fraction(3, 4, 64))


def test_planted_dropped_term_is_caught(monkeypatch):
    good = oracle.gemm_f64
    _pins_fail(monkeypatch, "gemm_f64", lambda a, b: good(a[:, :-1], b[:, :-1]),
               lambda: test_bf16_vs_fraction(3, 4, 16))


def test_planted_scale_sign_bug_is_caught(monkeypatch):
    good = oracle.decode_ue8m0
    _pins_fail(monkeypatch, "decode_ue8m0", lambda c: 1.0 / good(c),
               lambda: test_mxfp4_vs_fraction(2, 3, 64))


def test_planted_missing_column_scale_is_caught(monkeypatch):
    good = oracle.gemm_e4m3_rowcol
    _pins_fail(monkeypatch, "gemm_e4m3_rowcol", lambda qa, qb, sa, sb: good(qa, qb, sa, np.ones_like(sb)),
               lambda: test_e4m3_rowcol_vs_fraction(3, 4, 64))


def test_planted_pack_swizzle_bug_is_caught(monkeypatch):
    good = oracle.packed_offset

    def bad(n, kb, Kb, rows=128):
        o = good(n, kb, Kb, rows)
        return o - (o % 128) + (np.asarray(kb) % 128)  # forgets the chunk permutation
    monkeypatch.setattr(oracle, "packed_offset", bad)
    with pytest.raises(AssertionError):
        check_pack_layout(128)
    with pytest.raises(AssertionError):
        check_pack_layout(8)


# ---------------------------------------------------------------- fused epilogues

def test_epilogue_closed_forms_and_identities():
    x = np.linspace(-30, 30, 2001)[None, :]
    zero = np.zeros(x.shape[1])
    relu = oracle.apply_epilogue(x, "bias_relu", zero)
    silu = oracle.apply_epilogue(x, "bias_silu", zero)
    gelu = oracle.apply_epilogue(x, "bias_gelu", zero)
    # each activation f has f(x) - f(-x) = x (odd part x/2)
    for f in (relu, silu, gelu):
        assert np.allclose(f - f[:, ::-1], x, rtol=0, atol=1e-12)
    assert relu[0, 1000] == 0 and silu[0, 1000] == 0 and gelu[0, 1000] == 0
    assert silu[0, -1] == pytest.approx(30.0, rel=1e-12)          # sigmoid(30) = 1 - 9.4e-14
    assert gelu[0, -1] == pytest.approx(30.0, rel=1e-15)
    assert silu[0, 1000 + 66] == pytest.approx(x[0, 1066] / (1 + np.exp(-x[0, 1066])), rel=1e-15)
    # GELU(1) = Phi(1) = 0.8413447460685429 (standard normal CDF at 1)
    assert oracle.apply_epilogue(np.array([[1.0]]), "bias_gelu", np.zeros(1))[0, 0] == pytest.approx(
        0.8413447460685429, rel=1e-14)


def test_epilogue_vs_torch_library_routines():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(17)
    c = rng.standard_normal((64, 96)) * 4
    bias = rng.standard_normal(96)
    x = torch.from_numpy(c + bias[None, :])
    assert np.allclose(oracle.apply_epilogue(c, "bias_silu", bias), torch.nn.functional.silu(x).numpy(),
                       rtol=1e-13, atol=1e-15)
    assert np.allclose(oracle.apply_epilogue(c, "bias_gelu", bias),
                       torch.nn.functional.gelu(x, approximate="none").numpy(), rtol=1e-13, atol=1e-15)
    assert np.array_equal(oracle.apply_epilogue(c, "bias_relu", bias), torch.relu(x).numpy())
    # bias is added exactly, per output column
    assert np.array_equal(oracle.apply_epilogue(c, "bias", bias), c + bias[None, :])
    assert np.array_equal(oracle.apply_epilogue(c, "none"), c)
    with pytest.raises(ValueError):
        oracle.apply_epilogue(c, "bias_tanh", bias)


def test_planted_tanh_gelu_is_caught(monkeypatch):
    good = oracle.apply_epilogue

    def tanh_gelu(c, epilogue, bias=None):
        if epilogue != "bias_gelu":
            return good(c, epilogue, bias)
        x = np.asarray(c, np.float64) + np.asarray(bias, np.float64)[None, :]
        return 0.5 * x * (1 + np.tanh(np.sqrt(2 / np.pi) * (x + 0.044715 * x ** 3)))
    monkeypatch.setattr(oracle, "apply_epilogue", tanh_gelu)
    with pytest.raises(AssertionError):
        test_epilogue_vs_torch_library_routines()


# ---------------------------------------------------------------- FP16 operands

def test_fp16_decode_all_codes_vs_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)   # a library decode of the same codes
    got = oracle.decode_fp16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # hand-checked codes: 1.0, -2.0, 65504 (max), 2^-24 (smallest subnormal), 2^-14 (smallest normal)
    assert list(oracle.decode_fp16(np.array([0x3C00, 0xC000, 0x7BFF, 0x0001, 0x0400], np.uint16))) == [
        1.0, -2.0, 65504.0, 2.0 ** -24, 2.0 ** -14]


@pytest.mark.parametrize("M,N,K", [(3, 4, 16), (4, 2, 40)])
def test_fp16_vs_fraction(M, N, K):
    ops = inputs.make_operands("fp16", M, N, K, seed=12)
    av = ops.a.view(np.float16).astype(np.float64)
    bv = ops.b.view(np.float16).astype(np.float64)
    exact = frac_gemm(to_frac(av), to_frac(bv))
    got = oracle.gemm_operands(ops)
    for m in range(M):
        for n in range(N):
            # fp16 products are exact in fp64 and the sums of K of them round at most K times
            bound = sum(abs(Fraction(float(av[m, k])) * Fraction(float(bv[n, k]))) for k in range(K))
            assert abs(Fraction(got[m, n]) - exact[m][n]) <= bound * K * Fraction(1, 2 ** 52)


def test_fp16_identity_operand():
    K = 64
    b = inputs.fp16_rows(48, K, inputs._gen(3))
    eye = np.where(np.eye(K, dtype=bool), np.uint16(0x3C00), np.uint16(0))   # 0x3C00 is 1.0
    assert np.array_equal(oracle.gemm_fp16(eye, b), oracle.decode_fp16(b).T)


def test_fp16_recipe():
    ops = inputs.make_operands("fp16", 64, 32, 256, seed=4)
    v = ops.a.view(np.float16).astype(np.float64)
    assert ops.a.dtype == np.uint16 and ops.a.shape == (64, 256)
    assert abs(v.std() * np.sqrt(256) - 1.0) < 0.1       # N(0,1)/sqrt(K)
    again = inputs.make_operands("fp16", 64, 32, 256, seed=4)
    assert np.array_equal(ops.a, again.a) and np.array_equal(ops.b, again.b)


# ---------------------------------------------------------------- activation quantisers

def test_encode_e4m3_definition():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_e4m3(codes)
    finite = ~np.isnan(vals)
    assert np.array_equal(oracle.encode_e4m3(vals[finite]), codes[finite])   # every finite code round-trips
    assert oracle.encode_e4m3(np.array([np.nan]))[0] == 0x7F
    # saturation to +-448 (0x7E / 0xFE), never NaN
    assert list(oracle.encode_e4m3(np.array([448.0, 460.0, 464.0, 1e9, -500.0]))) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    # ties go to the even fraction: 1.0625 -> 1.0, 1.1875 -> 1.25; subnormal 2^-10 -> 0, 1.5*2^-9 -> 2*2^-9
    got = oracle.encode_e4m3(np.array([1.0625, 1.1875, 2.0 ** -10, 1.5 * 2.0 ** -9, -2.0 ** -12]))
    assert list(got) == [0x38, 0x3A, 0x00, 0x02, 0x80]


def test_encode_e4m3_vs_torch_cast():
    x = torch.randn(1_000_000, generator=torch.Generator().manual_seed(5), dtype=torch.float32) * 100
    x = x[x.abs() < 448]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()     # a library encoder
    assert np.array_equal(oracle.encode_e4m3(x.double().numpy()), ref)


def test_encode_e2m1_definition():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.encode_e2m1(oracle.decode_e2m1(codes)), codes)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert list(oracle.decode_e2m1(oracle.encode_e2m1(ties))) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert list(oracle.encode_e2m1(np.array([6.0, 7.0, 1e9, -1e9, -0.1]))) == [7, 7, 7, 15, 8]


def test_mx_block_exponent_edges():
    f32 = np.float32
    a = np.array([6.0, np.nextafter(f32(6.0), f32(7.0)), 3.0, 4.0, 0.0, 1e-38, 3e38, 0.75], dtype=np.float32)
    e = oracle.mx_block_exponent(a)
    assert list(e[:5]) == [0, 1, -1, 0, 0]
    for ai, ei in zip(a.astype(np.float64), e):               # smallest e with amax <= 6 * 2^e
        if ai > 0 and -127 < ei < 127:
            assert ai <= 6 * 2.0 ** ei and ai > 6 * 2.0 ** (ei - 1)
    rng = np.random.default_rng(8)
    r = np.abs(rng.standard_normal(100000).astype(np.float32)) * np.float32(2.0) ** rng.integers(-30, 30, 100000)
    assert np.array_equal(oracle.mx_block_exponent(r), inputs.ue8m0_block_exponent(r))


@pytest.mark.parametrize("R,K", [(64, 256), (300, 1024)])
def test_quantizers_match_the_input_recipes(R, K):
    """The oracle's quantisers and the input recipes (torch casts and their
    own encoders) give the same bytes on the same draws."""
    codes, s = inputs.e4m3_rows(R, K, inputs._gen(41))
    x = torch.randn((R, K), generator=inputs._gen(41), dtype=torch.float32).numpy()
    q, s2 = oracle.quantize_e4m3_rows(x)
    assert np.array_equal(q, codes) and np.array_equal(s2.view(np.uint32), s.view(np.uint32))
    packed, exps = inputs.mxfp4_rows(R, K, inputs._gen(42))
    x = torch.randn((R, K), generator=inputs._gen(42), dtype=torch.float32).numpy()
    p2, e2 = oracle.quantize_mxfp4_rows(x)
    assert np.array_equal(p2, packed) and np.array_equal(e2, exps)


def test_quantizer_error_bounds():
    x = (torch.randn((8, 512), generator=torch.Generator().manual_seed(3)) * 7).numpy()
    q, s = oracle.quantize_e4m3_rows(x)
    deq = oracle.decode_e4m3(q) * s[:, None].astype(np.float64)
    # half an ulp: 2^-4 relative for normals, half the subnormal step 2^-10 * s below 2^-6 * s
    assert np.all(np.abs(deq - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * (1 + 1e-6))
    p, e = oracle.quantize_mxfp4_rows(x)
    vals = oracle.decode_e2m1(oracle.unpack_e2m1_rows(p, 512)) * np.repeat(oracle.decode_ue8m0(e), 32, axis=1)
    step = np.repeat(np.ldexp(1.0, e.astype(np.int64) - 127), 32, axis=1)   # spacing 0.5 .. 2 times 2^e
    assert np.all(np.abs(vals - x) <= step * 1.0 + 1e-12)
    zero = np.zeros((2, 64), np.float32)
    q0, s0 = oracle.quantize_e4m3_rows(zero)
    assert np.all(q0 == 0) and np.all(s0 == 1.0)
    p0, e0 = oracle.quantize_mxfp4_rows(zero)
    assert np.all(p0 == 0) and np.all(e0 == 127)


def test_planted_truncating_e4m3_is_caught(monkeypatch):
    good = oracle.encode_e4m3

    def trunc(v):
        v = np.asarray(v, np.float64)
        f, ex = np.frexp(np.abs(v))
        q = np.ldexp(1.0, ex - 4)
        return good(np.sign(v) * np.floor(np.abs(v) / q) * q)
    monkeypatch.setattr(oracle, "encode_e4m3", trunc)
    with pytest.raises(AssertionError):
        test_encode_e4m3_vs_torch_cast()


# ---------------------------------------------------------------- W4A8 (int4 weights, int8 activations)

def test_unpack_int4_definition():
    b = np.arange(256, dtype=np.uint8)[None, :]
    v = oracle.unpack_int4_rows(b, 512)[0]
    lo, hi = v[0::2], v[1::2]
    for byte in range(256):
        n0, n1 = byte & 0xF, byte >> 4
        assert lo[byte] == (n0 - 16 if n0 >= 8 else n0) and hi[byte] == (n1 - 16 if n1 >= 8 else n1)


@pytest.mark.parametrize("M,N,K", [(3, 4, 16), (5, 3, 64)])
def test_w4a8_vs_brute_force(M, N, K):
    ops = inputs.make_operands("w4a8", M, N, K, seed=13)
    a = ops.a.astype(np.int64)
    b = oracle.unpack_int4_rows(ops.b, K).astype(np.int64)
    assert b.min() >= -8 and b.max() <= 7
    got = oracle.gemm_operands(ops)
    for m in range(M):
        for n in range(N):
            assert got[m, n] == sum(int(a[m, k]) * int(b[n, k]) for k in range(K))


def test_w4a8_identity_and_extremes():
    K = 64
    eye = np.eye(K, dtype=np.int8)
    b = inputs.int4_rows(24, K, inputs._gen(5))
    assert np.array_equal(oracle.gemm_w4a8(eye, b, K), oracle.unpack_int4_rows(b, K).T.astype(np.int64))
    a = np.full((2, 4096), -128, np.int8)
    bb = np.full((3, 2048), 0x88, np.uint8)           # every nibble -8
    assert np.all(oracle.gemm_w4a8(a, bb, 4096) == 4096 * 1024)


def test_w4a8_pack_word_order():
    # one row, K = 256 (128 bytes): values k = 0..7 in the first word are -8, -7, ..., -1
    vals = np.array([-8, -7, -6, -5, -4, -3, -2, -1] + [0] * 248, np.int16)
    nib = (vals & 0xF).astype(np.uint8)
    b = (nib[0::2] | (nib[1::2] << 4))[None, :].repeat(8, axis=0)   # an 8-row band
    p = oracle.pack_b(b, "w4a8")
    word = int(p[:4].view("<u4")[0])
    u = [v + 8 for v in range(-8, 0)]                   # offset binary 0..7
    for k, bit in enumerate(oracle.W4_NIBBLE_BITS):
        assert (word >> bit) & 0xF == u[k]
    for j in range(4):                                   # (word >> 4j) & 0x000F000F is the pair (k2j, k2j+1)
        pair = (word >> (4 * j)) & 0x000F000F
        assert pair & 0xFFFF == u[2 * j] and pair >> 16 == u[2 * j + 1]
    # a bijection of the bytes of B (as nibble multisets per word), with the 8-row band layout
    rng = np.random.default_rng(4)
    bb = rng.integers(0, 256, size=(16, 256), dtype=np.uint8)
    pk = oracle.pack_b(bb, "w4a8")
    assert pk.size == bb.size
    il = oracle.interleave_int4_words(bb)
    assert np.array_equal(pk, oracle.pack_b_bytes(il, 8, w4=True))


# ---------------------------------------------------------------- error diagnostic denominator

def _abs_sum_pins(dtype):
    K = 256 if dtype == "e2m1" else 192
    ops = inputs.make_operands(dtype, 9, 10, K, seed=71)
    c = oracle.gemm_operands(ops).astype(np.float64)
    s = oracle.gemm_abs_operands(ops)
    assert np.all(s >= np.abs(c) - 1e-12 * s)
    if dtype in ("int8", "w4a8"):
        a = np.abs(ops.a.astype(np.int16)).clip(0, 127).astype(np.int8)
        if dtype == "int8":
            b = np.abs(ops.b.astype(np.int16)).clip(0, 127).astype(np.int8)
        else:   # int4 nibbles 0..7 (non-negative), two per byte
            b = (ops.b & 0x77).astype(np.uint8)
        pos = inputs.Operands(dtype, 9, 10, K, a, b, None, None)
    elif dtype in ("bf16", "fp16"):
        pos = inputs.Operands(dtype, 9, 10, K, ops.a & 0x7FFF, ops.b & 0x7FFF, None, None)
    elif dtype == "e4m3":
        pos = inputs.Operands(dtype, 9, 10, K, ops.a & 0x7F, ops.b & 0x7F, ops.scale_a, ops.scale_b)
    else:   # E2M1: clear the sign bit of both nibbles
        pos = inputs.Operands(dtype, 9, 10, K, ops.a & 0x77, ops.b & 0x77, ops.scale_a, ops.scale_b)
    assert np.array_equal(oracle.gemm_abs_operands(pos), oracle.gemm_operands(pos).astype(np.float64))


@pytest.mark.parametrize("dtype", ["int8", "w4a8", "bf16", "fp16", "e4m3", "e2m1"])
def test_abs_sum_bounds_and_equality_for_nonnegative_operands(dtype):
    """S = sum |a||b| is at least |C| everywhere; with every operand value
    non-negative it equals C (the same product with no cancellation)."""
    _abs_sum_pins(dtype)


def test_abs_sum_of_sign_matrices_is_k():
    # A, B with entries +-1: every |a||b| is 1, so S = K while C varies
    K = 128
    rng = np.random.default_rng(9)
    a = rng.choice(np.array([-1, 1], np.int8), size=(6, K))
    b = rng.choice(np.array([-1, 1], np.int8), size=(7, K))
    ops = inputs.Operands("int8", 6, 7, K, a, b, None, None)
    assert np.all(oracle.gemm_abs_operands(ops) == K)
    c = oracle.gemm_operands(ops)
    assert oracle.max_err_over_abs(c + 1, c, np.full((6, 7), K)) == 1.0 / K


@pytest.mark.parametrize("dtype", ["e4m3", "e2m1"])
def test_planted_abs_sum_dropped_scale_is_caught(monkeypatch, dtype):
    # an S that leaves out the scales of B must fail one of the pins
    real = oracle.gemm_abs_operands

    def dropped(ops, rows=None, cols=None):
        if ops.dtype == "e4m3":
            ops = inputs.Operands(ops.dtype, ops.M, ops.N, ops.K, ops.a, ops.b, ops.scale_a, None)
        else:
            ops = inputs.Operands(ops.dtype, ops.M, ops.N, ops.K, ops.a, ops.b, ops.scale_a,
                                  np.full_like(ops.scale_b, 127))
        return real(ops, rows, cols)
    monkeypatch.setattr(oracle, "gemm_abs_operands", dropped)
    with pytest.raises(AssertionError):
        _abs_sum_pins(dtype)

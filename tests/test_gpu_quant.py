"""GPU parity of the activation quantiser (gemm_quantize_a) against the
oracle's encoders: codes and scales must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_preshuffle_gb300 as gp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_preshuffle_gb300 import build
    build.build()
    gp.load_library()


def special_rows(K):
    """Rows that put values exactly on rounding ties, zeros, saturation and
    subnormal inputs."""
    rows = []
    e4m3_ties = np.array([1.0625, 1.1875, -1.0625, 2.0 ** -10, 1.5 * 2.0 ** -9, 3.0, 448.0, -448.0], np.float64)
    r = np.resize(e4m3_ties, K).astype(np.float32)   # amax 448 -> s = 1: the values are the quotients
    rows.append(r)
    e2m1_ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -5.0, 0.0, 4.0], np.float64)
    rows.append(np.resize(e2m1_ties, K).astype(np.float32))   # every 32-block has amax 6 -> e = 0
    rows.append(np.zeros(K, np.float32))
    rows.append((np.resize([1e-40, -3e-41, 2e-45], K)).astype(np.float32))   # subnormal fp32 inputs
    rows.append((np.resize([3e38, -1e38, 1.0], K)).astype(np.float32))       # near the top of fp32
    rows.append((np.resize([3e-37, -1e-38, 5e-39], K)).astype(np.float32))   # s = amax/448 is subnormal
    return np.stack(rows)


@pytest.mark.parametrize("q", ["e4m3", "e2m1"])
@pytest.mark.parametrize("xd", ["fp32", "bf16"])
@pytest.mark.parametrize("M,K", [(1, 32), (37, 256), (300, 1024), (16, 7168), (5, 8192),
                                 (3, 16384), (2, 12288),   # bf16 rows past 8192 (fp32 past 12288): read twice
                                 (300000, 32),             # more rows than one grid: the striding loops
                                 (4000, 2048), (1000, 12288)])  # fp32: several rows per CTA through the staged ring
def test_quantize_bit_exact(q, xd, M, K):
    g = torch.Generator().manual_seed(M * 131 + K)
    x = torch.randn((M, K), generator=g, dtype=torch.float32) * torch.exp(torch.randn((M, 1), generator=g) * 3)
    if M >= 8:
        x[:6] = torch.from_numpy(special_rows(K))
    if xd == "bf16":
        x = x.to(torch.bfloat16)
    X = x.cuda()
    A, S = gp.quantize(X, q)
    torch.cuda.synchronize()
    xf = x.float().numpy()
    if q == "e4m3":
        ref_q, ref_s = oracle.quantize_e4m3_rows(xf)
        assert np.array_equal(S.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    else:
        ref_q, ref_s = oracle.quantize_mxfp4_rows(xf)
        assert np.array_equal(S.cpu().numpy(), ref_s)
    got = A.cpu().numpy()
    assert np.array_equal(got, ref_q), f"{int((got != ref_q).sum())} codes differ"


@pytest.mark.parametrize("q,M,N,K", [("e4m3", 200, 512, 1024), ("e2m1", 129, 512, 512)])
def test_quantize_then_gemm(q, M, N, K):
    """The quantiser's output feeds gemm_run directly; the product matches
    the oracle's quantise-then-multiply."""
    g = torch.Generator().manual_seed(9)
    x = torch.randn((M, K), generator=g)
    w = torch.randn((N, K), generator=g)
    A, SA = gp.quantize(x.cuda(), q)
    B, SB = gp.quantize(w.cuda(), q)
    if q == "e4m3":
        Bp = gp.preshuffle_b(B, "e4m3")
        C = gp.matmul(A, Bp, "e4m3", N, K, scale_a=SA, scale_b=SB)
        qa, sa = oracle.quantize_e4m3_rows(x.numpy())
        qb, sb = oracle.quantize_e4m3_rows(w.numpy())
        ref = oracle.gemm_e4m3_rowcol(qa, qb, sa, sb)
    else:
        Bp = gp.preshuffle_b(B, "e2m1", B_scales=SB)
        C = gp.matmul(A, Bp, "e2m1", N, K, scale_a=SA)
        pa, ea = oracle.quantize_mxfp4_rows(x.numpy())
        pb, eb = oracle.quantize_mxfp4_rows(w.numpy())
        ref = oracle.gemm_mxfp4(pa, pb, ea, eb, K)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    assert oracle.max_rel_err(C.float().cpu().numpy().astype(np.float64), ref) <= 8e-3


@pytest.mark.parametrize("q", ["e4m3", "e2m1"])
def test_quantizer_waits_for_the_gemm_reading_its_buffer(q):
    """Quantiser and GEMM launches overlap their neighbours on the stream
    (programmatic dependent launch).  Here one A buffer is quantised into,
    read by a GEMM, and quantised into again, three times back to back.
    Each quantiser must wait until the GEMM before it has read A, so every
    product matches its own input."""
    M, N, K = 1024, 4096, 4096
    g = torch.Generator().manual_seed(11)
    xs = [torch.randn((M, K), generator=g) for _ in range(3)]
    w = torch.randn((N, K), generator=g)
    Xs = [x.cuda() for x in xs]
    B, SB = gp.quantize(w.cuda(), q)
    if q == "e4m3":
        Bp = gp.preshuffle_b(B, "e4m3")
        A = torch.empty((M, K), dtype=torch.uint8, device="cuda")
        S = torch.empty((M,), dtype=torch.float32, device="cuda")
    else:
        Bp = gp.preshuffle_b(B, "e2m1", B_scales=SB)
        A = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
        S = torch.empty((M, K // 32), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    Cs = []
    for X in Xs:
        gp.gemm_quantize_a(X, "fp32", M, K, q, A, S, None)
        Cs.append(gp.matmul(A, Bp, q, N, K, scale_a=S, scale_b=SB if q == "e4m3" else None))
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    rows = np.r_[0:48, M - 48:M]
    if q == "e4m3":
        qb, sb = oracle.quantize_e4m3_rows(w.numpy())
    else:
        pb, eb = oracle.quantize_mxfp4_rows(w.numpy())
    for x, C in zip(xs, Cs):
        xr = x.numpy()[rows]
        if q == "e4m3":
            qa, sa = oracle.quantize_e4m3_rows(xr)
            ref = oracle.gemm_e4m3_rowcol(qa, qb, sa, sb)
        else:
            pa, ea = oracle.quantize_mxfp4_rows(xr)
            ref = oracle.gemm_mxfp4(pa, pb, ea, eb, K)
        c = C.float().cpu().numpy().astype(np.float64)[rows]
        assert oracle.max_rel_err(c, ref) <= 8e-3


def test_e4m3_near_midpoints_bit_exact():
    """Quotients within a few fp32 ulps of E4M3 rounding midpoints, where the
    kernel must fall back to the IEEE division to match fp32(x / s)."""
    rng = np.random.default_rng(11)
    K = 4096
    rows = []
    for amax in (448.0, 300.0, 1.0 / 3.0, 7.0e-3, 123456.0):
        s = np.float32(amax) / np.float32(448.0)
        mids = np.array([(1 + (k + 0.5) / 8) * 2.0 ** e for e in range(-6, 9) for k in range(8)], np.float64)
        mids = mids[mids < 448]
        target = rng.choice(mids, K) * rng.choice([-1, 1], K)
        x = (target * np.float64(s)).astype(np.float32)
        ulp = np.spacing(np.abs(x)).astype(np.float32)
        x = x + rng.integers(-6, 7, K).astype(np.float32) * ulp      # nudge by a few ulps either way
        x[0] = np.float32(amax)
        rows.append(x)
    x = np.stack(rows)
    A, S = gp.quantize(torch.from_numpy(x).cuda(), "e4m3")
    torch.cuda.synchronize()
    ref_q, ref_s = oracle.quantize_e4m3_rows(x)
    assert np.array_equal(S.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    got = A.cpu().numpy()
    assert np.array_equal(got, ref_q), f"{int((got != ref_q).sum())} codes differ"

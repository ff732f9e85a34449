"""The C-ABI library builds, loads and exports what include/gemm_preshuffle.h
declares; host-side validation rejects bad arguments before any CUDA call
(no GPU needed: these calls return before touching the device)."""
import ctypes

import pytest

import dense_gemm_preshuffle_gb300 as gp
from dense_gemm_preshuffle_gb300 import build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gp.load_library()


def test_exports_every_declared_symbol(lib):
    names = gp.header_functions()
    assert set(names) >= {"gemm_packed_b_bytes", "gemm_preshuffle_b", "gemm_unpack_b", "gemm_run", "gemm_run_ex",
                          "gemm_last_device_status", "gemm_status_string", "gemm_debug_skip_load"}
    for n in names:
        assert hasattr(lib, n), n


def test_rate_probe_is_built(lib):
    """build() also compiles the tensor-pipe rate probe the bench runs."""
    import os
    assert os.access(build.RATES_BIN, os.X_OK), build.RATES_BIN


def test_status_strings(lib):
    for code in range(8):
        assert gp.gemm_status_string(code).startswith("GP_")
    assert "unknown" in gp.gemm_status_string(99)


@pytest.mark.parametrize("dtype,N,K,expect", [
    ("e4m3", 256, 512, 256 * 512),
    ("int8", 7168, 4096, 7168 * 4096),
    ("bf16", 4096, 4096, 4096 * 4096 * 2),
    ("e2m1", 8192, 8192, 8192 * 4096 + 8192 * 256),
    ("bf16", 128, 64, 128 * 128),
    ("e4m3", 0, 0, 0),
    ("fp16", 256, 64, 256 * 64 * 2),
])
def test_packed_bytes(lib, dtype, N, K, expect):
    assert gp.gemm_packed_b_bytes(dtype, N, K) == expect


@pytest.mark.parametrize("dtype,N,K", [("e4m3", 100, 512), ("e4m3", 128, 100), ("bf16", 128, 32),
                                       ("e2m1", 128, 128), ("int8", -128, 128)])
def test_packed_bytes_shape_errors(lib, dtype, N, K):
    with pytest.raises(gp.GemmError) as e:
        gp.gemm_packed_b_bytes(dtype, N, K)
    assert e.value.code == 3


def test_bad_dtype(lib):
    out = ctypes.c_size_t()
    assert lib.gemm_packed_b_bytes(9, 128, 128, ctypes.byref(out)) == 1


FAKE = 0x10000  # an aligned, never-dereferenced address: validation fails before any use


@pytest.mark.parametrize("args,code", [
    # unsupported combinations
    (dict(dtype="int8", scale_mode="none", c_dtype="bf16"), 2),
    (dict(dtype="bf16", scale_mode="rowcol_f32", c_dtype="bf16"), 2),
    (dict(dtype="e2m1", scale_mode="none", c_dtype="bf16"), 2),
    (dict(dtype="fp16", scale_mode="rowcol_f32", c_dtype="fp16", scale_a=FAKE, scale_b=FAKE), 2),
    (dict(dtype="int8", scale_mode="none", c_dtype="fp16"), 2),
    # shape rules
    (dict(N=100), 3),
    (dict(K=96), 3),
    (dict(M=-1), 3),
    (dict(dtype="int8", c_dtype="int32", K=262144), 3),
    # pointers
    (dict(C=0), 1),
    (dict(A=0), 1),
    (dict(scale_mode="rowcol_f32", scale_a=None, scale_b=FAKE), 1),
    (dict(A=FAKE + 8), 4),
    (dict(C=FAKE + 4), 4),
])
def test_gemm_run_validation(lib, args, code):
    a = dict(A=FAKE, B=FAKE, dtype="e4m3", M=16, N=256, K=512, scale_mode="none", scale_a=None, scale_b=None,
             C=FAKE, c_dtype="bf16")
    a.update(args)
    rc = lib.gemm_run(a["A"] or None, a["B"], gp.DTYPES[a["dtype"]], a["M"], a["N"], a["K"],
                      gp.SCALE_MODES[a["scale_mode"]], a["scale_a"], a["scale_b"], a["C"] or None,
                      gp.DTYPES[a["c_dtype"]], None)
    assert rc == code


def test_empty_problem_is_a_noop(lib):
    # M == 0: nothing to compute, nothing touched, no CUDA call needed
    assert lib.gemm_run(None, None, gp.DTYPES["e4m3"], 0, 256, 512, 0, None, None, None, gp.DTYPES["bf16"], None) == 0
    assert lib.gemm_preshuffle_b(None, None, gp.DTYPES["int8"], 0, 128, None, None) == 0


def test_run_ex_rejects_unknown_flags(lib):
    rc = lib.gemm_run_ex(FAKE, FAKE, gp.DTYPES["e4m3"], 16, 256, 512, 0, None, None, 0, None, FAKE,
                         gp.DTYPES["bf16"], 4, None)
    assert rc == 1
    # the known flag passes validation; a shape error is still reported first-class
    rc = lib.gemm_run_ex(FAKE, FAKE, gp.DTYPES["e4m3"], 16, 100, 512, 0, None, None, 0, None, FAKE,
                         gp.DTYPES["bf16"], gp.GP_RUN_B_CONSTANT, None)
    assert rc == 3
    for f in (gp.GP_RUN_INDEPENDENT, gp.GP_RUN_B_CONSTANT | gp.GP_RUN_INDEPENDENT):
        rc = lib.gemm_run_ex(FAKE, FAKE, gp.DTYPES["int8"], 16, 100, 512, 0, None, None, 0, None, FAKE,
                             gp.DTYPES["int32"], f, None)
        assert rc == 3


@pytest.mark.parametrize("dtype,k_ok,k_bad", [("int8", 130944, 131072), ("w4a8", 2096896, 2097152)])
def test_integer_k_limit_keeps_the_exact_result_in_int32(lib, dtype, k_ok, k_bad):
    # at k_bad, (-128) * (-128) * K (int8) or (-128) * (-8) * K (int4) reaches
    # 2^31; M = 0 makes a valid call a no-op (the shape rules still apply)
    assert lib.gemm_run_ex(None, None, gp.DTYPES[dtype], 0, 256, k_bad, 0, None, None, 0, None, None,
                           gp.DTYPES["int32"], 0, None) == 3
    assert lib.gemm_run_ex(None, None, gp.DTYPES[dtype], 0, 256, k_ok, 0, None, None, 0, None, None,
                           gp.DTYPES["int32"], 0, None) == 0


@pytest.mark.parametrize("epi,bias,dtype,c_dtype,code", [
    (5, FAKE, "e4m3", "bf16", 1),        # unknown epilogue
    (-1, FAKE, "e4m3", "bf16", 1),
    (1, None, "e4m3", "bf16", 1),        # an epilogue needs a bias
    (0, FAKE, "e4m3", "bf16", 1),        # no epilogue takes no bias
    (2, FAKE, "int8", "int32", 2),       # float outputs only
    (4, FAKE + 4, "e4m3", "bf16", 4),    # bias must be 16-byte aligned
])
def test_run_ex_epilogue_validation(lib, epi, bias, dtype, c_dtype, code):
    mode = 0
    rc = lib.gemm_run_ex(FAKE, FAKE, gp.DTYPES[dtype], 16, 256, 512, mode, None, None, epi, bias, FAKE,
                         gp.DTYPES[c_dtype], 0, None)
    assert rc == code


@pytest.mark.parametrize("xd,qd,M,K,X,A,S,code", [
    ("e4m3", "e4m3", 4, 64, FAKE, FAKE, FAKE, 1),     # input must be fp32 or bf16
    ("fp32", "bf16", 4, 64, FAKE, FAKE, FAKE, 1),     # output must be e4m3 or e2m1
    ("fp32", "e4m3", 4, 48, FAKE, FAKE, FAKE, 3),     # K % 32
    ("fp32", "e2m1", -1, 64, FAKE, FAKE, FAKE, 3),
    ("fp32", "e4m3", 4, 64, None, FAKE, FAKE, 1),
    ("bf16", "e2m1", 4, 64, FAKE, FAKE + 8, FAKE, 4),
    ("fp32", "e4m3", 0, 64, None, None, None, 0),     # empty: no-op, nothing touched
])
def test_quantize_validation(lib, xd, qd, M, K, X, A, S, code):
    assert lib.gemm_quantize_a(X, gp.DTYPES[xd], M, K, gp.DTYPES[qd], A, S, None) == code

"""GB300 (sm_103a) preshuffle GEMM:  C[M,N] = A[M,K] . B[N,K]^T.

A thin ctypes binding over the C ABI in ``include/gemm_preshuffle.h``, with
the same function names.  It only marshals arguments: torch tensors become
device pointers, and the current torch stream becomes the launch stream.
Every step of the computation runs in the library's CUDA kernels.  If the
native library is missing, the binding raises instead of falling back.

Build the library with ``python -c "import __graft_entry__ as g; g.build()"``
(or ``python dense_gemm_preshuffle_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

__all__ = [
    "GP_OK", "GemmError", "DTYPES", "SCALE_MODES", "load_library", "library_path",
    "gemm_packed_b_bytes", "gemm_preshuffle_b", "gemm_unpack_b", "gemm_run",
    "gemm_last_device_status", "gemm_status_string", "gemm_debug_skip_load",
    "preshuffle_b", "matmul",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libgemm_preshuffle.so")
_HEADER = os.path.join(os.path.dirname(_HERE), "include", "gemm_preshuffle.h")

GP_OK = 0
DTYPES = {"bf16": 0, "e4m3": 1, "int8": 2, "e2m1": 3, "int32": 4, "fp16": 5, "fp32": 6, "w4a8": 7}
SCALE_MODES = {"none": 0, "rowcol_f32": 1, "block32_ue8m0": 2}
GP_RUN_DEFAULT = 0
GP_RUN_B_CONSTANT = 1
GP_RUN_INDEPENDENT = 2
EPILOGUES = {"none": 0, "bias": 1, "bias_relu": 2, "bias_silu": 3, "bias_gelu": 4}

_lib = None


class GemmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {gemm_status_string(code)} (status {code})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the native library; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"native library {_LIB_PATH} is missing: build it with "
            "`python -c \"import __graft_entry__ as g; g.build()\"` (needs nvcc 13)")
    lib = ctypes.CDLL(_LIB_PATH)
    i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.gemm_packed_b_bytes.argtypes = [i32, i64, i64, ctypes.POINTER(ctypes.c_size_t)]
    lib.gemm_preshuffle_b.argtypes = [vp, vp, i32, i64, i64, vp, vp]
    lib.gemm_unpack_b.argtypes = [vp, i32, i64, i64, vp, vp, vp]
    lib.gemm_run.argtypes = [vp, vp, i32, i64, i64, i64, i32, vp, vp, vp, i32, vp]
    lib.gemm_run_ex.argtypes = [vp, vp, i32, i64, i64, i64, i32, vp, vp, i32, vp, vp, i32, ctypes.c_uint, vp]
    lib.gemm_quantize_a.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp]
    lib.gemm_last_device_status.argtypes = [vp]
    lib.gemm_status_string.argtypes = [i32]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_debug_skip_load.argtypes = [i32]
    for name in ("gemm_packed_b_bytes", "gemm_preshuffle_b", "gemm_unpack_b", "gemm_run", "gemm_run_ex",
                 "gemm_quantize_a",
                 "gemm_last_device_status", "gemm_debug_skip_load"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def header_functions() -> list:
    """Names of the functions declared in include/gemm_preshuffle.h."""
    text = open(_HEADER).read()
    return re.findall(r"^\s*(?:int|const char\*)\s+(gemm_\w+)\s*\(", text, flags=re.M)


# ----------------------------------------------------------------- marshalling

def _dt(x) -> int:
    return DTYPES[x] if isinstance(x, str) else int(x)


def _sm(x) -> int:
    return SCALE_MODES[x] if isinstance(x, str) else int(x)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str) -> None:
    if code != GP_OK:
        raise GemmError(code, where)


# ----------------------------------------------------------------- the C ABI

def gemm_status_string(code: int) -> str:
    return load_library().gemm_status_string(int(code)).decode()


def gemm_packed_b_bytes(dtype, N: int, K: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().gemm_packed_b_bytes(_dt(dtype), N, K, ctypes.byref(out)), "gemm_packed_b_bytes")
    return out.value


def gemm_preshuffle_b(B, B_scales, dtype, N: int, K: int, B_packed, stream=None) -> None:
    _check(load_library().gemm_preshuffle_b(_ptr(B), _ptr(B_scales), _dt(dtype), N, K, _ptr(B_packed),
                                            _stream(stream)), "gemm_preshuffle_b")


def gemm_unpack_b(B_packed, dtype, N: int, K: int, B_out, B_scales_out=None, stream=None) -> None:
    _check(load_library().gemm_unpack_b(_ptr(B_packed), _dt(dtype), N, K, _ptr(B_out), _ptr(B_scales_out),
                                        _stream(stream)), "gemm_unpack_b")


def gemm_run(A, B_packed, dtype, M: int, N: int, K: int, scale_mode, scale_a, scale_b, C, c_dtype,
             stream=None) -> None:
    _check(load_library().gemm_run(_ptr(A), _ptr(B_packed), _dt(dtype), M, N, K, _sm(scale_mode), _ptr(scale_a),
                                   _ptr(scale_b), _ptr(C), _dt(c_dtype), _stream(stream)), "gemm_run")


def _epi(x) -> int:
    return EPILOGUES[x] if isinstance(x, str) else int(x)


def gemm_run_ex(A, B_packed, dtype, M: int, N: int, K: int, scale_mode, scale_a, scale_b, epilogue, bias, C,
                c_dtype, flags: int = GP_RUN_DEFAULT, stream=None) -> None:
    _check(load_library().gemm_run_ex(_ptr(A), _ptr(B_packed), _dt(dtype), M, N, K, _sm(scale_mode),
                                      _ptr(scale_a), _ptr(scale_b), _epi(epilogue), _ptr(bias), _ptr(C),
                                      _dt(c_dtype), int(flags), _stream(stream)), "gemm_run_ex")


def gemm_quantize_a(X, x_dtype, M: int, K: int, q_dtype, A_out, scales_out, stream=None) -> None:
    _check(load_library().gemm_quantize_a(_ptr(X), _dt(x_dtype), M, K, _dt(q_dtype), _ptr(A_out), _ptr(scales_out),
                                          _stream(stream)), "gemm_quantize_a")


def quantize(X, q_dtype, stream=None):
    """Quantise a device tensor X [M, K] (fp32 or bf16) for gemm_run's A.
    Returns (A codes, scale_a): E4M3 -> (uint8 [M, K], fp32 [M]);
    E2M1 -> (uint8 [M, K/2], uint8 [M, K/32])."""
    import torch
    M, K = X.shape
    xd = "bf16" if X.dtype == torch.bfloat16 else "fp32"
    if _dt(q_dtype) == DTYPES["e4m3"]:
        A = torch.empty((M, K), dtype=torch.uint8, device=X.device)
        S = torch.empty((M,), dtype=torch.float32, device=X.device)
    else:
        A = torch.empty((M, K // 2), dtype=torch.uint8, device=X.device)
        S = torch.empty((M, K // 32), dtype=torch.uint8, device=X.device)
    gemm_quantize_a(X, xd, M, K, q_dtype, A, S, stream)
    return A, S


def gemm_last_device_status(stream=None) -> int:
    return int(load_library().gemm_last_device_status(_stream(stream)))


def gemm_debug_skip_load(index: int) -> None:
    _check(load_library().gemm_debug_skip_load(int(index)), "gemm_debug_skip_load")


# ----------------------------------------------------------------- conveniences

def preshuffle_b(B, dtype, B_scales=None, stream=None):
    """Pack a device tensor B [N, K] (E2M1: [N, K/2] bytes) into a new uint8 tensor."""
    import torch
    N = B.shape[0]
    K = B.shape[1] * (2 if _dt(dtype) in (DTYPES["e2m1"], DTYPES["w4a8"]) else 1)
    out = torch.empty(gemm_packed_b_bytes(dtype, N, K), dtype=torch.uint8, device=B.device)
    gemm_preshuffle_b(B, B_scales, dtype, N, K, out, stream)
    return out


def matmul(A, B_packed, dtype, N: int, K: int, scale_a=None, scale_b=None, out=None, stream=None,
           b_constant: bool = False, epilogue: str = "none", bias=None, out_dtype: Optional[str] = None,
           independent: bool = False):
    """C = A . B^T with B packed; returns [M, N] in out_dtype ("bf16" or
    "fp16"; default fp16 for fp16 operands, bf16 for the other float types),
    int32 for int8.

    epilogue: "none", "bias", "bias_relu", "bias_silu" or "bias_gelu", with
    bias an fp32 [N] device tensor for all but "none".
    b_constant=True passes GP_RUN_B_CONSTANT: B_packed must not be written
    by any GPU work still in flight (pack once, then synchronise).
    independent=True passes GP_RUN_INDEPENDENT: no GPU work still in flight
    writes any operand of the call or touches `out`."""
    import torch
    d = _dt(dtype)
    M = A.shape[0]
    if out_dtype is None:
        out_dtype = "fp16" if d == DTYPES["fp16"] else "bf16"
    fdt = torch.float16 if out_dtype == "fp16" else torch.bfloat16
    if d in (DTYPES["int8"], DTYPES["w4a8"]):
        c_dtype, mode, tdt = "int32", "none", torch.int32
    elif d == DTYPES["e2m1"]:
        c_dtype, mode, tdt = out_dtype, "block32_ue8m0", fdt
    elif scale_a is not None:
        c_dtype, mode, tdt = out_dtype, "rowcol_f32", fdt
    else:
        c_dtype, mode, tdt = out_dtype, "none", fdt
    if out is None:
        out = torch.empty((M, N), dtype=tdt, device=A.device)
    gemm_run_ex(A, B_packed, d, M, N, K, mode, scale_a, scale_b, epilogue, bias, out, c_dtype,
                (GP_RUN_B_CONSTANT if b_constant else GP_RUN_DEFAULT) | (GP_RUN_INDEPENDENT if independent else 0),
                stream)
    return out

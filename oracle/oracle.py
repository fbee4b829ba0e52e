"""Python access to the plain CPU oracle in ``gemm_oracle.c``.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this module. The GPU library
(``dense_gemm_row_gb300``) never imports it and shares no code with it.

The oracle computes the definition of a row-major dense GEMM,
``C = alpha*A*B + beta*C`` ("Sgemm [128,128,8]", the comment above the kernel
and the host reference routine host_gemm), accumulating in float64 for fp32,
bf16 and fp16 inputs and in int64 for int8 inputs (C++ warp-matrix-function
page, type table). The C source states every reading it takes of the pages.

Inputs are torch CPU tensors, 2-D, with unit column stride; the row stride is
the leading dimension, so padded rows are supported and the padding is never
read. Results come back as numpy arrays: float64 (unrounded) for the floating
entry points, int32 for int8.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_LOCK = threading.Lock()
_LIB = None

_BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    for extra in (["-fopenmp"], []):
        cmd = ["gcc", *_BASE_FLAGS, *extra, _SRC, "-o", tmp, "-lm"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode == 0:
            os.replace(tmp, _LIB_PATH)
            return _LIB_PATH
    raise RuntimeError("oracle build failed:\n" + res.stderr)


def load(path: str):
    """Load an oracle library from ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    i64, f64, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    for name in ("oracle_gemm_f64", "oracle_gemm_f32", "oracle_gemm_bf16", "oracle_gemm_f16"):
        fn = getattr(lib, name)
        fn.argtypes = [i64, i64, i64, f64, vp, i64, vp, i64, f64, vp, i64]
        fn.restype = ctypes.c_int
    for name in ("oracle_gemm_s8", "oracle_gemm_u8"):
        fn = getattr(lib, name)
        fn.argtypes = [i64, i64, i64, ctypes.c_int32, vp, i64, vp, i64, ctypes.c_int32, vp, i64]
        fn.restype = ctypes.c_int
    lib.oracle_gemm_tf32.argtypes = [i64, i64, i64, f64, vp, i64, vp, i64, f64, vp, i64]
    lib.oracle_gemm_tf32.restype = ctypes.c_int
    for name in ("oracle_gemm_f16_f16", "oracle_gemm_bf16_bf16"):
        fn = getattr(lib, name)
        fn.argtypes = [i64, i64, i64, f64, vp, i64, vp, i64, f64, vp, i64]
        fn.restype = ctypes.c_int
    lib.oracle_encode_f16.argtypes = [f64]
    lib.oracle_encode_f16.restype = ctypes.c_uint16
    lib.oracle_encode_bf16.argtypes = [f64]
    lib.oracle_encode_bf16.restype = ctypes.c_uint16
    lib.oracle_round_tf32.argtypes = [ctypes.c_float]
    lib.oracle_round_tf32.restype = ctypes.c_float
    lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_bf16.restype = f64
    lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_f16.restype = f64
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = load(build())
        return _LIB


def num_threads() -> int:
    """Host threads the oracle runs on (OpenMP max threads, 1 without OpenMP)."""
    return int(_lib().oracle_num_threads())


def _ld(t: torch.Tensor, name: str) -> int:
    if t.device.type != "cpu":
        raise ValueError(f"oracle: {name} must be a CPU tensor")
    if t.dim() != 2:
        raise ValueError(f"oracle: {name} must be 2-D")
    if t.shape[0] > 0 and t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"oracle: {name} needs unit column stride")
    return max(int(t.stride(0)), int(t.shape[1]), 1)


def _check(status: int) -> None:
    if status != 0:
        raise ValueError(f"oracle: status {status}")


_FLOAT_DTYPES = {
    torch.float32: "oracle_gemm_f32",
    torch.bfloat16: "oracle_gemm_bf16",
    torch.float16: "oracle_gemm_f16",
    torch.float64: "oracle_gemm_f64",
}


def gemm(A: torch.Tensor, B: torch.Tensor, alpha: float = 1.0, beta: float = 0.0,
         C0: torch.Tensor | np.ndarray | None = None, tf32: bool = False) -> np.ndarray:
    """C = alpha*A*B + beta*C0 for float32/bfloat16/float16/float64 A and B.

    Returns the float64 result, not rounded to the inputs' type. ``C0`` (any
    float type, converted exactly to float64) is not read when beta == 0.
    tf32=True (float32 A and B only): the inputs are first reduced to tf32.
    """
    if A.dtype != B.dtype or A.dtype not in _FLOAT_DTYPES:
        raise TypeError("oracle.gemm: A and B must share one float dtype")
    if tf32 and A.dtype != torch.float32:
        raise TypeError("oracle.gemm: tf32 takes float32 inputs")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("oracle.gemm: inner dimensions differ")
    lda, ldb = _ld(A, "A"), _ld(B, "B")
    if C0 is None:
        C = np.zeros((M, N), dtype=np.float64)
    else:
        c0 = C0.detach().cpu().to(torch.float64).numpy() if isinstance(C0, torch.Tensor) \
            else np.asarray(C0, dtype=np.float64)
        C = np.array(c0, dtype=np.float64, order="C", copy=True)
        if C.shape != (M, N):
            raise ValueError("oracle.gemm: C0 has the wrong shape")
    fn = getattr(_lib(), "oracle_gemm_tf32" if tf32 else _FLOAT_DTYPES[A.dtype])
    _check(fn(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb, float(beta),
              C.ctypes.data, max(N, 1)))
    return C


def gemm_out16(A: torch.Tensor, B: torch.Tensor, alpha: float = 1.0, beta: float = 0.0,
               C0: torch.Tensor | None = None) -> torch.Tensor:
    """16-bit A, B and C of one format (float16 or bfloat16): the exact result
    rounded once to that format. Returns a CPU tensor of the inputs' dtype."""
    if A.dtype != B.dtype or A.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("oracle.gemm_out16: A and B must both be float16 or bfloat16")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("oracle.gemm_out16: inner dimensions differ")
    lda, ldb = _ld(A, "A"), _ld(B, "B")
    if C0 is None:
        C = torch.zeros((M, N), dtype=A.dtype)
    else:
        if C0.dtype != A.dtype or tuple(C0.shape) != (M, N):
            raise ValueError("oracle.gemm_out16: C0 must be M x N of the inputs' dtype")
        C = C0.detach().cpu().contiguous().clone()
    name = "oracle_gemm_bf16_bf16" if A.dtype == torch.bfloat16 else "oracle_gemm_f16_f16"
    _check(getattr(_lib(), name)(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                                 float(beta), C.data_ptr(), max(N, 1)))
    return C


def gemm_s8(A: torch.Tensor, B: torch.Tensor, alpha: int = 1, beta: int = 0,
            C0: torch.Tensor | np.ndarray | None = None) -> np.ndarray:
    """int8 (or uint8) A and B, int64 accumulation, int32 wrap-around output."""
    if A.dtype != B.dtype or A.dtype not in (torch.int8, torch.uint8):
        raise TypeError("oracle.gemm_s8: A and B must both be int8 or both uint8")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("oracle.gemm_s8: inner dimensions differ")
    lda, ldb = _ld(A, "A"), _ld(B, "B")
    if C0 is None:
        C = np.zeros((M, N), dtype=np.int32)
    else:
        c0 = C0.detach().cpu().numpy() if isinstance(C0, torch.Tensor) else np.asarray(C0)
        if c0.dtype != np.int32:
            raise TypeError("oracle.gemm_s8: C0 must be int32")
        C = np.array(c0, dtype=np.int32, order="C", copy=True)
        if C.shape != (M, N):
            raise ValueError("oracle.gemm_s8: C0 has the wrong shape")
    fn = _lib().oracle_gemm_u8 if A.dtype == torch.uint8 else _lib().oracle_gemm_s8
    _check(fn(M, N, K, int(alpha), A.data_ptr(), lda, B.data_ptr(), ldb, int(beta),
              C.ctypes.data, max(N, 1)))
    return C


gemm_u8 = gemm_s8


def gemm_rows(A: torch.Tensor, B: torch.Tensor, rows, alpha=1.0, beta=0.0, C0=None):
    """The oracle restricted to the listed output rows (for sampled checks at full
    size). Rows of C are independent, so this is the same computation as the
    full oracle followed by selecting those rows."""
    idx = torch.as_tensor(rows, dtype=torch.long)
    a = A.index_select(0, idx).contiguous()
    c0 = None
    if C0 is not None:
        c0t = C0 if isinstance(C0, torch.Tensor) else torch.from_numpy(np.asarray(C0))
        c0 = c0t.index_select(0, idx)
    if A.dtype in (torch.int8, torch.uint8):
        return gemm_s8(a, B, int(alpha), int(beta), c0)
    return gemm(a, B, alpha, beta, c0)


def decode_bf16(bits: int) -> float:
    return float(_lib().oracle_decode_bf16(bits))


def decode_f16(bits: int) -> float:
    return float(_lib().oracle_decode_f16(bits))


def encode_f16(x: float) -> int:
    """Bits of x rounded to IEEE binary16 (nearest, ties to even)."""
    return int(_lib().oracle_encode_f16(float(x)))


def encode_bf16(x: float) -> int:
    """Bits of x rounded to bfloat16 (nearest, ties to even)."""
    return int(_lib().oracle_encode_bf16(float(x)))


def round_tf32(x: float) -> float:
    """The fp32 value x reduced to tf32 (13 lowest fraction bits cleared)."""
    return float(_lib().oracle_round_tf32(float(x)))

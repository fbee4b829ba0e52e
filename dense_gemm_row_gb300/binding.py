"""ctypes binding of libdense_gemm_row.so (include/dense_gemm_row.h).

Argument marshalling only: every step of the computation runs in the CUDA
library. Importing this module loads the library and raises ImportError when
it has not been built; there is no fallback.

Two layers:

* ``gemm_f32 / gemm_bf16 / gemm_f16 / gemm_s8(M, N, K, alpha, A, lda, B, ldb,
  beta, C, ldc, stream=None)`` mirror the C entry points. A, B and C are raw
  device addresses (int) or tensors (their ``data_ptr()`` is passed). ``stream``
  is a raw ``cudaStream_t`` (int), a ``torch.cuda.Stream``, or None for torch's
  current stream. A non-zero status raises :class:`GemmError`.
* ``gemm(A, B, C, alpha, beta)`` takes 2-D CUDA tensors with unit column stride
  (row stride = leading dimension), picks the entry point from A's dtype and
  runs on torch's current stream.

The extended entry points (strided-batched GEMM with transposed operands) have
the same two layers: ``gemm_f32_ex / gemm_bf16_ex / gemm_f16_ex / gemm_s8_ex(
opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
strideC, batch, stream=None)`` (opX: OP_N or OP_T) and ``gemm_batched(A, B, C,
alpha, beta, trans_a=False, trans_b=False)`` for 3-D tensors (a 2-D operand,
or one expanded along the batch with stride 0, is shared by every entry).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdense_gemm_row.so")

STATUS = {
    0: "GEMM_OK",
    1: "GEMM_ERR_INVALID_VALUE",
    2: "GEMM_ERR_UNSUPPORTED_LAYOUT",
    3: "GEMM_ERR_LAUNCH",
    4: "GEMM_ERR_DEVICE",
    5: "GEMM_ERR_TIMEOUT",
    6: "GEMM_ERR_TOO_LARGE",
}

# Every function include/dense_gemm_row.h declares.
EXPORTED = ("gemm_f32", "gemm_bf16", "gemm_f16", "gemm_s8", "gemm_u8", "gemm_f16_f16",
            "gemm_bf16_bf16", "gemm_tf32", "gemm_f64", "gemm_f32_ex", "gemm_bf16_ex",
            "gemm_f16_ex", "gemm_s8_ex", "gemm_s8_noalloc", "gemm_status_string",
            "gemm_check_device_error", "gemm_selftest_wait_timeout", "gemm_last_launch_error",
            "gemm_peak_ffma", "gemm_peak_tc_f16", "gemm_pool_usage", "gemm_version")

OP_N, OP_T = 0, 1  # gemm_op_t


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = int(status)
        msg = f"{where}: {STATUS.get(self.status, self.status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m dense_gemm_row_gb300.build` "
            "(or __graft_entry__.build()). There is no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    f32, i32 = ctypes.c_float, ctypes.c_int32
    for name in ("gemm_f32", "gemm_bf16", "gemm_f16", "gemm_f16_f16", "gemm_bf16_bf16",
                 "gemm_tf32"):
        fn = getattr(lib, name)
        fn.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        fn.restype = ctypes.c_int
    f64 = ctypes.c_double
    lib.gemm_f64.argtypes = [i64, i64, i64, f64, vp, i64, vp, i64, f64, vp, i64, vp]
    lib.gemm_f64.restype = ctypes.c_int
    for name in ("gemm_s8", "gemm_s8_noalloc", "gemm_u8"):
        fn = getattr(lib, name)
        fn.argtypes = [i64, i64, i64, i32, vp, i64, vp, i64, i32, vp, i64, vp]
        fn.restype = ctypes.c_int
    op = ctypes.c_int
    for name, sc in (("gemm_f32_ex", f32), ("gemm_bf16_ex", f32), ("gemm_f16_ex", f32),
                     ("gemm_s8_ex", i32)):
        fn = getattr(lib, name)
        fn.argtypes = [op, op, i64, i64, i64, sc, vp, i64, i64, vp, i64, i64, sc, vp, i64, i64,
                       i64, vp]
        fn.restype = ctypes.c_int
    lib.gemm_status_string.argtypes = [ctypes.c_int]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_check_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.gemm_check_device_error.restype = ctypes.c_int
    lib.gemm_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
    lib.gemm_selftest_wait_timeout.restype = ctypes.c_int
    lib.gemm_last_launch_error.argtypes = []
    lib.gemm_last_launch_error.restype = ctypes.c_char_p
    lib.gemm_peak_ffma.argtypes = [i32, vp, ctypes.POINTER(f64), vp]
    lib.gemm_peak_ffma.restype = ctypes.c_int
    lib.gemm_peak_tc_f16.argtypes = [i32, ctypes.POINTER(f64), vp]
    lib.gemm_peak_tc_f16.restype = ctypes.c_int
    lib.gemm_version.argtypes = []
    lib.gemm_version.restype = ctypes.c_int
    lib.gemm_pool_usage.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.c_int]
    lib.gemm_pool_usage.restype = ctypes.c_int
    return lib


lib = _load()


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(status: int, where: str) -> None:
    if status != 0:
        detail = lib.gemm_last_launch_error().decode() if status == 3 else ""
        raise GemmError(status, where, detail)


def gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_f32(M, N, K, alpha, _addr(A), lda, _addr(B), ldb, beta, _addr(C), ldc,
                        _stream(stream)), "gemm_f32")


def gemm_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_bf16(M, N, K, alpha, _addr(A), lda, _addr(B), ldb, beta, _addr(C), ldc,
                         _stream(stream)), "gemm_bf16")


def gemm_f16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_f16(M, N, K, alpha, _addr(A), lda, _addr(B), ldb, beta, _addr(C), ldc,
                        _stream(stream)), "gemm_f16")


def gemm_s8(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_s8(M, N, K, int(alpha), _addr(A), lda, _addr(B), ldb, int(beta), _addr(C),
                       ldc, _stream(stream)), "gemm_s8")


def gemm_u8(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_u8(M, N, K, int(alpha), _addr(A), lda, _addr(B), ldb, int(beta), _addr(C),
                       ldc, _stream(stream)), "gemm_u8")


def gemm_f16_f16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_f16_f16(M, N, K, alpha, _addr(A), lda, _addr(B), ldb, beta, _addr(C), ldc,
                            _stream(stream)), "gemm_f16_f16")


def gemm_bf16_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_bf16_bf16(M, N, K, alpha, _addr(A), lda, _addr(B), ldb, beta, _addr(C), ldc,
                              _stream(stream)), "gemm_bf16_bf16")


def gemm_tf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_tf32(M, N, K, alpha, _addr(A), lda, _addr(B), ldb, beta, _addr(C), ldc,
                         _stream(stream)), "gemm_tf32")


def gemm_f64(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(lib.gemm_f64(M, N, K, float(alpha), _addr(A), lda, _addr(B), ldb, float(beta),
                        _addr(C), ldc, _stream(stream)), "gemm_f64")


def gemm_s8_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    """gemm_s8 on the library's fixed scratch array: allocates no device memory.
    Problems needing more than 64 MiB of widened operands raise GemmError
    (GEMM_ERR_TOO_LARGE); calls that overlap on the GPU race on the array."""
    _check(lib.gemm_s8_noalloc(M, N, K, int(alpha), _addr(A), lda, _addr(B), ldb, int(beta),
                               _addr(C), ldc, _stream(stream)), "gemm_s8_noalloc")


def _ex(name, cast):
    def call(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC,
             batch, stream=None):
        _check(getattr(lib, name)(int(opA), int(opB), M, N, K, cast(alpha), _addr(A), lda,
                                  strideA, _addr(B), ldb, strideB, cast(beta), _addr(C), ldc,
                                  strideC, batch, _stream(stream)), name)
    call.__name__ = name
    call.__doc__ = (f"{name}: strided-batched C_b = alpha*op(A_b)*op(B_b) + beta*C_b "
                    "(include/dense_gemm_row.h).")
    return call


gemm_f32_ex = _ex("gemm_f32_ex", float)
gemm_bf16_ex = _ex("gemm_bf16_ex", float)
gemm_f16_ex = _ex("gemm_f16_ex", float)
gemm_s8_ex = _ex("gemm_s8_ex", int)


def peak_ffma(iters, sink, stream=None) -> float:
    """Enqueue the packed-FP32-FMA peak microbenchmark; returns its flop count."""
    f = ctypes.c_double(0.0)
    _check(lib.gemm_peak_ffma(int(iters), _addr(sink), ctypes.byref(f), _stream(stream)),
           "gemm_peak_ffma")
    return f.value


def peak_tc_f16(iters, stream=None) -> float:
    """Enqueue the tcgen05 kind::f16 peak microbenchmark; returns its flop count."""
    f = ctypes.c_double(0.0)
    _check(lib.gemm_peak_tc_f16(int(iters), ctypes.byref(f), _stream(stream)), "gemm_peak_tc_f16")
    return f.value


def pool_usage(reset_high: bool = False) -> tuple[int, int]:
    """(high-water mark of bytes in use, bytes reserved) of the library's memory
    pool on the current device; reset_high clears the mark after reading."""
    used = ctypes.c_int64(0)
    reserved = ctypes.c_int64(0)
    _check(lib.gemm_pool_usage(ctypes.byref(used), ctypes.byref(reserved), int(reset_high)),
           "gemm_pool_usage")
    return used.value, reserved.value


def check_device_error() -> int:
    """Reads and clears the device error word; raises GemmError(GEMM_ERR_TIMEOUT)
    if a kernel gave up a bounded wait. Returns the raw word otherwise (0)."""
    w = ctypes.c_uint32(0)
    st = lib.gemm_check_device_error(ctypes.byref(w))
    if st != 0:
        raise GemmError(st, f"device error word 0x{w.value:08x}")
    return int(w.value)


def _ld(t, name) -> int:
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.shape[0] > 0 and t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} needs unit column stride (row-major)")
    return max(int(t.stride(0)), int(t.shape[1]), 1)


def gemm(A, B, C, alpha=1.0, beta=0.0, stream=None, tf32=False):
    """C = alpha*A*B + beta*C for 2-D CUDA tensors; the dtypes select the entry
    point: float32 -> gemm_f32 (gemm_tf32 with tf32=True), float64 -> gemm_f64,
    bfloat16 / float16 with a float32 C -> gemm_bf16 / gemm_f16, with a C of the
    inputs' dtype -> gemm_bf16_bf16 / gemm_f16_f16, int8 -> gemm_s8 and uint8
    -> gemm_u8 (C int32)."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError("gemm: shapes do not chain (A: MxK, B: KxN, C: MxN)")
    if A.dtype != B.dtype:
        raise TypeError("gemm: A and B must share a dtype")
    fns = {torch.float32: (gemm_tf32 if tf32 else gemm_f32, torch.float32),
           torch.float64: (gemm_f64, torch.float64),
           torch.bfloat16: (gemm_bf16, torch.float32), torch.float16: (gemm_f16, torch.float32),
           torch.int8: (gemm_s8, torch.int32), torch.uint8: (gemm_u8, torch.int32)}
    if A.dtype not in fns:
        raise TypeError(f"gemm: unsupported dtype {A.dtype}")
    fn, c_dtype = fns[A.dtype]
    if A.dtype in (torch.bfloat16, torch.float16) and C.dtype == A.dtype:
        fn, c_dtype = (gemm_bf16_bf16 if A.dtype == torch.bfloat16 else gemm_f16_f16), A.dtype
    if C.dtype != c_dtype:
        raise TypeError(f"gemm: C must be {c_dtype} for {A.dtype} inputs")
    fn(M, N, K, alpha, A, _ld(A, "A"), B, _ld(B, "B"), beta, C, _ld(C, "C"), stream)
    return C


def _mat(t, name):
    """(matrix stride, row stride) of a 2-D or 3-D operand with unit column
    stride; a 2-D operand is one matrix shared by every batch entry."""
    if t.dim() not in (2, 3):
        raise ValueError(f"{name} must be 2-D or 3-D")
    rows, cols = t.shape[-2], t.shape[-1]
    if rows > 0 and cols > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name} needs unit column stride (row-major)")
    ld = max(int(t.stride(-2)), int(cols), 1)
    mstride = int(t.stride(0)) if t.dim() == 3 and t.shape[0] > 1 else 0
    return mstride, ld


def gemm_batched(A, B, C, alpha=1.0, beta=0.0, trans_a=False, trans_b=False, stream=None):
    """C[b] = alpha * op(A[b]) * op(B[b]) + beta * C[b] for CUDA tensors.

    C is (batch, M, N). A is (batch, M, K), or (batch, K, M) with trans_a; B is
    (batch, K, N), or (batch, N, K) with trans_b. A 2-D A or B (or one expanded
    along the batch, stride 0) is shared by every entry. Rows must have unit
    column stride; row and matrix strides are passed through. dtypes as gemm()."""
    import torch
    if C.dim() != 3:
        raise ValueError("gemm_batched: C must be 3-D (batch, M, N)")
    batch, M, N = C.shape
    K = A.shape[-2] if trans_a else A.shape[-1]
    a_rows = A.shape[-1] if trans_a else A.shape[-2]
    b_k = B.shape[-1] if trans_b else B.shape[-2]
    b_n = B.shape[-2] if trans_b else B.shape[-1]
    if a_rows != M or b_k != K or b_n != N:
        raise ValueError("gemm_batched: shapes do not chain")
    for t, name in ((A, "A"), (B, "B")):
        if t.dim() == 3 and t.shape[0] not in (1, batch):
            raise ValueError(f"gemm_batched: {name} has {t.shape[0]} matrices, C {batch}")
    if A.dtype != B.dtype:
        raise TypeError("gemm_batched: A and B must share a dtype")
    fns = {torch.float32: (gemm_f32_ex, torch.float32),
           torch.bfloat16: (gemm_bf16_ex, torch.float32),
           torch.float16: (gemm_f16_ex, torch.float32), torch.int8: (gemm_s8_ex, torch.int32)}
    if A.dtype not in fns:
        raise TypeError(f"gemm_batched: unsupported dtype {A.dtype}")
    fn, c_dtype = fns[A.dtype]
    if C.dtype != c_dtype:
        raise TypeError(f"gemm_batched: C must be {c_dtype} for {A.dtype} inputs")
    sa, lda = _mat(A, "A")
    sb, ldb = _mat(B, "B")
    sc, ldc = _mat(C, "C")
    fn(OP_T if trans_a else OP_N, OP_T if trans_b else OP_N, M, N, K, alpha, A, lda, sa, B, ldb,
       sb, beta, C, ldc, sc, batch, stream)
    return C

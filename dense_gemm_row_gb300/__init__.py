"""dense_gemm_row_gb300 -- row-major dense GEMM for GB300 (sm_103a).

    C = alpha * A * B + beta * C

The compute path is the C-ABI library ``libdense_gemm_row.so`` built from
``csrc/``; :mod:`dense_gemm_row_gb300.binding` is a thin ctypes binding over
it. Touching a binding name (``gemm_f32``, ``gemm`` ...) loads the library and
raises ImportError if it is missing: there is no fallback path.
"""
import importlib

__all__ = ["gemm_f32", "gemm_bf16", "gemm_f16", "gemm_s8", "gemm_s8_noalloc", "gemm", "GemmError",
           "check_device_error", "lib"]


def __getattr__(name):
    if name in __all__:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)

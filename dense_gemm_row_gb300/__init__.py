"""dense_gemm_row_gb300 -- row-major dense GEMM for GB300 (sm_103a).

    C = alpha * A * B + beta * C

The compute path is the C-ABI library ``libdense_gemm_row.so`` built from
``csrc/``; :mod:`dense_gemm_row_gb300.gemm` is a thin ctypes binding over it.
Importing a binding symbol loads the library and raises if it is missing: there
is no fallback path.
"""

__all__ = ["gemm_f32", "gemm_bf16", "gemm_f16", "gemm_s8", "gemm", "GemmError", "lib"]


def __getattr__(name):
    if name in __all__:
        from . import gemm as _g
        return getattr(_g, name)
    raise AttributeError(name)

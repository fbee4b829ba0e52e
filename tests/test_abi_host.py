"""Host-side checks of the C-ABI library: it loads, exports every symbol the
public header declares, and rejects bad arguments on the host before anything
is launched (these calls never reach the GPU, so they run without one)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dense_gemm_row.h")

OK, INVALID, LAYOUT = 0, 1, 2


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GEMM_API\s+[\w\s\*]+?\b(gemm_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gemm_f32", "gemm_bf16", "gemm_f16", "gemm_s8", "gemm_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(gemm_mod):
    names = declared_functions()
    for n in names:
        assert hasattr(gemm_mod.lib, n), n
    assert set(names) == set(gemm_mod.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", gemm_mod.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported
    # Nothing of the library's internals leaks into the dynamic symbol table.
    assert not [s for s in exported if "dgr" in s]


def test_library_needs_no_cuda_shared_runtime(gemm_mod):
    out = subprocess.run(["readelf", "-d", gemm_mod.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    needed = re.findall(r"Shared library: \[(.+?)\]", out)
    assert not [n for n in needed if n.startswith(("libcudart", "libcuda.", "libtorch"))], needed


def test_status_strings_and_version(gemm_mod):
    lib = gemm_mod.lib
    for code, name in gemm_mod.STATUS.items():
        assert lib.gemm_status_string(code).decode() == name
    assert lib.gemm_status_string(99).decode() == "GEMM_ERR_UNKNOWN"
    assert lib.gemm_version() >= 100


FAKE = 1 << 20  # a non-NULL address that is never dereferenced: checks fail first


PLAIN = ["gemm_f32", "gemm_bf16", "gemm_f16", "gemm_s8", "gemm_u8", "gemm_f16_f16",
         "gemm_bf16_bf16", "gemm_tf32", "gemm_f64"]
INT_ALPHA = ("gemm_s8", "gemm_u8")


@pytest.mark.parametrize("fn", PLAIN)
def test_invalid_arguments_rejected_on_host(gemm_mod, fn):
    f = getattr(gemm_mod.lib, fn)
    a = 1 if fn in INT_ALPHA else 1.0
    cases = [
        (-1, 8, 8, 8, 8, 8),    # negative M
        (8, -1, 8, 8, 8, 8),    # negative N
        (8, 8, -1, 8, 8, 8),    # negative K
        (8, 8, 16, 8, 8, 8),    # lda < K
        (8, 16, 8, 8, 8, 16),   # ldb < N
        (8, 16, 8, 8, 16, 8),   # ldc < N
        (2**31, 8, 8, 8, 8, 8),  # M too large
    ]
    for M, N, K, lda, ldb, ldc in cases:
        assert f(M, N, K, a, FAKE, lda, FAKE, ldb, a, FAKE, ldc, None) == INVALID, (M, N, K)
    # NULL operands of non-empty matrices
    assert f(8, 8, 8, a, None, 8, FAKE, 8, a, FAKE, 8, None) == INVALID
    assert f(8, 8, 8, a, FAKE, 8, None, 8, a, FAKE, 8, None) == INVALID
    assert f(8, 8, 8, a, FAKE, 8, FAKE, 8, a, None, 8, None) == INVALID


@pytest.mark.parametrize("fn", PLAIN)
def test_empty_output_is_a_no_op(gemm_mod, fn):
    f = getattr(gemm_mod.lib, fn)
    a = 1 if fn in INT_ALPHA else 1.0
    assert f(0, 8, 8, a, None, 8, None, 8, a, None, 8, None) == OK
    assert f(8, 0, 8, a, None, 8, None, 8, a, None, 0, None) == OK


@pytest.mark.parametrize("fn", ["gemm_bf16", "gemm_f16", "gemm_f16_f16", "gemm_bf16_bf16"])
def test_tensor_core_layout_rule(gemm_mod, fn):
    """16-byte aligned A and B bases and lda, ldb multiples of 8, else
    GEMM_ERR_UNSUPPORTED_LAYOUT (checked before any device work)."""
    f = getattr(gemm_mod.lib, fn)
    assert f(8, 8, 8, 1.0, FAKE + 2, 8, FAKE, 8, 0.0, FAKE, 8, None) == LAYOUT
    assert f(8, 8, 8, 1.0, FAKE, 8, FAKE + 8, 8, 0.0, FAKE, 8, None) == LAYOUT
    assert f(8, 8, 12, 1.0, FAKE, 12, FAKE, 8, 0.0, FAKE, 8, None) == LAYOUT
    assert f(8, 12, 8, 1.0, FAKE, 8, FAKE, 12, 0.0, FAKE, 12, None) == LAYOUT


EX = ["gemm_f32_ex", "gemm_bf16_ex", "gemm_f16_ex", "gemm_s8_ex"]
N_, T_ = 0, 1


def call_ex(f, fn, opA=N_, opB=N_, M=8, N=8, K=8, A=FAKE, lda=8, sA=64, B=FAKE, ldb=8, sB=64,
            C=FAKE, ldc=8, sC=64, batch=2):
    a = 1 if fn == "gemm_s8_ex" else 1.0
    return f(opA, opB, M, N, K, a, A, lda, sA, B, ldb, sB, a, C, ldc, sC, batch, None)


@pytest.mark.parametrize("fn", EX)
def test_extended_invalid_arguments_rejected_on_host(gemm_mod, fn):
    f = getattr(gemm_mod.lib, fn)
    assert call_ex(f, fn, opA=2) == INVALID               # not a gemm_op_t
    assert call_ex(f, fn, opB=-1) == INVALID
    assert call_ex(f, fn, batch=-1) == INVALID
    assert call_ex(f, fn, batch=2**31) == INVALID
    assert call_ex(f, fn, sA=-8) == INVALID               # negative strides
    assert call_ex(f, fn, sB=-8) == INVALID
    assert call_ex(f, fn, sC=-8) == INVALID
    assert call_ex(f, fn, sC=8 * 7 + 7) == INVALID        # C matrices overlap: < (M-1)*ldc + N
    # Stored row lengths follow the operand form: A^T rows hold M, B^T rows hold K.
    assert call_ex(f, fn, opA=T_, M=16, lda=8) == INVALID
    assert call_ex(f, fn, opB=T_, K=16, lda=16, ldb=8) == INVALID
    assert call_ex(f, fn, opA=N_, K=16, lda=8) == INVALID
    assert call_ex(f, fn, A=None) == INVALID
    assert call_ex(f, fn, C=None) == INVALID


@pytest.mark.parametrize("fn", EX)
def test_extended_empty_is_a_no_op(gemm_mod, fn):
    f = getattr(gemm_mod.lib, fn)
    assert call_ex(f, fn, batch=0, A=None, B=None, C=None) == OK
    assert call_ex(f, fn, M=0, A=None, B=None, C=None) == OK
    assert call_ex(f, fn, N=0, A=None, B=None, C=None) == OK


@pytest.mark.parametrize("fn", ["gemm_bf16_ex", "gemm_f16_ex"])
def test_extended_tensor_core_layout_rule(gemm_mod, fn):
    """Matrix strides of A and B in whole 16-byte units when batch > 1, on top
    of the plain entry points' base and row-stride rule."""
    f = getattr(gemm_mod.lib, fn)
    assert call_ex(f, fn, sA=68) == LAYOUT
    assert call_ex(f, fn, sB=12) == LAYOUT
    assert call_ex(f, fn, A=FAKE + 2) == LAYOUT
    assert call_ex(f, fn, opA=T_, lda=12, M=12, ldc=12, N=8, sC=256) == LAYOUT


def test_tf32_needs_aligned_elements(gemm_mod):
    f = gemm_mod.lib.gemm_tf32
    assert f(8, 8, 8, 1.0, FAKE + 2, 8, FAKE, 8, 0.0, FAKE, 8, None) == LAYOUT
    assert f(8, 8, 8, 1.0, FAKE, 8, FAKE + 1, 8, 0.0, FAKE, 8, None) == LAYOUT


def test_peak_microbenchmarks_check_arguments_on_host(gemm_mod):
    """Iteration counts outside 1 .. 2^24 and a missing sink are rejected before
    any device work."""
    lib = gemm_mod.lib
    assert lib.gemm_peak_ffma(0, FAKE, None, None) == INVALID
    assert lib.gemm_peak_ffma((1 << 24) + 1, FAKE, None, None) == INVALID
    assert lib.gemm_peak_ffma(16, None, None, None) == INVALID
    assert lib.gemm_peak_tc_f16(0, None, None) == INVALID
    assert lib.gemm_peak_tc_f16(-5, None, None) == INVALID
    assert lib.gemm_peak_tc_f16((1 << 20) + 1, None, None) == INVALID

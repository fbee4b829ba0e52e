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


@pytest.mark.parametrize("fn", ["gemm_f32", "gemm_bf16", "gemm_f16", "gemm_s8"])
def test_invalid_arguments_rejected_on_host(gemm_mod, fn):
    f = getattr(gemm_mod.lib, fn)
    a = 1 if fn == "gemm_s8" else 1.0
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


@pytest.mark.parametrize("fn", ["gemm_f32", "gemm_bf16", "gemm_f16", "gemm_s8"])
def test_empty_output_is_a_no_op(gemm_mod, fn):
    f = getattr(gemm_mod.lib, fn)
    a = 1 if fn == "gemm_s8" else 1.0
    assert f(0, 8, 8, a, None, 8, None, 8, a, None, 8, None) == OK
    assert f(8, 0, 8, a, None, 8, None, 8, a, None, 0, None) == OK


@pytest.mark.parametrize("fn", ["gemm_bf16", "gemm_f16"])
def test_tensor_core_layout_rule(gemm_mod, fn):
    """16-byte aligned A and B bases and lda, ldb multiples of 8, else
    GEMM_ERR_UNSUPPORTED_LAYOUT (checked before any device work)."""
    f = getattr(gemm_mod.lib, fn)
    assert f(8, 8, 8, 1.0, FAKE + 2, 8, FAKE, 8, 0.0, FAKE, 8, None) == LAYOUT
    assert f(8, 8, 8, 1.0, FAKE, 8, FAKE + 8, 8, 0.0, FAKE, 8, None) == LAYOUT
    assert f(8, 8, 12, 1.0, FAKE, 12, FAKE, 8, 0.0, FAKE, 8, None) == LAYOUT
    assert f(8, 12, 8, 1.0, FAKE, 8, FAKE, 12, 0.0, FAKE, 12, None) == LAYOUT

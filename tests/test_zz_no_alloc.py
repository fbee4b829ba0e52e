"""gemm_s8_noalloc: the int8 GEMM for callers that cannot allocate device memory.

Such callers exist because the library's own gemm_s8 takes scratch for its
fp16-widened operands from a stream-ordered pool: a process whose device memory
is reserved in full by another allocator, a latency-critical loop that must not
enter the driver's allocation path, or a deployment that forbids allocation
after start-up cannot allow that. gemm_s8_noalloc works on a fixed scratch
array inside the library instead.

Through the C ABI, this checks that two calls in a row return exactly what
gemm_s8 returns (int8 results are compared bit for bit, as everywhere in these
tests), that a call after the first one leaves the device's free memory
unchanged, and that a problem too large for the fixed scratch is refused before
anything is launched. This file is collected last on purpose, and it also
passes when run on its own in a fresh process.
"""
import pytest
import torch

from dense_gemm_row_gb300 import workloads as w

pytestmark = pytest.mark.gpu

TOO_LARGE = 6


def call(lib, name, p, C, stream):
    M, K = p.A.shape
    N = p.B.shape[1]
    return getattr(lib, name)(M, N, K, int(p.alpha), p.A.data_ptr(), p.A.stride(0),
                              p.B.data_ptr(), p.B.stride(0), int(p.beta), C.data_ptr(),
                              C.stride(0), stream)


def test_noalloc_matches_gemm_s8_on_two_calls_in_a_row(gemm_mod):
    lib = gemm_mod.lib
    gemm_mod.check_device_error()
    stream = torch.cuda.current_stream().cuda_stream
    problems = [
        w.problem(1000, 1500, 2100, torch.int8, "int8", 301, alpha=3, beta=-2, c_dist="int"),
        w.problem(333, 257, 4096, torch.int8, "int8", 302, alpha=-1, beta=5, c_dist="int"),
    ]
    for i, p in enumerate(problems):
        p = p.to("cuda")
        c_ref = p.C0.clone()
        c_new = p.C0.clone()
        assert call(lib, "gemm_s8", p, c_ref, stream) == 0
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert call(lib, "gemm_s8_noalloc", p, c_new, stream) == 0
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert torch.equal(c_new, c_ref), f"call {i + 1}: gemm_s8_noalloc differs from gemm_s8"
        if i > 0:
            # The first call may load the library's module (and with it the
            # scratch array); no later call may take device memory.
            assert free_after == free_before
    assert gemm_mod.check_device_error() == 0


def test_noalloc_refuses_problems_beyond_its_scratch(gemm_mod):
    fake = 1 << 20  # never dereferenced: the size check comes first
    lib = gemm_mod.lib
    assert lib.gemm_s8_noalloc(8192, 8192, 8192, 1, fake, 8192, fake, 8192, 0, fake, 8192,
                               None) == TOO_LARGE
    assert lib.gemm_status_string(TOO_LARGE).decode() == "GEMM_ERR_TOO_LARGE"
    # 4096^3 is the largest square problem that fits.
    assert lib.gemm_s8_noalloc(4097, 4097, 4097, 1, fake, 4097, fake, 4097, 0, fake, 4097,
                               None) == TOO_LARGE

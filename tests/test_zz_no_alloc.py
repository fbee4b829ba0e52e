"""gemm_s8_noalloc: the int8 GEMM for callers that cannot allocate device memory.

Such callers exist because the library's own gemm_s8 takes scratch for its
fp16-widened operands from a stream-ordered pool: a process whose device memory
is reserved in full by another allocator, a latency-critical loop that must not
enter the driver's allocation path, or a deployment that forbids allocation
after start-up cannot allow that. gemm_s8_noalloc works on a fixed scratch
array inside the library instead.

Through the C ABI, this checks, on every problem, that two calls in a row each
return the oracle's exact result (int8 results are compared bit for bit, as
everywhere in these tests) and the same bits as gemm_s8, that neither call
takes anything from the library's memory pool (its high-water mark stays at
zero while only gemm_s8_noalloc runs) and that the second call leaves the
device's free memory unchanged. gemm_s8_noalloc runs before gemm_s8 on each
problem, so that gemm_s8's pool blocks are not yet in use when the mark is
read. The problems reach every route the entry point takes: plain tensor-core
tiles, the split-k tail of a partial last wave (4096^3, the largest square
problem the fixed scratch admits; its tail flags live in the same array) and
the short, wide kernel for M <= 32. A problem too large for the fixed scratch
must be refused before anything is launched. This file is collected last on
purpose, and it also passes when run on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from dense_gemm_row_gb300 import workloads as w

pytestmark = pytest.mark.gpu

TOO_LARGE = 6

PROBLEMS = [
    # (M, N, K, alpha, beta, seed)
    (1000, 1500, 2100, 3, -2, 301),   # tensor-core tiles, ragged edges
    (333, 257, 4096, -1, 5, 302),     # ragged, four 1024-k chunks
    (16, 4096, 4096, 2, -1, 303),     # short and wide: transposed-role kernel
    (4096, 4096, 4096, 1, 0, 304),    # largest square size: split-k tail
]


def call(lib, name, p, C, stream):
    M, K = p.A.shape
    N = p.B.shape[1]
    return getattr(lib, name)(M, N, K, int(p.alpha), p.A.data_ptr(), p.A.stride(0),
                              p.B.data_ptr(), p.B.stride(0), int(p.beta), C.data_ptr(),
                              C.stride(0), stream)


@pytest.mark.parametrize("shape", PROBLEMS, ids=lambda s: "x".join(map(str, s[:3])))
def test_noalloc_matches_oracle_on_two_calls_in_a_row(gemm_mod, oracle_mod, shape):
    M, N, K, alpha, beta, seed = shape
    lib = gemm_mod.lib
    gemm_mod.check_device_error()
    stream = torch.cuda.current_stream().cuda_stream
    p = w.problem(M, N, K, torch.int8, "int8", seed, alpha=alpha, beta=beta, c_dist="int")
    ref = oracle_mod.gemm_s8(p.A, p.B, alpha, beta, p.C0)
    d = p.to("cuda")
    torch.cuda.synchronize()
    gemm_mod.pool_usage(reset_high=True)
    results = []
    for i in range(2):
        c = d.C0.clone()
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert call(lib, "gemm_s8_noalloc", d, c, stream) == 0
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        np.testing.assert_array_equal(c.cpu().numpy(), ref,
                                      err_msg=f"call {i + 1}: gemm_s8_noalloc != oracle")
        results.append(c)
        if i > 0:
            # The first call on a device may load the library's module (and
            # with it the scratch array); no later call may take memory.
            assert free_after == free_before, "a repeated call took device memory"
    used_high, _ = gemm_mod.pool_usage()
    assert used_high == 0, f"gemm_s8_noalloc drew {used_high} bytes from the library's pool"
    c_pool = d.C0.clone()
    assert call(lib, "gemm_s8", d, c_pool, stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(results[1], c_pool), "gemm_s8_noalloc differs from gemm_s8"
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

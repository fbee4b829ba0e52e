"""The bounded-wait failure path on the GPU, exercised without any fault: a
wait that nothing satisfies gives up after its limit, the device error word
reports GEMM_ERR_TIMEOUT, and the context keeps working."""
import pytest
import torch

from dense_gemm_row_gb300 import workloads as w

pytestmark = pytest.mark.gpu

TIMEOUT = 5
WAIT_TEST_CODE = 7


def test_bounded_wait_reports_timeout_and_context_survives(gemm_mod, oracle_mod):
    lib = gemm_mod.lib
    gemm_mod.check_device_error()
    assert lib.gemm_selftest_wait_timeout(0, None) == 1          # limit out of range
    assert lib.gemm_selftest_wait_timeout(2_000_000, None) == 1
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.gemm_selftest_wait_timeout(20_000, stream) == 0    # 20 ms
    torch.cuda.synchronize()
    with pytest.raises(gemm_mod.GemmError) as e:
        gemm_mod.check_device_error()
    assert e.value.status == TIMEOUT
    # The word was cleared by the read, and the context still computes.
    assert gemm_mod.check_device_error() == 0
    p = w.problem(256, 512, 128, torch.bfloat16, "normal", 11)
    C = torch.zeros(256, 512, device="cuda")
    gemm_mod.gemm(p.A.cuda(), p.B.cuda(), C)
    torch.cuda.synchronize()
    ref = oracle_mod.gemm(p.A, p.B)
    import numpy as np
    assert np.linalg.norm(C.cpu().numpy() - ref) / np.linalg.norm(ref) <= 1e-5
    assert gemm_mod.check_device_error() == 0


def test_error_word_records_the_wait_code(gemm_mod):
    import ctypes
    lib = gemm_mod.lib
    gemm_mod.check_device_error()
    assert lib.gemm_selftest_wait_timeout(5_000, None) == 0
    torch.cuda.synchronize()
    word = ctypes.c_uint32(0)
    assert lib.gemm_check_device_error(ctypes.byref(word)) == TIMEOUT
    assert word.value & 1
    assert (word.value >> 8) & 0xFF == WAIT_TEST_CODE

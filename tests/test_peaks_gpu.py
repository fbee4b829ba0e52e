"""GPU checks of the peak-rate microbenchmarks that cross-check the roofline
denominators: both run to completion without a device error and report a rate
that is plausible for one GB300-class GPU (well above what either pipe could
give if the kernel were not doing the work, and not above the dense rate at
the maximum clock)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def timed(fn):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    e0.record(s)
    flops = fn()
    e1.record(s)
    e1.synchronize()
    return flops / (e0.elapsed_time(e1) / 1e3) / 1e12


def test_ffma_peak(gemm_mod):
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.zeros(1, device="cuda")
    gemm_mod.peak_ffma(64, sink)
    tflops = timed(lambda: gemm_mod.peak_ffma(8192, sink))
    assert gemm_mod.check_device_error() == 0
    ceiling = sm * 128 * 2 * 2.2e9 / 1e12  # 128 lanes x FMA at most 2.2 GHz
    assert 0.25 * ceiling < tflops <= ceiling, tflops
    assert sink.item() == 0.0  # the sentinel is never hit


def test_tensor_core_peak(gemm_mod):
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    gemm_mod.peak_tc_f16(64)
    tflops = timed(lambda: gemm_mod.peak_tc_f16(4096))
    assert gemm_mod.check_device_error() == 0
    ceiling = sm * 8192 * 2.2e9 / 1e12  # dense kind::f16 rate at most 2.2 GHz
    assert 0.25 * ceiling < tflops <= ceiling, tflops

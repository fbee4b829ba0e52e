"""GPU parity of the further type-table entry points against the CPU oracle:
gemm_u8 (bit-exact), gemm_f16_f16 / gemm_bf16_bf16 (16-bit C), gemm_tf32 and
gemm_f64. Each bar is derived from the arithmetic the entry point promises:

* u8: exact integers, so bit-exact.
* 16-bit C: the GPU accumulates in fp32 and rounds once to 16 bits; the oracle
  rounds the exact result once. Every element must lie within one rounding of
  the output format (unit roundoff u = 2^-11 for fp16, 2^-8 for bf16) plus the
  worst-case fp32 accumulation error (K + 2) * 2^-24 * (|alpha| (|A||B|)_ij +
  |beta| |C0_ij|) of the exact result. At least 90 % of the elements must
  equal the oracle's rounded value bit for bit: the fp32 accumulation moves a
  result across a rounding boundary only where the exact value lies within
  the accumulation error of one (measured: 2 % of the elements at K = 4100,
  fp16, U[-1, 1) data), while truncating instead of rounding would disagree on
  about half. Where every partial sum is an exact fp32 integer the 16-bit
  result must equal the oracle's everywhere, which pins ties-to-even.
* tf32: inputs reduced to tf32, products exact in fp32, fp32 accumulation:
  relative Frobenius <= 1e-5 against the oracle's tf32 reading, and bit-exact
  where every partial sum is an exact fp32 integer.
* f64: both sides round in double; elementwise |got - ref| <= (2K + 4) *
  2^-53 * (|alpha| (|A||B|)_ij + |beta| |C0_ij|).
"""
import numpy as np
import pytest
import torch

from dense_gemm_row_gb300 import workloads as w
from tests.gpu_util import Banded, dev_copy, rel_frobenius

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1, 1), (7, 9, 13), (33, 65, 17), (129, 257, 255), (300, 520, 200),
          (257, 130, 1000), (64, 256, 4100)]


@pytest.fixture(autouse=True)
def clean_error_word(gemm_mod):
    gemm_mod.check_device_error()
    yield
    torch.cuda.synchronize()
    assert gemm_mod.check_device_error() == 0


def u8_matrix(rows, cols, seed, hi=256):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, hi, (rows, cols), generator=g, dtype=torch.int32).to(torch.uint8)


# ----------------------------------------------------------------------- u8

@pytest.mark.parametrize("aligned", [True, False], ids=["c_aligned", "c_unaligned"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_u8_bit_exact(gemm_mod, oracle_mod, shape, aligned):
    M, N, K = shape
    A = u8_matrix(M, K, 1 + M)
    B = u8_matrix(K, N, 2 + N)
    C0 = w.matrix(M, N, torch.float32, "int8", 3 + K).to(torch.int32)
    out = Banded(C0, None if aligned else N + 1, aligned)
    gemm_mod.gemm(dev_copy(A, 0), dev_copy(B, 0), out.C, 7, -3)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.result().numpy(), oracle_mod.gemm_u8(A, B, 7, -3, C0))
    out.check_canaries()


def test_u8_extremes_exact_chunks_and_wrap(gemm_mod, oracle_mod):
    """All-255 operands: every 256-k chunk sums to 256 * 65025 < 2^24 (exact in
    the fp32 accumulator); K = 40000 takes the int32 result past 2^31 (wraps)."""
    for K in (4100, 40000):
        A = torch.full((40, K), 255, dtype=torch.uint8)
        B = torch.full((K, 72), 255, dtype=torch.uint8)
        C = torch.zeros(40, 72, dtype=torch.int32, device="cuda")
        gemm_mod.gemm(A.cuda(), B.cuda(), C)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(C.cpu().numpy(), oracle_mod.gemm_u8(A, B))


def test_u8_large(gemm_mod, oracle_mod):
    M = N = K = 2048
    A, B = u8_matrix(M, K, 11), u8_matrix(K, N, 12)
    C = torch.empty(M, N, dtype=torch.int32, device="cuda")
    gemm_mod.gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.cpu().numpy(), oracle_mod.gemm_u8(A, B))


# ------------------------------------------------------------------ 16-bit C

U16 = {torch.float16: 2.0**-11, torch.bfloat16: 2.0**-8}


def check_out16(got, A, B, alpha, beta, C0, oracle_mod):
    dtype = A.dtype
    K = A.shape[1]
    got = got.contiguous()
    exp16 = oracle_mod.gemm_out16(A, B, alpha, beta, C0 if beta != 0 else None)
    ref = oracle_mod.gemm(A, B, alpha, beta, C0.double() if beta != 0 else None)
    mag = abs(alpha) * oracle_mod.gemm(A.abs(), B.abs())
    if beta != 0:
        mag = mag + abs(beta) * np.abs(C0.double().numpy())
    g = got.double().numpy()
    bound = U16[dtype] * np.abs(ref) + (K + 2) * 2.0**-24 * mag * (1 + U16[dtype]) + 1e-30
    bad = np.abs(g - ref) > bound
    assert not bad.any(), f"{bad.sum()} elements outside one rounding of the exact result"
    same = (got.view(torch.int16) == exp16.view(torch.int16)).double().mean().item()
    assert same >= 0.90, f"only {same:.4f} of the elements equal the oracle's rounded value"


@pytest.mark.parametrize("aligned", [True, False], ids=["c_aligned", "c_unaligned"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=str)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_out16(gemm_mod, oracle_mod, shape, dtype, aligned):
    M, N, K = shape
    ld = lambda c: (c + 7) // 8 * 8  # noqa: E731  tensor-core row-stride rule
    A = w.matrix(M, K, dtype, "uniform_pm1", 20 + M, ld=ld(K))
    B = w.matrix(K, N, dtype, "uniform_pm1", 21 + N, ld=ld(N))
    C0 = w.matrix(M, N, dtype, "uniform_pm1", 22 + K)
    # 16-bit canaries: the Banded helper holds 32-bit values, so band a 16-bit
    # view by hand: C inside a buffer of NaN with odd or aligned row stride.
    ldc = ld(N) if aligned else N + 1
    guard = 128 if aligned else 129
    flat = torch.full((guard + M * ldc + 131,), float("nan"), dtype=dtype, device="cuda")
    C = flat[guard:guard + M * ldc].view(M, ldc)[:, :N]
    C.copy_(C0)
    gemm_mod.gemm(dev_copy(A, float("nan")), dev_copy(B, float("nan")), C, 1.25, -0.5)
    torch.cuda.synchronize()
    check_out16(C.cpu(), A, B, 1.25, -0.5, C0, oracle_mod)
    mask = torch.ones(flat.shape, dtype=torch.bool)
    mask[guard:guard + M * ldc].view(M, ldc)[:, :N] = False
    assert torch.isnan(flat.cpu()[mask]).all(), "a kernel wrote outside C"


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=str)
def test_out16_integer_results_round_to_nearest_even(gemm_mod, oracle_mod, dtype):
    """Integer inputs of magnitude <= 40 with K = 96: every sum is an integer
    below 2^24 (exact in fp32), many above 2^11 (fp16) or 2^8 (bf16), so the
    16-bit result is the exact integer rounded to nearest even, element for
    element."""
    g = torch.Generator().manual_seed(33)
    M, N, K = 200, 264, 96
    A = torch.randint(-40, 41, (M, K), generator=g).to(dtype)
    B = torch.randint(-40, 41, (K, N), generator=g).to(dtype)
    C = torch.zeros(M, N, dtype=dtype, device="cuda")
    gemm_mod.gemm(A.cuda(), B.cuda(), C, 1.0, 0.0)
    torch.cuda.synchronize()
    exp = oracle_mod.gemm_out16(A, B, 1.0, 0.0)
    assert torch.equal(C.cpu().view(torch.int16), exp.view(torch.int16))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=str)
def test_out16_beta_zero_and_k_zero(gemm_mod, oracle_mod, dtype):
    M, N, K = 130, 264, 72
    A = w.matrix(M, K, dtype, "normal", 30)
    B = w.matrix(K, N, dtype, "normal", 31)
    C = torch.full((M, N), float("nan"), dtype=dtype, device="cuda")
    gemm_mod.gemm(A.cuda(), B.cuda(), C, 0.5, 0.0)
    torch.cuda.synchronize()
    check_out16(C.cpu(), A, B, 0.5, 0.0, torch.zeros(M, N, dtype=dtype), oracle_mod)
    C0 = w.matrix(M, N, dtype, "normal", 32)
    C.copy_(C0)
    Z = torch.zeros(M, 0, dtype=dtype, device="cuda")
    gemm_mod.gemm(Z, torch.zeros(0, N, dtype=dtype, device="cuda"), C, 1.0, -3.0)
    torch.cuda.synchronize()
    exp = oracle_mod.gemm_out16(A[:, :0].contiguous(), B[:0].contiguous(), 1.0, -3.0, C0)
    assert torch.equal(C.cpu().view(torch.int16), exp.view(torch.int16))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=str)
def test_out16_large(gemm_mod, oracle_mod, dtype):
    M, N, K = 2048, 2048, 4096
    A = w.matrix(M, K, dtype, "normal", 40)
    B = w.matrix(K, N, dtype, "normal", 41)
    C = torch.empty(M, N, dtype=dtype, device="cuda")
    gemm_mod.gemm(A.cuda(), B.cuda(), C, 1.0, 0.0)
    torch.cuda.synchronize()
    check_out16(C.cpu(), A, B, 1.0, 0.0, torch.zeros(M, N, dtype=dtype), oracle_mod)


# ----------------------------------------------------------------------- tf32

def test_tf32_input_reduction_is_truncation(gemm_mod, oracle_mod):
    """1 + 2^-10 + 2^-11 lies halfway between two tf32 values; truncation gives
    1 + 2^-10, round-to-nearest-even 1 + 2^-9. With B = 1 and K = 1 the
    product is the reduced value itself, exactly."""
    v = 1 + 2**-10 + 2**-11
    A = torch.tensor([[v, -v, 1 + 2**-12, 3.0]], dtype=torch.float32).t().contiguous()  # 4 x 1
    B = torch.ones(1, 8, dtype=torch.float32)
    C = torch.zeros(4, 8, dtype=torch.float32, device="cuda")
    gemm_mod.gemm(A.cuda(), B.cuda(), C, tf32=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.cpu().double().numpy(), oracle_mod.gemm(A, B, tf32=True))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tf32_parity(gemm_mod, oracle_mod, shape):
    M, N, K = shape
    A = w.matrix(M, K, torch.float32, "uniform_pm1", 50 + M, ld=K + 3)
    B = w.matrix(K, N, torch.float32, "uniform_pm1", 51 + N, ld=N + 1)
    C0 = w.matrix(M, N, torch.float32, "uniform_pm1", 52 + K)
    out = Banded(C0, N + 3, aligned=False)
    gemm_mod.gemm(dev_copy(A, float("nan")), dev_copy(B, float("nan")), out.C, 1.5, -0.5,
                  tf32=True)
    torch.cuda.synchronize()
    ref = oracle_mod.gemm(A, B, 1.5, -0.5, C0, tf32=True)
    err = rel_frobenius(out.result().numpy(), ref)
    assert err <= 1e-5, f"relative Frobenius error {err:.3e}"
    out.check_canaries()


def test_tf32_integer_inputs_bit_exact(gemm_mod, oracle_mod):
    """Integers below 2^11 are exact in tf32; with K = 256 and |values| < 64
    every partial sum is an integer below 2^24, so the result is exact."""
    g = torch.Generator().manual_seed(60)
    M, N, K = 300, 520, 256
    A = torch.randint(-63, 64, (M, K), generator=g).float()
    B = torch.randint(-63, 64, (K, N), generator=g).float()
    C = torch.zeros(M, N, device="cuda")
    gemm_mod.gemm(A.cuda(), B.cuda(), C, tf32=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.cpu().double().numpy(), oracle_mod.gemm(A, B, tf32=True))


def test_tf32_large(gemm_mod, oracle_mod):
    M, N, K = 2048, 2048, 4096
    A = w.matrix(M, K, torch.float32, "normal", 61)
    B = w.matrix(K, N, torch.float32, "normal", 62)
    C = torch.empty(M, N, device="cuda")
    gemm_mod.gemm(A.cuda(), B.cuda(), C, tf32=True)
    torch.cuda.synchronize()
    ref = oracle_mod.gemm(A, B, tf32=True)
    assert rel_frobenius(C.cpu().numpy(), ref) <= 1e-5


# ----------------------------------------------------------------------- f64

@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_f64_parity(gemm_mod, oracle_mod, shape):
    M, N, K = shape
    A = w.matrix(M, K, torch.float64, "normal", 70 + M, ld=K + 1)
    B = w.matrix(K, N, torch.float64, "normal", 71 + N, ld=N + 2)
    C0 = w.matrix(M, N, torch.float64, "normal", 72 + K)
    C = dev_copy(C0, float("nan"))
    gemm_mod.gemm(dev_copy(A, float("nan")), dev_copy(B, float("nan")), C, 0.75, -1.5)
    torch.cuda.synchronize()
    ref = oracle_mod.gemm(A, B, 0.75, -1.5, C0)
    mag = 0.75 * (np.abs(A.numpy()) @ np.abs(B.numpy())) + 1.5 * np.abs(C0.numpy())
    bound = (2 * K + 4) * 2.0**-53 * mag
    assert (np.abs(C.cpu().numpy() - ref) <= bound).all()

"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

None of these re-types the oracle's own formula. They check it against values
printed on the pages, hand-computed tiny products, exact rational brute force,
closed forms (identity, zero), invariants (alpha/beta linearity, additivity
over a split of K, independence of rows), library routines on special cases
(numpy int64 and float64 matmul, numpy/torch 16-bit float decoding) and the
int32 wrap-around of an int64 result.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def t32(x):
    return torch.tensor(x, dtype=torch.float32)


# ---------------------------------------------------------------- page values

def test_dlog_worked_example(oracle_mod):
    """dlog page, V1 2D Thread: the inner product 1*2 + 1*3 = 5 (row 0 of A with
    column 0 of B, printed under the label C[0][1]; see the fixture's reading)
    and the k = 0 outer-product term [[2,2],[6,6]]."""
    g = json.load(open(os.path.join(GOLDEN, "dlog_outer_inner_2x2.json")))
    A, B = t32(g["A"]), t32(g["B"])
    C = oracle_mod.gemm(A, B)
    assert C[0, 0] == g["printed"]["inner_product_value"]
    assert C[0, 1] == 1 * 2 + 1 * 4  # what the label C[0][1] would hold
    term0 = oracle_mod.gemm(A[:, 0:1].contiguous(), B[0:1, :].contiguous())
    np.testing.assert_array_equal(term0, np.array(g["printed"]["outer_product_term_k0"]))
    # Outer-product form: the product is the sum of its K rank-1 terms.
    term1 = oracle_mod.gemm(A[:, 1:2].contiguous(), B[1:2, :].contiguous())
    np.testing.assert_array_equal(C, term0 + term1)


def test_hand_computed_rectangular(oracle_mod):
    """2x3 times 3x2, written out by hand: rows of A dotted with columns of B."""
    A = t32([[1, 2, 3], [4, 5, 6]])
    B = t32([[7, 8], [9, 10], [11, 12]])
    # 1*7+2*9+3*11 = 58, 1*8+2*10+3*12 = 64, 4*7+5*9+6*11 = 139, 4*8+5*10+6*12 = 154
    np.testing.assert_array_equal(oracle_mod.gemm(A, B), [[58, 64], [139, 154]])
    C0 = t32([[1, -1], [2, 0.5]])
    # alpha=2, beta=-1: 2*58-1 = 115, 2*64+1 = 129, 2*139-2 = 276, 2*154-0.5 = 307.5
    np.testing.assert_array_equal(oracle_mod.gemm(A, B, 2.0, -1.0, C0),
                                  [[115, 129], [276, 307.5]])
    # B times A is a different (3x3) product; its corner is 7*1+8*4 = 39.
    assert oracle_mod.gemm(B, A)[0, 0] == 39


@pytest.mark.parametrize("seed", range(12))
def test_exact_rational_brute_force(oracle_mod, seed):
    """Tiny shapes against exact rational arithmetic. Values are small dyadic
    rationals, so every product and partial sum is exact in double and the
    oracle must agree exactly."""
    rng = np.random.default_rng(seed)
    M, N, K = (int(x) for x in rng.integers(1, 6, size=3))
    A = rng.integers(-16, 17, size=(M, K)) / 8.0
    B = rng.integers(-16, 17, size=(K, N)) / 4.0
    C0 = rng.integers(-16, 17, size=(M, N)) / 2.0
    alpha, beta = float(rng.integers(-4, 5)) / 2.0, float(rng.integers(-4, 5)) / 4.0
    got = oracle_mod.gemm(t32(A), t32(B), alpha, beta, t32(C0))
    for i in range(M):
        for j in range(N):
            acc = sum((Fraction(A[i, k]) * Fraction(B[k, j]) for k in range(K)), Fraction(0))
            want = Fraction(alpha) * acc + (Fraction(beta) * Fraction(C0[i, j]) if beta else 0)
            assert Fraction(got[i, j]) == want, (i, j)


# ---------------------------------------------------------------- closed forms

def test_identity_closed_form(oracle_mod):
    """A = I: the product is B itself, so C = alpha*B + beta*C0."""
    from dense_gemm_row_gb300 import workloads as w
    K, N = 37, 23
    B = w.matrix(K, N, torch.float32, "uniform_pm1", 11)
    C0 = w.matrix(K, N, torch.float32, "uniform_pm1", 12)
    I = torch.eye(K, dtype=torch.float32)
    np.testing.assert_array_equal(oracle_mod.gemm(I, B), B.double().numpy())
    got = oracle_mod.gemm(I, B, 0.5, 2.0, C0)
    np.testing.assert_array_equal(got, 0.5 * B.double().numpy() + 2.0 * C0.double().numpy())


def test_zero_closed_form(oracle_mod):
    from dense_gemm_row_gb300 import workloads as w
    A = torch.zeros(9, 14)
    B = w.matrix(14, 5, torch.float32, "normal", 3)
    C0 = w.matrix(9, 5, torch.float32, "normal", 4)
    np.testing.assert_array_equal(oracle_mod.gemm(A, B, 3.0, -0.25, C0),
                                  -0.25 * C0.double().numpy())
    np.testing.assert_array_equal(oracle_mod.gemm(A, B), np.zeros((9, 5)))


def test_k_zero_and_empty(oracle_mod):
    C0 = t32([[1.5, -2.0, 3.0]])
    A = torch.zeros(1, 0)
    B = torch.zeros(0, 3)
    np.testing.assert_array_equal(oracle_mod.gemm(A, B, 2.0, 2.0, C0), [[3.0, -4.0, 6.0]])
    np.testing.assert_array_equal(oracle_mod.gemm(A, B, 2.0, 0.0, C0), [[0.0, 0.0, 0.0]])
    assert oracle_mod.gemm(torch.zeros(0, 4), torch.zeros(4, 3)).shape == (0, 3)
    assert oracle_mod.gemm(torch.zeros(2, 4), torch.zeros(4, 0)).shape == (2, 0)


# ------------------------------------------------------------------ invariants

def test_alpha_beta_linearity(oracle_mod):
    """oracle(alpha, beta) = alpha*oracle(1, 0) + beta*C0, exact on small integers."""
    from dense_gemm_row_gb300 import workloads as w
    A = w.matrix(31, 17, torch.float32, "int0_99", 5)
    B = w.matrix(17, 29, torch.float32, "int0_99", 6)
    C0 = w.matrix(31, 29, torch.float32, "int0_99", 7)
    base = oracle_mod.gemm(A, B)
    for alpha, beta in [(1.5, -0.5), (-2.0, 0.25), (0.0, 1.0), (1.0, 1.0)]:
        got = oracle_mod.gemm(A, B, alpha, beta, C0)
        np.testing.assert_array_equal(got, alpha * base + beta * C0.double().numpy())


def test_k_split_additivity(oracle_mod):
    """Splitting K in two: A*B = A[:, :k]*B[:k] + A[:, k:]*B[k:], exact on integers."""
    from dense_gemm_row_gb300 import workloads as w
    A = w.matrix(20, 50, torch.float32, "int0_99", 8)
    B = w.matrix(50, 13, torch.float32, "int0_99", 9)
    full = oracle_mod.gemm(A, B)
    left = oracle_mod.gemm(A[:, :21].contiguous(), B[:21].contiguous())
    right = oracle_mod.gemm(A[:, 21:].contiguous(), B[21:].contiguous())
    np.testing.assert_array_equal(full, left + right)


def test_rows_are_independent(oracle_mod):
    from dense_gemm_row_gb300 import workloads as w
    p = w.problem(40, 33, 27, torch.float32, "uniform_pm1", 13, alpha=1.25, beta=-0.75,
                  c_dist="uniform_pm1")
    full = oracle_mod.gemm(p.A, p.B, p.alpha, p.beta, p.C0)
    rows = [39, 0, 17, 17, 5]
    np.testing.assert_array_equal(oracle_mod.gemm_rows(p.A, p.B, rows, p.alpha, p.beta, p.C0),
                                  full[rows])


def test_leading_dimension_padding_never_read(oracle_mod):
    """NaN-poisoned row padding in A, B and C must not reach the result."""
    from dense_gemm_row_gb300 import workloads as w
    p = w.problem(19, 21, 23, torch.float32, "uniform_pm1", 14, alpha=2.0, beta=0.5,
                  c_dist="uniform_pm1")
    q = w.problem(19, 21, 23, torch.float32, "uniform_pm1", 14, alpha=2.0, beta=0.5,
                  c_dist="uniform_pm1", lda=29, ldb=32, ldc=40)
    assert q.A.stride(0) == 29 and q.B.stride(0) == 32
    got = oracle_mod.gemm(q.A, q.B, q.alpha, q.beta, q.C0)
    assert np.isfinite(got).all()
    np.testing.assert_array_equal(got, oracle_mod.gemm(p.A, p.B, p.alpha, p.beta, p.C0))


def test_beta_zero_does_not_read_c(oracle_mod):
    from dense_gemm_row_gb300 import workloads as w
    A = w.matrix(8, 8, torch.float32, "normal", 15)
    B = w.matrix(8, 8, torch.float32, "normal", 16)
    nan_c = torch.full((8, 8), float("nan"))
    got = oracle_mod.gemm(A, B, 1.0, 0.0, nan_c)
    np.testing.assert_array_equal(got, oracle_mod.gemm(A, B))
    assert np.isnan(oracle_mod.gemm(A, B, 1.0, 1.0, nan_c)).all()


# ----------------------------------------------------- special cases vs libraries

def test_integer_valued_fp32_matches_int64(oracle_mod):
    """Integers 0..99 (the tiled-multiply page's rand()%100 data) at K = 128:
    every sum is an integer below 2^24, so the double result equals the exact
    int64 product computed by numpy."""
    from dense_gemm_row_gb300 import workloads as w
    p = w.config("f32_int128")
    got = oracle_mod.gemm(p.A, p.B)
    exact = p.A.numpy().astype(np.int64) @ p.B.numpy().astype(np.int64)
    assert exact.max() < 2 ** 24
    np.testing.assert_array_equal(got, exact.astype(np.float64))


def test_tiled_page_odd_shape_exact(oracle_mod):
    """The tiled-multiply page's harness shape: A 47 x 804 times B 804 x 53 with
    integers 0..99. 804 * 99^2 < 2^24, so the result is exact."""
    from dense_gemm_row_gb300 import workloads as w
    A = w.matrix(47, 804, torch.float32, "int0_99", 21)
    B = w.matrix(804, 53, torch.float32, "int0_99", 22)
    exact = A.numpy().astype(np.int64) @ B.numpy().astype(np.int64)
    np.testing.assert_array_equal(oracle_mod.gemm(A, B), exact.astype(np.float64))


def test_float64_matches_numpy_matmul(oracle_mod):
    """Random normal data: double oracle vs numpy's float64 matmul (another
    summation order) to within a few ulps of the row norms."""
    from dense_gemm_row_gb300 import workloads as w
    A = w.matrix(65, 130, torch.float32, "normal", 23)
    B = w.matrix(130, 71, torch.float32, "normal", 24)
    got = oracle_mod.gemm(A, B)
    ref = A.double().numpy() @ B.double().numpy()
    bound = 1e-13 * (np.abs(A.double().numpy()) @ np.abs(B.double().numpy()))
    assert (np.abs(got - ref) <= bound).all()


def test_decode_bf16_all_patterns(oracle_mod):
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.decode_bf16(b) for b in range(65536)])
    np.testing.assert_array_equal(got, ref)  # NaNs compare equal positionally


def test_decode_f16_all_patterns(oracle_mod):
    ref = np.arange(0, 65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.decode_f16(b) for b in range(65536)])
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_half_inputs_equal_double_on_decoded_values(oracle_mod, dtype):
    """The 16-bit entry points see exactly the rounded values: running them
    equals running the double entry point on torch's exact widening."""
    from dense_gemm_row_gb300 import workloads as w
    p = w.problem(33, 45, 70, dtype, "normal", 25, alpha=0.75, beta=-1.5, c_dist="normal")
    got = oracle_mod.gemm(p.A, p.B, p.alpha, p.beta, p.C0)
    ref = oracle_mod.gemm(p.A.double(), p.B.double(), p.alpha, p.beta, p.C0)
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------------------ int8

def test_int8_extremes(oracle_mod):
    K = 300
    A = torch.full((3, K), -128, dtype=torch.int8)
    B = torch.full((K, 4), -128, dtype=torch.int8)
    assert (oracle_mod.gemm_s8(A, B) == K * 16384).all()
    B2 = torch.full((K, 4), 127, dtype=torch.int8)
    assert (oracle_mod.gemm_s8(A, B2) == -K * 16256).all()


def test_int8_matches_numpy_int64(oracle_mod):
    from dense_gemm_row_gb300 import workloads as w
    p = w.problem(70, 90, 333, torch.int8, "int8", 26, alpha=3, beta=-2, c_dist="int")
    got = oracle_mod.gemm_s8(p.A, p.B, 3, -2, p.C0)
    exact = 3 * (p.A.numpy().astype(np.int64) @ p.B.numpy().astype(np.int64)) \
        - 2 * p.C0.numpy().astype(np.int64)
    wrapped = ((exact + 2 ** 31) % 2 ** 32 - 2 ** 31).astype(np.int32)
    np.testing.assert_array_equal(got, wrapped)


def test_int8_wraparound_matches_big_integers(oracle_mod):
    """Results that overflow int32 wrap modulo 2^32 (two's complement)."""
    K = 8192
    A = torch.full((2, K), -128, dtype=torch.int8)
    B = torch.full((K, 2), -128, dtype=torch.int8)
    C0 = torch.tensor([[2**31 - 1, -2**31], [123456789, -987654321]], dtype=torch.int32)
    alpha, beta = 2**31 - 1, -2**31
    got = oracle_mod.gemm_s8(A, B, alpha, beta, C0)
    acc = K * 16384
    for i in range(2):
        for j in range(2):
            v = (alpha * acc + beta * int(C0[i, j])) % 2 ** 32
            v = v - 2 ** 32 if v >= 2 ** 31 else v
            assert got[i, j] == v


def test_int8_beta_zero_and_padding(oracle_mod):
    from dense_gemm_row_gb300 import workloads as w
    p = w.problem(17, 19, 40, torch.int8, "int8", 27)
    q = w.problem(17, 19, 40, torch.int8, "int8", 27, lda=48, ldb=64)
    junk = torch.full((17, 19), -5, dtype=torch.int32)
    np.testing.assert_array_equal(oracle_mod.gemm_s8(q.A, q.B, 1, 0, junk),
                                  oracle_mod.gemm_s8(p.A, p.B))


def test_bad_shapes_rejected(oracle_mod):
    lib = oracle_mod._lib()
    assert lib.oracle_gemm_f64(-1, 2, 2, 1.0, None, 2, None, 2, 0.0, None, 2) == -1
    assert lib.oracle_gemm_f64(2, 2, 3, 1.0, None, 2, None, 2, 0.0, None, 2) == -1  # lda < K
    assert lib.oracle_gemm_s8(2, 4, 3, 1, None, 3, None, 3, 0, None, 4) == -1  # ldb < N


def test_ldc_padding_direct(oracle_mod):
    """C with row stride ldc > N, through the C entry points directly: the
    padding columns keep their poison and the M x N window holds the product."""
    import ctypes
    lib = oracle_mod._lib()
    A = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])          # 3 x 2
    B = np.array([[1.0, 0.0, -1.0], [2.0, 1.0, 0.5]])          # 2 x 3
    ldc = 5
    C = np.full((3, ldc), np.nan)
    C[:, :3] = 1.0
    st = lib.oracle_gemm_f64(3, 3, 2, 1.0, A.ctypes.data, 2, B.ctypes.data, 3, 2.0,
                             C.ctypes.data, ldc)
    assert st == 0
    # rows: [1+4, 0+2, -1+1] = [5, 2, 0]; [3+8, 4, -3+2] = [11, 4, -1]; [5+12, 6, -5+3]
    np.testing.assert_array_equal(C[:, :3], np.array([[5, 2, 0], [11, 4, -1], [17, 6, -2]]) + 2.0)
    assert np.isnan(C[:, 3:]).all()
    Ci = np.full((2, 4), -7, dtype=np.int32)
    a8 = np.array([[1, -2], [3, 4]], dtype=np.int8)
    b8 = np.array([[5, 6, 7], [-8, 9, 10]], dtype=np.int8)
    st = lib.oracle_gemm_s8(2, 3, 2, 1, a8.ctypes.data, 2, b8.ctypes.data, 3, 0,
                            Ci.ctypes.data, 4)
    assert st == 0
    # [5+16, 6-18, 7-20] = [21, -12, -13]; [15-32, 18+36, 21+40] = [-17, 54, 61]
    np.testing.assert_array_equal(Ci[:, :3], [[21, -12, -13], [-17, 54, 61]])
    assert (Ci[:, 3] == -7).all()


# ------------------------------------------------------------------ uint8 (u8 -> int)

def test_uint8_matches_numpy_int64(oracle_mod):
    """unsigned char inputs (the WMMA table's u8 -> int row) against numpy's
    int64 matmul, then int32 wrap-around."""
    g = torch.Generator().manual_seed(31)
    A = torch.randint(0, 256, (37, 300), generator=g, dtype=torch.int32).to(torch.uint8)
    B = torch.randint(0, 256, (300, 29), generator=g, dtype=torch.int32).to(torch.uint8)
    C0 = torch.randint(-1000, 1000, (37, 29), generator=g, dtype=torch.int32)
    got = oracle_mod.gemm_u8(A, B, 5, -3, C0)
    exact = 5 * (A.numpy().astype(np.int64) @ B.numpy().astype(np.int64)) \
        - 3 * C0.numpy().astype(np.int64)
    np.testing.assert_array_equal(got, ((exact + 2**31) % 2**32 - 2**31).astype(np.int32))


def test_uint8_extremes_and_wrap(oracle_mod):
    """All-255 operands: every entry is 65025 * K (no sign), and K = 40000
    overflows int32 and wraps."""
    for K in (1, 1000, 40000):
        A = torch.full((2, K), 255, dtype=torch.uint8)
        B = torch.full((K, 3), 255, dtype=torch.uint8)
        v = (65025 * K) % 2**32
        v = v - 2**32 if v >= 2**31 else v
        assert (oracle_mod.gemm_u8(A, B) == v).all()


def test_uint8_hand_computed(oracle_mod):
    A = torch.tensor([[200, 1], [0, 255]], dtype=torch.uint8)
    B = torch.tensor([[3, 128], [250, 2]], dtype=torch.uint8)
    # [200*3 + 1*250, 200*128 + 1*2] = [850, 25602]; [0 + 255*250, 0 + 255*2] = [63750, 510]
    np.testing.assert_array_equal(oracle_mod.gemm_u8(A, B), [[850, 25602], [63750, 510]])


# ------------------------------------------------------------- 16-bit encoders

def test_encode_f16_round_trips_every_pattern(oracle_mod):
    """Every finite binary16 value encodes back to its own bits (-0 included);
    every NaN pattern encodes to a NaN."""
    for h in range(65536):
        x = oracle_mod.decode_f16(h)
        e = oracle_mod.encode_f16(x)
        if np.isnan(x):
            assert (e & 0x7c00) == 0x7c00 and (e & 0x3ff) != 0
        else:
            assert e == h, (hex(h), x, hex(e))


def test_encode_bf16_round_trips_every_pattern(oracle_mod):
    for h in range(65536):
        x = oracle_mod.decode_bf16(h)
        e = oracle_mod.encode_bf16(x)
        if np.isnan(x):
            assert (e & 0x7f80) == 0x7f80 and (e & 0x7f) != 0
        else:
            assert e == h, (hex(h), x, hex(e))


def _f16_probe_values(seed):
    """Random doubles over binary16's range, plus exact midpoints between
    neighbouring binary16 values and points just off them (the round-to-even
    cases), subnormals and overflow."""
    rng = np.random.default_rng(seed)
    vals = list(rng.standard_normal(2000) * np.exp2(rng.integers(-26, 17, 2000)))
    h = rng.integers(0, 0x7bff, 500).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    vals += list(mid) + list(-mid) + list(np.nextafter(mid, 0)) + list(np.nextafter(mid, 1e9))
    vals += [65504.0, 65519.99, 65520.0, -65520.0, 1e6, 2**-24, 2**-25, 3 * 2**-26, 1e-9, 0.0]
    return vals


@pytest.mark.parametrize("seed", range(3))
def test_encode_f16_matches_numpy(oracle_mod, seed):
    """numpy's float64 -> float16 cast rounds to nearest, ties to even, in one
    step: the library reference for binary16 rounding."""
    with np.errstate(over="ignore"):
        for x in _f16_probe_values(seed):
            assert oracle_mod.encode_f16(x) == int(np.float16(x).view(np.uint16)), x


@pytest.mark.parametrize("seed", range(3))
def test_encode_bf16_matches_torch_on_float32_values(oracle_mod, seed):
    """torch's float32 -> bfloat16 cast rounds to nearest, ties to even; for
    values that are exact in float32 it is the one rounding of the value."""
    g = torch.Generator().manual_seed(100 + seed)
    x = torch.randn(3000, generator=g) * torch.exp2(torch.randint(-140, 120, (3000,), generator=g)
                                                     .float())
    bits16 = torch.randint(0, 0x7f7f, (500,), generator=g, dtype=torch.int32)
    lo = (bits16 << 16).view(torch.float32)
    mid = ((bits16 << 16) + 0x8000).view(torch.float32)   # exact midpoint to the next value
    x = torch.cat([x, lo, mid, -mid, mid.nextafter(torch.zeros(1)),
                   torch.tensor([3.3895313892515355e38, 3.40282e38, 1e-40, 1e-45])])
    ref = x.to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xffff
    for v, r in zip(x.tolist(), ref.tolist()):
        assert oracle_mod.encode_bf16(v) == r, v


def test_encode_ties_go_to_even(oracle_mod):
    """Hand cases: halfway between two binary16 values the even one wins."""
    # 1 + 2^-11 lies halfway between 1 (even) and 1 + 2^-10 (odd)
    assert oracle_mod.encode_f16(1 + 2**-11) == 0x3C00
    # 1 + 3 * 2^-11 lies halfway between 1 + 2^-10 (odd) and 1 + 2^-9 (even)
    assert oracle_mod.encode_f16(1 + 3 * 2**-11) == 0x3C02
    # bfloat16 keeps 7 fraction bits: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6
    assert oracle_mod.encode_bf16(1 + 2**-8) == 0x3F80
    assert oracle_mod.encode_bf16(1 + 3 * 2**-8) == 0x3F82


# ------------------------------------------------------------- 16-bit outputs

@pytest.mark.parametrize("seed", range(4))
def test_f16_output_equals_numpy_rounding_of_exact_result(oracle_mod, seed):
    """Small-integer fp16 inputs make the product exact in float64, so numpy's
    float64 arithmetic and its one-step float16 cast give the exact answer."""
    g = torch.Generator().manual_seed(200 + seed)
    M, N, K = 9, 11, 37
    A = torch.randint(-40, 41, (M, K), generator=g).to(torch.float16)
    B = torch.randint(-40, 41, (K, N), generator=g).to(torch.float16)
    C0 = (torch.randn(M, N, generator=g) * 100).to(torch.float16)
    alpha, beta = 0.3, -1.75
    got = oracle_mod.gemm_out16(A, B, alpha, beta, C0)
    acc = A.double().numpy() @ B.double().numpy()
    ref = (alpha * acc + beta * C0.double().numpy()).astype(np.float16)
    np.testing.assert_array_equal(got.numpy().view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("seed", range(4))
def test_bf16_output_equals_torch_rounding_of_exact_result(oracle_mod, seed):
    """Integer results below 2^24 are exact in float32, where torch's bf16
    cast is the one rounding of the exact value."""
    g = torch.Generator().manual_seed(300 + seed)
    M, N, K = 7, 13, 50
    A = torch.randint(-60, 61, (M, K), generator=g).to(torch.bfloat16)
    B = torch.randint(-60, 61, (K, N), generator=g).to(torch.bfloat16)
    C0 = torch.randint(-5000, 5000, (M, N), generator=g).to(torch.bfloat16)
    got = oracle_mod.gemm_out16(A, B, 2.0, 3.0, C0)
    exact = 2 * (A.to(torch.int64) @ B.to(torch.int64)) + 3 * C0.to(torch.int64)
    ref = exact.to(torch.float32).to(torch.bfloat16)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_out16_beta_zero_does_not_read_c(oracle_mod):
    A = torch.ones(3, 4, dtype=torch.float16)
    B = torch.ones(4, 5, dtype=torch.float16)
    C0 = torch.full((3, 5), float("nan"), dtype=torch.float16)
    got = oracle_mod.gemm_out16(A, B, 1.0, 0.0, C0)
    assert (got == 4).all()


# ------------------------------------------------------------------------ tf32

def test_round_tf32_hand_values(oracle_mod):
    """tf32 keeps 10 fraction bits; the 13 lower ones are cleared (truncation)."""
    assert oracle_mod.round_tf32(1.0) == 1.0
    assert oracle_mod.round_tf32(1 + 2**-10) == 1 + 2**-10          # representable
    assert oracle_mod.round_tf32(1 + 2**-11) == 1.0                  # below the last bit
    assert oracle_mod.round_tf32(1 + 2**-10 + 2**-11 + 2**-20) == 1 + 2**-10
    assert oracle_mod.round_tf32(-(1 + 2**-10 + 2**-11)) == -(1 + 2**-10)  # toward zero
    assert oracle_mod.round_tf32(3 * 2**-130) == 3 * 2**-130         # subnormal, few bits
    x = float(np.float32(np.pi))
    assert oracle_mod.round_tf32(x) == 3.140625                      # 1.1001001000b * 2


def test_tf32_gemm_on_tf32_exact_inputs_is_the_fp32_gemm(oracle_mod):
    """Inputs that already fit in tf32 (integers below 2^11) are unchanged, so
    the tf32 GEMM equals the exact integer product."""
    g = torch.Generator().manual_seed(41)
    A = torch.randint(-1000, 1001, (21, 33), generator=g).float()
    B = torch.randint(-1000, 1001, (33, 17), generator=g).float()
    got = oracle_mod.gemm(A, B, 1.0, 0.0, tf32=True)
    np.testing.assert_array_equal(got, (A.to(torch.int64) @ B.to(torch.int64)).double().numpy())


def test_tf32_gemm_ignores_low_fraction_bits(oracle_mod):
    """Brute force on a tiny case: adding 2^-12 to a value near 1 (below tf32's
    last fraction bit) must not change the tf32 product."""
    A = torch.tensor([[1 + 2**-12, 2.0], [3.0, 1 + 2**-10 + 2**-13]], dtype=torch.float32)
    B = torch.tensor([[1 + 2**-11, 1.0], [1.0, 4.0]], dtype=torch.float32)
    got = oracle_mod.gemm(A, B, 1.0, 0.0, tf32=True)
    a = [[Fraction(1), Fraction(2)], [Fraction(3), 1 + Fraction(1, 1024)]]
    b = [[Fraction(1), Fraction(1)], [Fraction(1), Fraction(4)]]
    for i in range(2):
        for j in range(2):
            assert got[i, j] == float(sum(a[i][k] * b[k][j] for k in range(2)))

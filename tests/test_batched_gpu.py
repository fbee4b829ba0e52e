"""GPU parity of the extended entry points (gemm_*_ex: strided-batched GEMM with
transposed operands) against the CPU oracle applied to each batch entry.

For every entry b the oracle computes alpha * op(A_b) * op(B_b) + beta * C_b
with op(X) materialised on the CPU (a transposed copy), so the oracle itself
is the plain GEMM it always was. Operands live in flat buffers with poisoned
row padding and gaps between matrices; the outputs sit in a canary-filled
buffer, so reads of padding and writes outside any C window both show.
Bars as for the plain entry points: bit-exact for int8, relative Frobenius
<= 1e-5 (per batch entry) for the floating types."""
import numpy as np
import pytest
import torch

from dense_gemm_row_gb300 import workloads as w
from tests.gpu_util import CANARY_F32, CANARY_I32, GUARD_ALIGNED, GUARD_UNALIGNED, rel_frobenius

pytestmark = pytest.mark.gpu

TOL = 1e-5
DTYPES = [torch.float32, torch.bfloat16, torch.float16, torch.int8]
OPS = ["NN", "NT", "TN", "TT"]


@pytest.fixture(autouse=True)
def clean_error_word(gemm_mod):
    gemm_mod.check_device_error()
    yield
    torch.cuda.synchronize()
    assert gemm_mod.check_device_error() == 0


def is_half(dtype):
    return dtype in (torch.bfloat16, torch.float16)


def pad_ld(dtype, cols, extra):
    """A row stride >= cols: the tensor-core entry points need multiples of 8."""
    ld = cols + extra
    return (ld + 7) // 8 * 8 if is_half(dtype) else ld


def gap_for(dtype, gap):
    return (gap + 7) // 8 * 8 if is_half(dtype) else gap


class BandedStack:
    """`batch` M x N outputs (row stride ldc, matrix stride M*ldc + gap) in one
    flat device buffer, with canaries before, after, between and in padding."""

    def __init__(self, C0s, ldc, gap, aligned=True):
        self.batch = len(C0s)
        self.M, self.N = C0s[0].shape
        self.ldc, self.stride = ldc, self.M * ldc + gap
        self.guard = GUARD_ALIGNED if aligned else GUARD_UNALIGNED
        dtype = C0s[0].dtype
        self.canary = CANARY_I32 if dtype == torch.int32 else CANARY_F32
        n = self.guard + self.batch * self.stride + GUARD_UNALIGNED
        self.flat = torch.full((n,), self.canary, dtype=dtype, device="cuda")
        for b, c0 in enumerate(C0s):
            self.mat(b).copy_(c0)

    @property
    def base(self):
        return self.flat[self.guard:]

    def mat(self, b, flat=None):
        flat = self.flat if flat is None else flat
        off = self.guard + b * self.stride
        return flat[off:off + (self.M - 1) * self.ldc + self.N].as_strided(
            (self.M, self.N), (self.ldc, 1))

    def results(self):
        flat = self.flat.cpu()
        return [self.mat(b, flat).clone() for b in range(self.batch)]

    def check_canaries(self):
        flat = self.flat.cpu()
        mask = torch.ones_like(flat, dtype=torch.bool)
        for b in range(self.batch):
            self.mat(b, mask).fill_(False)
        assert bool((flat[mask] == self.canary).all()), "a kernel wrote outside the C windows"


def op_of(m, t):
    return m.t().contiguous() if t else m


def run_case(gemm_mod, oracle_mod, dtype, ops, batch, M, N, K, *, seed, alpha=None, beta=None,
             a_shared=False, b_shared=False, gap=3, extra=5, aligned=True, c_nan=False):
    a_t, b_t = ops[0] == "T", ops[1] == "T"
    is_int = dtype == torch.int8
    dist = "int8" if is_int else "uniform_pm1"
    alpha = (3 if is_int else 1.5) if alpha is None else alpha
    beta = (-2 if is_int else -0.5) if beta is None else beta
    a_rows, a_cols = (K, M) if a_t else (M, K)
    b_rows, b_cols = (N, K) if b_t else (K, N)
    sa = w.stack(1 if a_shared else batch, a_rows, a_cols, dtype, dist, seed,
                 ld=pad_ld(dtype, a_cols, extra), gap=gap_for(dtype, gap))
    sb = w.stack(1 if b_shared else batch, b_rows, b_cols, dtype, dist, seed + 1000,
                 ld=pad_ld(dtype, b_cols, extra), gap=gap_for(dtype, gap))
    out_dtype = torch.int32 if is_int else torch.float32
    c_dist = "int8" if is_int else "uniform_pm1"
    if c_nan and not is_int:
        c_dist = "nan"
    C0s = [w.matrix(M, N, torch.float32, c_dist, seed + 2000 + b).to(out_dtype)
           for b in range(batch)]
    # Aligned: C base, row stride and matrix stride in whole 16-byte units (the
    # tensor-core epilogue then writes through TMA when N % 4 == 0).
    ldc = (N + 3 + 3) // 4 * 4 if aligned else N + 1
    out = BandedStack(C0s, ldc, gap=4 if aligned else 5, aligned=aligned)
    A_dev, B_dev = sa.flat.cuda(), sb.flat.cuda()
    fn = {torch.float32: gemm_mod.gemm_f32_ex, torch.bfloat16: gemm_mod.gemm_bf16_ex,
          torch.float16: gemm_mod.gemm_f16_ex, torch.int8: gemm_mod.gemm_s8_ex}[dtype]
    fn(gemm_mod.OP_T if a_t else gemm_mod.OP_N, gemm_mod.OP_T if b_t else gemm_mod.OP_N,
       M, N, K, alpha, A_dev, sa.ld, 0 if a_shared else sa.stride, B_dev, sb.ld,
       0 if b_shared else sb.stride, beta, out.base, ldc, out.stride, batch)
    torch.cuda.synchronize()
    got = out.results()
    for b in range(batch):
        A_b = op_of(sa.mat(0 if a_shared else b), a_t)
        B_b = op_of(sb.mat(0 if b_shared else b), b_t)
        if is_int:
            ref = oracle_mod.gemm_s8(A_b, B_b, int(alpha), int(beta), C0s[b])
            np.testing.assert_array_equal(got[b].numpy(), ref, err_msg=f"batch entry {b}")
        else:
            ref = oracle_mod.gemm(A_b, B_b, alpha, beta, None if beta == 0 else C0s[b])
            err = rel_frobenius(got[b].numpy(), ref)
            assert err <= TOL, f"batch entry {b}: relative Frobenius error {err:.3e}"
    out.check_canaries()


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_batched_transposed_multi_tile(gemm_mod, oracle_mod, dtype, ops):
    """Three entries of 300 x 520 x 200: several 256 x 256 tiles per entry with
    ragged edges in m, n and k, few enough tiles that the k-split tail runs."""
    run_case(gemm_mod, oracle_mod, dtype, ops, 3, 300, 520, 200, seed=11)


@pytest.mark.parametrize("aligned_ld", [False, True], ids=["ld_odd", "ld_mod4"])
@pytest.mark.parametrize("ops", OPS)
def test_f32_batch_full_grid(gemm_mod, oracle_mod, ops, aligned_ld):
    """fp32 batches of at least two waves of resident CTAs (40 entries of 4 x 4
    tiles) run the 128-thread SIMT shape, in every operand form: ragged sizes
    with odd row strides (4-byte copies), and 512-wide operands with row and
    matrix strides in whole 16-byte units (16-byte copies)."""
    if aligned_ld:
        run_case(gemm_mod, oracle_mod, torch.float32, ops, 40, 512, 512, 136, seed=23,
                 gap=4, extra=4)
    else:
        run_case(gemm_mod, oracle_mod, torch.float32, ops, 40, 500, 510, 137, seed=29)


@pytest.mark.parametrize("aligned_ld", [False, True], ids=["ld_odd", "ld_mod4"])
@pytest.mark.parametrize("ops", ["NT", "TT"])
def test_f32_transposed_b_many_rows(gemm_mod, oracle_mod, ops, aligned_ld):
    """fp32, B stored N x K, one problem of at least two waves of tiles and
    >= 1024 rows: B is first transposed into scratch, then the straight-B
    kernel runs. Ragged N with an odd row stride (4-byte transpose reads) and
    16-byte-aligned strides."""
    if aligned_ld:
        run_case(gemm_mod, oracle_mod, torch.float32, ops, 1, 3200, 3200, 136, seed=31,
                 gap=4, extra=4)
    else:
        run_case(gemm_mod, oracle_mod, torch.float32, ops, 1, 3200, 3203, 137, seed=37)


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_single_entry_transposed(gemm_mod, oracle_mod, dtype, ops):
    """batch = 1 with transposes, deep k (the int8 path's exact 1024-k chunks)."""
    run_case(gemm_mod, oracle_mod, dtype, ops, 1, 130, 264, 2100, seed=21)


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_unaligned_c_stack(gemm_mod, oracle_mod, dtype, ops):
    """C 4 bytes off a 16-byte boundary with an odd row stride: plain stores."""
    run_case(gemm_mod, oracle_mod, dtype, ops, 2, 97, 75, 61, seed=31, aligned=False)


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_bmm_shape_of_the_survey(gemm_mod, oracle_mod, dtype):
    """(10, 16, 64) x (10, 64, 128): the batched product of the dlog page's
    PyTorch survey (section 矩阵相乘的若干写法, torch.bmm)."""
    run_case(gemm_mod, oracle_mod, dtype, "NN", 10, 16, 128, 64, seed=41, gap=0, extra=0)


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_qk_transpose_of_the_survey(gemm_mod, oracle_mod, dtype):
    """Q K^T over (batch 2 x heads 8) entries of 10 x 64: the einsum
    'b h q d, b h k d -> b h q k' of the same section, as B transposed."""
    run_case(gemm_mod, oracle_mod, dtype, "NT", 16, 10, 10, 64, seed=51, gap=0, extra=0)


@pytest.mark.parametrize("shared", ["a", "b"])
@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_shared_operand_stride_zero(gemm_mod, oracle_mod, dtype, shared):
    """A stride of 0: one matrix used by every entry (broadcast)."""
    run_case(gemm_mod, oracle_mod, dtype, "NT" if shared == "a" else "TN", 4, 140, 136, 96,
             seed=61, a_shared=shared == "a", b_shared=shared == "b")


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_many_small_entries(gemm_mod, oracle_mod, dtype):
    """More entries than units of work: 200 entries of 24 x 40 x 72."""
    run_case(gemm_mod, oracle_mod, dtype, "TN", 200, 24, 40, 72, seed=71)


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_k_zero_and_beta_zero(gemm_mod, oracle_mod, dtype):
    """K = 0 scales every C entry by beta; beta = 0 never reads C (NaN C0 for
    the floating types would otherwise show)."""
    run_case(gemm_mod, oracle_mod, dtype, "TT", 3, 40, 36, 0, seed=81)
    run_case(gemm_mod, oracle_mod, dtype, "NT", 3, 40, 36, 24, seed=82, beta=0, c_nan=True)


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_plain_form_matches_plain_entry(gemm_mod, dtype):
    """OP_N, OP_N, batch = 1 is the plain entry point: identical bits."""
    is_int = dtype == torch.int8
    M, N, K = 77, 96, 136
    dist = "int8" if is_int else "normal"
    A = w.matrix(M, K, dtype, dist, 5).cuda()
    B = w.matrix(K, N, dtype, dist, 6).cuda()
    out_dtype = torch.int32 if is_int else torch.float32
    C1 = torch.zeros(M, N, dtype=out_dtype, device="cuda")
    C2 = torch.zeros(M, N, dtype=out_dtype, device="cuda")
    gemm_mod.gemm(A, B, C1)
    gemm_mod.gemm_batched(A.unsqueeze(0), B.unsqueeze(0), C2.unsqueeze(0))
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def test_gemm_batched_tensor_api(gemm_mod, oracle_mod):
    """The tensor-level wrapper: 3-D operands, a transposed view passed as the
    stored matrix, and an operand expanded along the batch (stride 0)."""
    batch, M, N, K = 5, 72, 90, 56  # stored row lengths M and K: multiples of 8
    A = torch.stack([w.matrix(K, M, torch.bfloat16, "normal", 90 + b) for b in range(batch)])
    Bs = w.matrix(N, K, torch.bfloat16, "normal", 99)
    C = torch.zeros(batch, M, N, dtype=torch.float32, device="cuda")
    # A stored (batch, K, M) -> trans_a; B one N x K matrix for every entry -> trans_b
    Ad = A.cuda()
    Bd = Bs.cuda().unsqueeze(0).expand(batch, N, K)
    gemm_mod.gemm_batched(Ad, Bd, C, 2.0, 0.0, trans_a=True, trans_b=True)
    torch.cuda.synchronize()
    got = C.cpu()
    for b in range(batch):
        ref = oracle_mod.gemm(A[b].t().contiguous(), Bs.t().contiguous(), 2.0, 0.0)
        assert rel_frobenius(got[b].numpy(), ref) <= TOL

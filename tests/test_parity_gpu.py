"""GPU parity: every C-ABI entry point against the CPU oracle on the same seeded
inputs. Bit-exact for int8 and for integer-valued fp32 (and for integer-valued
16-bit inputs whose sums stay below 2^24); relative Frobenius error <= 1e-5
against the float64 oracle otherwise."""
import itertools

import numpy as np
import pytest
import torch

from dense_gemm_row_gb300 import workloads as w
from tests.gpu_util import (Banded, assert_within, dev_copy, fp32_accumulation_bound,
                            rel_frobenius)

pytestmark = pytest.mark.gpu

TOL = 1e-5
FLOAT_DTYPES = [torch.float32, torch.bfloat16, torch.float16]
ALL_DTYPES = FLOAT_DTYPES + [torch.int8]


@pytest.fixture(autouse=True)
def clean_error_word(gemm_mod):
    gemm_mod.check_device_error()
    yield
    torch.cuda.synchronize()
    assert gemm_mod.check_device_error() == 0


def poison_of(dtype):
    return w.INT8_POISON if dtype == torch.int8 else float("nan")


def run_gpu(gemm_mod, p: w.Problem, ldc=None, aligned=True) -> tuple[torch.Tensor, Banded]:
    A = dev_copy(p.A, poison_of(p.A.dtype))
    B = dev_copy(p.B, poison_of(p.B.dtype))
    out = Banded(p.C0.contiguous(), ldc, aligned)
    gemm_mod.gemm(A, B, out.C, p.alpha, p.beta)
    torch.cuda.synchronize()
    return out.result(), out


def oracle_of(oracle_mod, p: w.Problem, rows=None):
    if rows is None:
        if p.A.dtype == torch.int8:
            return oracle_mod.gemm_s8(p.A, p.B, int(p.alpha), int(p.beta), p.C0)
        return oracle_mod.gemm(p.A, p.B, p.alpha, p.beta, p.C0)
    return oracle_mod.gemm_rows(p.A, p.B, rows, p.alpha, p.beta, p.C0)


def assert_parity(got, ref, exact):
    got = got.numpy() if isinstance(got, torch.Tensor) else got
    if exact:
        np.testing.assert_array_equal(got.astype(np.float64) if got.dtype != np.int32 else got,
                                      ref)
    else:
        err = rel_frobenius(got, ref)
        assert err <= TOL, f"relative Frobenius error {err:.3e} > {TOL}"


# ----------------------------------------------------------- the five configs

def test_config_f32_int128_bit_exact(gemm_mod, oracle_mod):
    p = w.config("f32_int128")
    got, out = run_gpu(gemm_mod, p)
    assert_parity(got, oracle_of(oracle_mod, p), exact=True)
    out.check_canaries()


def test_config_f32_ragged(gemm_mod, oracle_mod):
    p = w.config("f32_ragged")
    got, out = run_gpu(gemm_mod, p)
    assert_parity(got, oracle_of(oracle_mod, p), exact=False)
    out.check_canaries()


@pytest.mark.parametrize("name", ["f32_4096", "bf16_8192", "f16_8192", "s8_8192"])
def test_config_full_size(gemm_mod, oracle_mod, name):
    """Full-size configs in the launch configuration the benchmark times (the
    plain C-ABI call, contiguous A, B and C), every element of C against the
    oracle. int8: bit-exact. Floating: relative Frobenius error <= 1e-5 and,
    element by element, within the worst-case fp32 accumulation error of the
    exact result, so that one wrong tile cannot hide in the norm."""
    p = w.config(name)
    got, out = run_gpu(gemm_mod, p)
    ref = oracle_of(oracle_mod, p)
    if p.A.dtype == torch.int8:
        assert_parity(got, ref, exact=True)
    else:
        assert_parity(got, ref, exact=False)
        assert_within(got.numpy(), ref,
                      fp32_accumulation_bound(oracle_mod, p.A, p.B, p.alpha, p.beta, p.C0))
    out.check_canaries()


# ------------------------------------------------------------- edge sweep

EDGE = [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 63, 65, 127, 128, 129, 255, 257]


def edge_shapes(count, seed):
    rng = np.random.default_rng(seed)
    allc = list(itertools.product(EDGE, EDGE, EDGE))
    idx = rng.choice(len(allc), size=count, replace=False)
    picked = [allc[i] for i in idx]
    return picked + [(1, 1, 1), (257, 257, 257), (129, 1, 257), (1, 257, 129)]


def ld_for(dtype, cols):
    # The tensor-core entry points need row strides that are multiples of 8.
    if dtype in (torch.bfloat16, torch.float16):
        return (cols + 7) // 8 * 8
    return None


@pytest.mark.parametrize("c_layout", ["c_aligned", "c_unaligned"])
@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
@pytest.mark.parametrize("shape", edge_shapes(24, 3), ids=lambda s: "x".join(map(str, s)))
def test_edge_sweep(gemm_mod, oracle_mod, dtype, shape, c_layout):
    """Aligned C: 16-byte aligned base and ldc % 4 == 0 (tensor-core epilogue
    through TMA stores / reduce-adds). Unaligned C: plain guarded stores."""
    M, N, K = shape
    if dtype == torch.int8:
        p = w.problem(M, N, K, dtype, "int8", 100 + M + 7 * N + 13 * K, alpha=3, beta=-2,
                      c_dist="int")
    else:
        p = w.problem(M, N, K, dtype, "uniform_pm1", 100 + M + 7 * N + 13 * K, alpha=1.5,
                      beta=-0.5, c_dist="uniform_pm1", lda=ld_for(dtype, K), ldb=ld_for(dtype, N))
    aligned = c_layout == "c_aligned"
    ldc = (N + 4) // 4 * 4 + 4 if aligned else N + 3
    got, out = run_gpu(gemm_mod, p, ldc=ldc, aligned=aligned)
    assert_parity(got, oracle_of(oracle_mod, p), exact=(dtype == torch.int8))
    out.check_canaries()


@pytest.mark.parametrize("c_layout", ["c_aligned", "c_unaligned"])
@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
def test_many_tiles_ragged_tail(gemm_mod, oracle_mod, dtype, c_layout):
    """Several tiles in each direction plus a ragged tail in M, N and K."""
    M, N, K = 397, 611, 1111
    if dtype == torch.int8:
        p = w.problem(M, N, K, dtype, "int8", 41, alpha=-1, beta=1, c_dist="int",
                      lda=1120, ldb=640)
    else:
        p = w.problem(M, N, K, dtype, "normal", 41, alpha=0.5, beta=2.0, c_dist="normal",
                      lda=1120, ldb=616)
    aligned = c_layout == "c_aligned"
    got, out = run_gpu(gemm_mod, p, ldc=652 if aligned else 651, aligned=aligned)
    assert_parity(got, oracle_of(oracle_mod, p), exact=(dtype == torch.int8))
    out.check_canaries()


@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
def test_tiled_page_odd_shape_exact(gemm_mod, oracle_mod, dtype):
    """The tiled-multiply page's harness: 47 x 804 times 804 x 53 with integers
    0..99 (rand() % 100). Every partial sum is an integer below 2^24 and the
    values are exact in every input type, so every path must be bit-exact."""
    M, K, N = 47, 804, 53
    A = w.matrix(M, K, torch.float32, "int0_99", 51)
    B = w.matrix(K, N, torch.float32, "int0_99", 52)
    if dtype == torch.int8:
        A, B = A - 50, B - 50  # int8 range
        C0 = torch.zeros(M, N, dtype=torch.int32)
    else:
        C0 = torch.zeros(M, N)
    lda, ldb = (808, 56) if dtype in (torch.bfloat16, torch.float16) else (K, N)
    Ap = torch.zeros((M, lda), dtype=dtype)[:, :K]
    Bp = torch.zeros((K, ldb), dtype=dtype)[:, :N]
    Ap.copy_(A)
    Bp.copy_(B)
    one, zero = (1, 0) if dtype == torch.int8 else (1.0, 0.0)
    p = w.Problem("odd", Ap, Bp, C0, one, zero)
    got, out = run_gpu(gemm_mod, p)
    assert_parity(got, oracle_of(oracle_mod, p), exact=True)
    out.check_canaries()


# ------------------------------------------------------------ special cases

@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
def test_beta_zero_never_reads_c(gemm_mod, oracle_mod, dtype):
    M, N, K = 130, 260, 70
    if dtype == torch.int8:
        p = w.problem(M, N, K, dtype, "int8", 61, alpha=2, beta=0)
        p.C0 = torch.full((M, N), -7, dtype=torch.int32)
    else:
        p = w.problem(M, N, K, dtype, "normal", 61, alpha=2.0, beta=0.0, c_dist="nan",
                      lda=ld_for(dtype, K), ldb=ld_for(dtype, N))
    got, _ = run_gpu(gemm_mod, p)
    if dtype != torch.int8:
        assert torch.isfinite(got).all()
    assert_parity(got, oracle_of(oracle_mod, p), exact=(dtype == torch.int8))


@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
def test_alpha_zero_and_k_zero(gemm_mod, oracle_mod, dtype):
    M, N = 67, 45
    for K, alpha in ((33, 0), (0, 1)):
        if dtype == torch.int8:
            p = w.problem(M, N, K, dtype, "int8", 71, alpha=alpha, beta=-3, c_dist="int")
        else:
            # beta = -2: beta*C is exact in fp32, so the fp32 result equals the
            # float64 oracle bit for bit.
            p = w.problem(M, N, K, dtype, "normal", 71, alpha=float(alpha), beta=-2.0,
                          c_dist="normal", lda=ld_for(dtype, max(K, 1)), ldb=ld_for(dtype, N))
        got, out = run_gpu(gemm_mod, p, ldc=N + 3)
        ref = oracle_of(oracle_mod, p)
        # alpha*acc + beta*C with alpha = 0 or an empty sum is exactly beta*C.
        assert_parity(got, ref, exact=True)
        out.check_canaries()


def test_int8_extremes_and_chunk_boundary(gemm_mod, oracle_mod):
    """All -128: every output is K * 16384. At K = 8192 the int8 path's exact
    fp32 partial sums reach 2^24 per 1024-long chunk."""
    for K in (1023, 1024, 1025, 8192):
        A = torch.full((200, K), -128, dtype=torch.int8)
        B = torch.full((K, 300), -128, dtype=torch.int8)
        p = w.Problem("ext", A, B, torch.zeros(200, 300, dtype=torch.int32), 1, 0)
        got, _ = run_gpu(gemm_mod, p)
        assert (got == K * 16384).all()
        B2 = torch.full((K, 300), 127, dtype=torch.int8)
        p2 = w.Problem("ext2", A, B2, torch.zeros(200, 300, dtype=torch.int32), 1, 0)
        got2, _ = run_gpu(gemm_mod, p2)
        assert (got2 == -K * 16256).all()


def test_int8_wraparound(gemm_mod, oracle_mod):
    p = w.problem(150, 270, 2048, torch.int8, "int8", 81, alpha=2**31 - 1, beta=-2**31,
                  c_dist="int")
    got, _ = run_gpu(gemm_mod, p)
    assert_parity(got, oracle_of(oracle_mod, p), exact=True)


@pytest.mark.parametrize("dtype", FLOAT_DTYPES, ids=str)
def test_identity_returns_b(gemm_mod, dtype):
    """A = I: C = B exactly (each output is one product by 1 plus zeros)."""
    K, N = 256, 264
    I = torch.eye(K, dtype=dtype)
    B = w.matrix(K, N, dtype, "normal", 91)
    p = w.Problem("eye", I, B, torch.zeros(K, N), 1.0, 0.0)
    got, _ = run_gpu(gemm_mod, p)
    np.testing.assert_array_equal(got.numpy(), B.to(torch.float32).numpy())


def test_streams_are_respected(gemm_mod, oracle_mod):
    """Work is enqueued on the given stream: results are ready after that
    stream is synchronised."""
    p = w.problem(512, 512, 512, torch.bfloat16, "normal", 95)
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.zeros(512, 512, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gemm_mod.gemm_bf16(512, 512, 512, 1.0, A, 512, B, 512, 0.0, C, 512, s)
    s.synchronize()
    assert rel_frobenius(C.cpu().numpy(), oracle_of(oracle_mod, p)) <= TOL


# ------------------------------------------------------ work split across SMs

@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
@pytest.mark.parametrize("shape", [(4096, 4096, 1024), (2304, 6400, 2048), (300, 4100, 3072),
                                   (16, 8192, 4096), (520, 130, 9000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_split_tail_shapes(gemm_mod, oracle_mod, dtype, shape):
    """Shapes whose tile count leaves a partial last wave (so leftover tiles are
    split along k between SMs, later parts adding into C), with beta != 0 so
    that part 0's beta*C and the later parts' additions both matter. Every
    element is checked, in both C layouts (the inputs are the same for both)."""
    M, N, K = shape
    ref = None
    for aligned in (True, False):
        if dtype == torch.int8:
            p = w.problem(M, N, K, dtype, "int8", 131 + M, alpha=-3, beta=7, c_dist="int")
        else:
            p = w.problem(M, N, K, dtype, "normal", 131 + M, alpha=0.75, beta=-1.25,
                          c_dist="normal", lda=ld_for(dtype, K), ldb=ld_for(dtype, N))
        ldc = (N + 3) // 4 * 4 if aligned else N + 1
        got, out = run_gpu(gemm_mod, p, ldc=ldc, aligned=aligned)
        if ref is None:
            ref = oracle_of(oracle_mod, p)
        assert_parity(got, ref, exact=(dtype == torch.int8))
        out.check_canaries()


@pytest.mark.parametrize("shape,ldb", [((3203, 3202, 301), None), ((2560, 4100, 520), None),
                                       ((3200, 3200, 200), 3201)],
                         ids=["n_mod4_2", "vec_b_ragged_k", "ldb_odd"])
def test_f32_full_grid_shapes(gemm_mod, oracle_mod, shape, ldb):
    """fp32 grids of at least two waves of resident CTAs run the 128-thread
    SIMT shape (8 x 16 outputs per thread, 8-deep k tiles): 16-byte and 4-byte
    copies of B, ragged M, N and K, both C layouts; every element."""
    M, N, K = shape
    ref = None
    for aligned in (True, False):
        p = w.problem(M, N, K, torch.float32, "normal", 171 + M, alpha=-0.5, beta=1.5,
                      c_dist="normal", ldb=ldb)
        ldc = (N + 3) // 4 * 4 if aligned else N + 1
        got, out = run_gpu(gemm_mod, p, ldc=ldc, aligned=aligned)
        if ref is None:
            ref = oracle_of(oracle_mod, p)
        assert_parity(got, ref, exact=False)
        out.check_canaries()


# ---------------------------------------------------------- short, wide shapes

@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
@pytest.mark.parametrize("M", [1, 5, 16, 17, 32, 33, 48, 64, 65])
def test_skinny_shapes(gemm_mod, oracle_mod, dtype, M):
    """Few rows of A (for M <= 32: the transposed-role tensor-core kernel, and
    for fp32 / int8 the small-M kernel when A and B rows are 16-byte multiples;
    fp32 with 33..64 rows: two small-M passes; the tiled kernels above), a
    ragged N and a K that is split across SMs, with beta != 0; every output
    checked. K = 3008 keeps int8 rows 16-byte multiples, K = 3000 does not
    (fallback paths)."""
    N = 2056
    for aligned, K in ((True, 3008), (False, 3000), (True, 3000)):
        if dtype == torch.int8:
            p = w.problem(M, N, K, dtype, "int8", 211 + M, alpha=5, beta=-3, c_dist="int")
        else:
            p = w.problem(M, N, K, dtype, "normal", 211 + M, alpha=-0.5, beta=1.5,
                          c_dist="normal", lda=ld_for(dtype, K), ldb=ld_for(dtype, N))
        ldc = N if aligned else N + 1
        got, out = run_gpu(gemm_mod, p, ldc=ldc, aligned=aligned)
        assert_parity(got, oracle_of(oracle_mod, p), exact=(dtype == torch.int8))
        out.check_canaries()


@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
@pytest.mark.parametrize("shape", [(1, 8192, 8192), (16, 8192, 8192), (64, 8192, 8192),
                                   (8192, 1, 8192), (8192, 16, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bench_memory_bound_shapes_from_hbm(gemm_mod, oracle_mod, dtype, shape):
    """The short, wide and tall, narrow shapes the bench times, at its sizes,
    with the large operand read from HBM: several different large operands
    (together more than twice the L2; four for int8, two otherwise) are used
    by back-to-back calls in turn, as the bench does, so TMA and load
    completions arrive in the order DRAM gives them. Every element of every
    call against the oracle (int8 bit-exact)."""
    M, N, K = shape
    if dtype in (torch.bfloat16, torch.float16) and N < 8:
        pytest.skip("16-bit B rows must be a whole number of 16-byte units")
    tall = M > N
    copies = 4 if dtype == torch.int8 else 2
    dist = "int8" if dtype == torch.int8 else "normal"
    small = w.matrix(*((K, N) if tall else (M, K)), dtype, dist, 7100 + M + N)
    bigs = [w.matrix(*((M, K) if tall else (K, N)), dtype, dist, 7200 + j) for j in range(copies)]
    small_d = small.cuda()
    bigs_d = [b.cuda() for b in bigs]
    out_dt = torch.int32 if dtype == torch.int8 else torch.float32
    outs = [torch.zeros(M, N, dtype=out_dt, device="cuda") for _ in range(copies)]
    for j in range(copies):
        A, B = (bigs_d[j], small_d) if tall else (small_d, bigs_d[j])
        gemm_mod.gemm(A, B, outs[j])
    torch.cuda.synchronize()
    assert gemm_mod.check_device_error() == 0
    for j in range(copies):
        A, B = (bigs[j], small) if tall else (small, bigs[j])
        if dtype == torch.int8:
            np.testing.assert_array_equal(outs[j].cpu().numpy(), oracle_mod.gemm_s8(A, B))
        else:
            assert_parity(outs[j].cpu(), oracle_mod.gemm(A, B), exact=False)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.int8], ids=str)
@pytest.mark.parametrize("shape", [(9, 2048, 4096), (24, 4160, 8200), (32, 8192, 2048),
                                   (16, 19200, 1024), (40, 3000, 3000), (64, 4096, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_skinny_cluster_split(gemm_mod, oracle_mod, dtype, shape):
    """9..64 rows and 16..151 column blocks of 128: the cluster form of the
    transposed-role kernel (the CTAs that split one column block's k range form
    a cluster and add their partial sums in CTA order through distributed
    shared memory). int8 with K not a multiple of 16 takes the same kernel on
    widened operands (1024-k units). Every output checked (M is small)."""
    M, N, K = shape
    if dtype == torch.int8:
        K = K + 3  # rows not 16-byte multiples: not the small-M kernel
        p = w.problem(M, N, K, dtype, "int8", 401 + M, alpha=3, beta=-2, c_dist="int")
    else:
        p = w.problem(M, N, K, dtype, "normal", 401 + M, alpha=0.5, beta=-1.0, c_dist="normal")
    got, out = run_gpu(gemm_mod, p)
    assert_parity(got, oracle_of(oracle_mod, p), exact=(dtype == torch.int8))
    out.check_canaries()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("shape", [(1, 128, 8192), (16, 2056, 1000), (32, 39000, 256),
                                   (64, 4096, 64), (5, 640, 4104)],
                         ids=lambda s: "x".join(map(str, s)))
def test_skinny_cluster_edges(gemm_mod, oracle_mod, dtype, shape):
    """Cluster form of the transposed-role kernel at its edges: one column
    block whose k range is split eight ways (1 x 128 x 8192), a ragged N and K
    (17 blocks, 16 k-blocks of which the last is partial, clusters of 8), more
    column blocks than fit on the device at once (305 blocks: no split, several
    waves), a single k-block (no split) and a ragged k split into parts of
    unequal length. beta != 0 with C read through an unaligned row stride;
    every output checked, and a second call gives the same bits."""
    M, N, K = shape
    p = w.problem(M, N, K, dtype, "normal", 701 + M + N, alpha=0.75, beta=-1.25,
                  c_dist="normal", lda=ld_for(dtype, K), ldb=ld_for(dtype, N))
    got, out = run_gpu(gemm_mod, p, ldc=N + 1, aligned=False)
    assert_parity(got, oracle_of(oracle_mod, p), exact=False)
    out.check_canaries()
    again, _ = run_gpu(gemm_mod, p, ldc=N + 1, aligned=False)
    assert torch.equal(got, again)


@pytest.mark.parametrize("shape", [(10, 2048, 1024), (16, 2064, 8192), (16, 39040, 1024),
                                   (48, 4096, 3072), (12, 2048, 4112), (64, 2048, 2048),
                                   (33, 2080, 5120), (5, 2048, 2048), (9, 4096, 1040)],
                         ids=lambda s: "x".join(map(str, s)))
def test_skinny_int8_cluster(gemm_mod, oracle_mod, shape):
    """int8 with A and B rows in whole 16-byte units and 5..64 rows: the
    cluster form reads both operands as bytes and widens them in shared memory
    (row bounds 16, 32 and 64), splitting k on 1024-k chunks across a cluster:
    one chunk (no split), a ragged N, more column blocks than fit at once,
    three chunks (clusters of 2), a ragged last chunk, 64 rows, and the 5- and
    9-row problems it takes from the dp4a kernel; beta != 0, every output
    bit-exact, and a second call gives the same bits."""
    M, N, K = shape
    p = w.problem(M, N, K, torch.int8, "int8", 801 + M, alpha=-5, beta=3, c_dist="int")
    got, out = run_gpu(gemm_mod, p, ldc=N + 3, aligned=False)
    assert_parity(got, oracle_of(oracle_mod, p), exact=True)
    out.check_canaries()
    again, _ = run_gpu(gemm_mod, p, ldc=N + 3, aligned=False)
    assert torch.equal(got, again)


@pytest.mark.parametrize("M", [20, 64])
def test_skinny_int8_cluster_cold_operands(gemm_mod, oracle_mod, M):
    """The int8 cluster form on operands read from HBM, not L2: four
    different 8192 x 8192 B matrices (268 MB, twice the L2) used in turn by
    eight back-to-back calls, so that TMA copies of one k-block can land
    after those of the next. With 17 to 64 rows the ring of raw stages has 3
    stages shared by the two converter groups, whose waits must not run ahead
    of the other group's use of a stage. Every output bit-exact."""
    N = K = 8192
    g = torch.Generator().manual_seed(4242 + M)
    A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    Bs = [torch.randint(-128, 128, (K, N), generator=g, dtype=torch.int8) for _ in range(4)]
    A_d = A.cuda()
    B_d = [b.cuda() for b in Bs]
    outs = [torch.empty(M, N, dtype=torch.int32, device="cuda") for _ in range(8)]
    for j, C in enumerate(outs):
        gemm_mod.gemm_s8(M, N, K, 1, A_d, K, B_d[j % 4], N, 0, C, N)
    torch.cuda.synchronize()
    assert gemm_mod.check_device_error() == 0
    refs = [oracle_mod.gemm_s8(A, b) for b in Bs]
    for j, C in enumerate(outs):
        np.testing.assert_array_equal(C.cpu().numpy(), refs[j % 4])


@pytest.mark.parametrize("shape", [(10, 2048, 2048, 1000), (16, 4100, 4112, 3072),
                                   (16, 8192, 8192, 4101), (24, 4096, 4096, 2048),
                                   (32, 2048, 2064, 3000), (33, 2048, 2064, 2049),
                                   (48, 4096, 4096, 1024), (64, 8192, 8192, 3072),
                                   (64, 4100, 4112, 4101), (12, 16384, 16384, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_skinny_int8_b_as_stored(gemm_mod, oracle_mod, shape):
    """int8 with 10..64 rows, at least 16 column blocks and B rows in whole
    16-byte units: the transposed-role kernel reads B as stored and its
    converter warps widen each tile to fp16 in shared memory (A slots for 16,
    32 or 64 rows). Ragged N under a padded row stride, K not a multiple of
    the 64-deep tile (zero-filled tail), beta != 0; every output bit-exact."""
    M, N, ldb, K = shape
    p = w.problem(M, N, K, torch.int8, "int8", 601 + M, alpha=-3, beta=2, c_dist="int", ldb=ldb)
    got, out = run_gpu(gemm_mod, p)
    assert_parity(got, oracle_of(oracle_mod, p), exact=True)
    out.check_canaries()


def test_skinny_int8_b_as_stored_extremes(gemm_mod, oracle_mod):
    """All -128: every 1024-k chunk sums to 1024 * 16384 = 2^24, the largest
    value the exact fp32 chunks must hold; K = 4096 spans four chunks."""
    M, N, K = 32, 2048, 4096
    A = torch.full((M, K), -128, dtype=torch.int8)
    B = torch.full((K, N), -128, dtype=torch.int8)
    C = torch.zeros(M, N, dtype=torch.int32, device="cuda")
    gemm_mod.gemm(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.cpu().numpy(), oracle_mod.gemm_s8(A, B))


def _ld16(dtype, cols):
    """A row stride in whole 16-byte units (the narrow-N kernel's condition on A)."""
    per = {torch.float32: 4, torch.bfloat16: 8, torch.float16: 8, torch.int8: 16}[dtype]
    return (cols + per - 1) // per * per


@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
@pytest.mark.parametrize("shape", [(512, 1, 1000), (4097, 3, 3001), (2048, 8, 8192),
                                   (600, 5, 4100), (8192, 1, 8192), (1111, 2, 37),
                                   (1500, 9, 2049), (2050, 16, 4100), (8192, 16, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_narrow_n_shapes(gemm_mod, oracle_mod, dtype, shape):
    """Tall, narrow problems (N <= 16, at least 512 rows; 16-bit inputs N <= 2,
    wider ones take the tiled tensor-core kernel) on the narrow-N kernel:
    A streamed once with 16-byte loads (its row stride padded to 16 bytes),
    B staged in shared memory in 1024-k chunks (512 for 16 fp32 columns; a
    ragged last chunk, a K shorter than one 16-byte load of a lane's slice), N
    rounded up to 1, 2, 4, 8 or 16 (two output elements per lane at 16), rows
    that do not fill the last CTA; beta != 0 with an unaligned C; every element
    checked, and a second call gives the same bits."""
    M, N, K = shape
    ldb = _ld16(dtype, N) if dtype in (torch.bfloat16, torch.float16) else None  # ldb % 8 == 0
    if dtype == torch.int8:
        p = w.problem(M, N, K, dtype, "int8", 951 + M, alpha=-3, beta=2, c_dist="int",
                      lda=_ld16(dtype, K))
    else:
        p = w.problem(M, N, K, dtype, "normal", 951 + M, alpha=0.5, beta=-1.5, c_dist="normal",
                      lda=_ld16(dtype, K), ldb=ldb)
    got, out = run_gpu(gemm_mod, p, ldc=N + 1, aligned=False)
    assert_parity(got, oracle_of(oracle_mod, p), exact=(dtype == torch.int8))
    out.check_canaries()
    again, _ = run_gpu(gemm_mod, p, ldc=N + 1, aligned=False)
    assert torch.equal(got, again)


@pytest.mark.parametrize("dtype", [torch.float32, torch.int8], ids=str)
@pytest.mark.parametrize("shape,ldb", [((1030, 6, 2050), 8), ((2049, 13, 1500), 16),
                                       ((600, 12, 3000), 12), ((512, 4, 1025), 4)],
                         ids=["6in8", "13in16", "12in12", "4in4"])
def test_narrow_n_vector_staging(gemm_mod, oracle_mod, dtype, shape, ldb):
    """The narrow-N kernel's vector staging of B (row stride a multiple of 4:
    fp32 in 16-byte loads of 4 columns, int8 in 4 x 4 byte blocks transposed
    in registers), including a last group of columns that ends inside the row
    padding (6 of 8, 13 of 16), a ragged last chunk of k, and K not a multiple
    of 4 (rows of a block beyond K are zeros); every element checked."""
    M, N, K = shape
    if dtype == torch.int8:
        p = w.problem(M, N, K, dtype, "int8", 77 + N, alpha=2, beta=-3, c_dist="int",
                      lda=_ld16(dtype, K), ldb=ldb)
    else:
        p = w.problem(M, N, K, dtype, "normal", 77 + N, alpha=1.5, beta=0.25, c_dist="normal",
                      lda=_ld16(dtype, K), ldb=ldb)
    got, out = run_gpu(gemm_mod, p, ldc=N)
    assert_parity(got, oracle_of(oracle_mod, p), exact=(dtype == torch.int8))
    out.check_canaries()


@pytest.mark.parametrize("dtype", ALL_DTYPES, ids=str)
@pytest.mark.parametrize("shape", [(8, 520, 8192), (32, 1024, 4096), (1, 128, 16384),
                                   (3, 4096, 2048)], ids=lambda s: "x".join(map(str, s)))
def test_deep_k_split(gemm_mod, oracle_mod, dtype, shape):
    """Few column blocks and a long k range: k is split many ways across SMs and
    the last part of each column block adds all parts' partial sums in order."""
    M, N, K = shape
    if dtype == torch.int8:
        p = w.problem(M, N, K, dtype, "int8", 307 + N, alpha=-7, beta=2, c_dist="int")
    else:
        p = w.problem(M, N, K, dtype, "normal", 307 + N, alpha=1.25, beta=-0.75,
                      c_dist="normal", lda=ld_for(dtype, K), ldb=ld_for(dtype, N))
    got, out = run_gpu(gemm_mod, p, ldc=N)
    assert_parity(got, oracle_of(oracle_mod, p), exact=(dtype == torch.int8))
    out.check_canaries()
    # Deterministic: the same call gives the same bits.
    again, _ = run_gpu(gemm_mod, p, ldc=N)
    assert torch.equal(got, again)

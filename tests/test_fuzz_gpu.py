"""Seeded random sweep over the extended entry points (gemm_{f32,bf16,f16,s8}_ex)
against the CPU oracle: element type, operand forms, batch count, shared
operands (matrix stride 0), short-wide / mid / full-grid sizes, padded row
strides and gaps between matrices, alpha and beta (including beta = 0 over a
NaN-filled C, which must not be read), aligned and unaligned C. Each case
goes through the same checks as the targeted batched tests (per-entry oracle,
canaries around every C window; bit-exact for int8, relative Frobenius
<= 1e-5 otherwise). Sizes come in four classes: short and wide, a few ragged
tiles, full grids, and deep k over few tiles. The plain form with batch 1
takes the plain entry points' routes (short-wide kernels, SIMT grid forms,
k-split tail), so the sweep also crosses the routing thresholds at random
points."""
import numpy as np
import pytest
import torch

from tests.test_batched_gpu import run_case

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.bfloat16, torch.float16, torch.int8]
OPS = ["NN", "NN", "NN", "NT", "TN", "TT"]


@pytest.fixture(autouse=True)
def clean_error_word(gemm_mod):
    gemm_mod.check_device_error()
    yield
    torch.cuda.synchronize()
    assert gemm_mod.check_device_error() == 0


def draw_cases(count, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(count):
        dtype = DTYPES[rng.integers(len(DTYPES))]
        ops = OPS[rng.integers(len(OPS))]
        size = rng.integers(4)
        if size == 0:    # short and wide
            M, N, K = rng.integers(1, 71), rng.integers(64, 1100), rng.integers(16, 1500)
            batch = 1
        elif size == 1:  # a few tiles each way, ragged
            M, N, K = rng.integers(65, 700), rng.integers(65, 700), rng.integers(1, 900)
            batch = int(rng.choice([1, 1, 2, 3]))
        elif size == 2:  # enough tiles for the full-grid forms
            M, N, K = rng.integers(700, 1400), rng.integers(700, 1400), rng.integers(64, 400)
            batch = 1
        else:            # deep k over few tiles: the k-split tail, int8 1024-k chunks
            M, N, K = rng.integers(64, 300), rng.integers(64, 300), rng.integers(2000, 6000)
            batch = int(rng.choice([1, 1, 2]))
        is_int = dtype == torch.int8
        if is_int:
            alpha = int(rng.integers(-3, 4))
            beta = int(rng.choice([0, 0, 1, -2, 3]))
        else:
            alpha = float(rng.integers(-8, 9)) / 4 or 1.0
            beta = float(rng.choice([0.0, 0.0, 1.0, -0.5, 1.25]))
        cases.append(dict(
            dtype=dtype, ops=ops, batch=batch, M=int(M), N=int(N), K=int(K), seed=1000 + i,
            alpha=alpha, beta=beta,
            a_shared=bool(batch > 1 and rng.random() < 0.25),
            b_shared=bool(batch > 1 and rng.random() < 0.25),
            gap=int(rng.integers(0, 8)), extra=int(rng.integers(0, 10)),
            aligned=bool(rng.random() < 0.6),
            c_nan=bool(beta == 0 and not is_int and rng.random() < 0.5)))
    return cases


CASES = draw_cases(192, seed=2026)


def case_id(c):
    return (f"{str(c['dtype']).split('.')[-1]}-{c['ops']}-b{c['batch']}-"
            f"{c['M']}x{c['N']}x{c['K']}")


@pytest.mark.parametrize("case", CASES, ids=[case_id(c) for c in CASES])
def test_random_forms(gemm_mod, oracle_mod, case):
    c = dict(case)
    run_case(gemm_mod, oracle_mod, c.pop("dtype"), c.pop("ops"), c.pop("batch"), c.pop("M"),
             c.pop("N"), c.pop("K"), **c)

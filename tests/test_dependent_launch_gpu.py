"""Chained calls on one stream: the tensor-core kernels start as programmatic
dependents of the previous kernel on the stream (their set-up overlaps its
tail) and must not read any operand before that kernel has finished writing
it. Each chain feeds one call's output to the next call as an input, with no
synchronisation in between, and compares the final output with the CPU oracle
applied to the intermediate the GPU produced (read back afterwards).
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import rel_frobenius

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("second_m", [16, 512], ids=["short-wide", "tiled"])
def test_chain_bf16_output_feeds_next_call(gemm_mod, oracle_mod, second_m):
    """Y1 = X W1 with a bf16 C (tiled tensor-core kernel), then Z = Y1[:m] W2
    (the short, wide cluster kernel for m = 16, the tiled kernel for m = 512),
    four chains back to back on one stream, each rewriting Y1 first."""
    M, K1, N1, N2 = 512, 2048, 1024, 4096
    X = _bf16((M, K1), 1).cuda()
    W1 = _bf16((K1, N1), 2).cuda()
    W2 = _bf16((N1, N2), 3).cuda()
    Y1 = torch.empty(M, N1, dtype=torch.bfloat16, device="cuda")
    Z = torch.empty(second_m, N2, dtype=torch.float32, device="cuda")
    lib = gemm_mod
    for rep in range(4):
        # a different scale each time, so a stale Y1 would show in Z
        lib.gemm_bf16_bf16(M, N1, K1, float(rep + 1), X, K1, W1, N1, 0.0, Y1, N1)
        lib.gemm_bf16(second_m, N2, N1, 1.0, Y1, N1, W2, N2, 0.0, Z, N2)
    torch.cuda.synchronize()
    assert lib.check_device_error() == 0
    y1 = Y1[:second_m].cpu()
    ref = oracle_mod.gemm(y1, W2.cpu(), 1.0, 0.0,
                          torch.zeros(second_m, N2, dtype=torch.float32))
    err = rel_frobenius(Z.cpu().numpy(), ref)
    assert err <= TOL, f"relative Frobenius error {err:.3e} > {TOL}"
    # and Y1 is the last chain's (scale 4) product
    ref1 = oracle_mod.gemm(X[:8].cpu(), W1.cpu(), 4.0, 0.0, torch.zeros(8, N1))
    got1 = Y1[:8].float().cpu().numpy()
    np.testing.assert_allclose(got1, ref1, rtol=2 ** -7, atol=1e-2)


def test_chain_int8_widening_then_kernel_back_to_back(gemm_mod, oracle_mod):
    """gemm_s8 at a size that takes the widening launch (which also zeroes the
    kernel's split-k flags) and the tensor-core kernel started as its
    dependent, three times back to back with different operands; every output
    bit-exact."""
    M = N = K = 2048
    outs, refs = [], []
    for seed in range(3):
        g = torch.Generator().manual_seed(900 + seed)
        A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
        B = torch.randint(-128, 128, (K, N), generator=g, dtype=torch.int8)
        C = torch.empty(M, N, dtype=torch.int32, device="cuda")
        gemm_mod.gemm_s8(M, N, K, 1, A.cuda(), K, B.cuda(), N, 0, C, N)
        outs.append(C)
        refs.append((A, B))
    torch.cuda.synchronize()
    assert gemm_mod.check_device_error() == 0
    for C, (A, B) in zip(outs, refs):
        np.testing.assert_array_equal(C.cpu().numpy(), oracle_mod.gemm_s8(A, B))

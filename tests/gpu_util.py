"""Helpers shared by the GPU parity tests: device copies that keep row padding
(poisoned), canary-banded outputs, and the comparison metrics."""
from __future__ import annotations

import numpy as np
import torch

CANARY_F32 = -12345.678
CANARY_I32 = -1234567
GUARD_ALIGNED = 256    # canary elements before the C window: keeps C 16-byte aligned
GUARD_UNALIGNED = 257  # ... or moves C off every 16-byte boundary


def dev_copy(t: torch.Tensor, poison) -> torch.Tensor:
    """Copies a (possibly row-padded) CPU matrix to the GPU with the same row
    stride; the padding columns hold ``poison``."""
    rows, cols = t.shape
    ld = max(int(t.stride(0)), cols, 1) if rows > 0 else max(cols, 1)
    buf = torch.full((rows, ld), poison, dtype=t.dtype, device="cuda")
    buf[:, :cols].copy_(t)
    return buf[:, :cols]


class Banded:
    """An M x N output with row stride ldc, embedded in a flat buffer with a band
    of canary values before, after, and in every row's padding."""

    def __init__(self, C0: torch.Tensor, ldc: int | None = None, aligned: bool = True):
        """aligned: C starts on a 16-byte boundary (the tensor-core epilogue then
        writes through TMA when ldc is a multiple of 4); otherwise it starts 4
        bytes past one, which forces the plain-store epilogue."""
        M, N = C0.shape
        self.M, self.N = M, N
        self.ldc = max(N, 1) if ldc is None else ldc
        self.guard = GUARD_ALIGNED if aligned else GUARD_UNALIGNED
        self.canary = CANARY_I32 if C0.dtype == torch.int32 else CANARY_F32
        self.flat = torch.full((self.guard + M * self.ldc + GUARD_UNALIGNED,), self.canary,
                               dtype=C0.dtype, device="cuda")
        self.C = self.flat[self.guard:self.guard + M * self.ldc].view(M, self.ldc)[:, :N]
        self.C.copy_(C0)

    def result(self) -> torch.Tensor:
        return self.C.cpu()

    def check_canaries(self):
        flat = self.flat.cpu()
        mask = torch.ones_like(flat, dtype=torch.bool)
        window = mask[self.guard:self.guard + self.M * self.ldc].view(self.M, self.ldc)
        window[:, :self.N] = False
        outside = flat[mask]
        if flat.dtype.is_floating_point:
            ok = (outside == self.canary).all()
        else:
            ok = (outside == self.canary).all()
        assert bool(ok), "a kernel wrote outside the C window"


def rel_frobenius(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    if denom == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return float(num / denom)


def fp32_accumulation_bound(oracle_mod, A: torch.Tensor, B: torch.Tensor, alpha: float,
                            beta: float, C0) -> np.ndarray:
    """Elementwise worst-case error of a GEMM whose products are exact in fp32
    and whose sums are accumulated in fp32: (K + 2) * 2^-24 * (|alpha| (|A||B|)_ij
    + |beta| |C0_ij|) -- K additions and the alpha / beta epilogue, each with a
    relative error of at most one unit roundoff 2^-24. |A||B| comes from the
    oracle on the absolute values (exact in every input format)."""
    K = A.shape[1]
    absprod = oracle_mod.gemm(A.abs(), B.abs(), 1.0, 0.0)
    bound = abs(float(alpha)) * absprod
    if beta != 0 and C0 is not None:
        c0 = C0.detach().cpu().to(torch.float64).numpy() if isinstance(C0, torch.Tensor) \
            else np.asarray(C0, dtype=np.float64)
        bound += abs(float(beta)) * np.abs(c0)
    return (K + 2) * 2.0 ** -24 * bound


def assert_within(got, ref, bound, what=""):
    """|got - ref| <= bound everywhere; names the worst element otherwise."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - np.asarray(ref, dtype=np.float64))
    bad = err > bound
    if bad.any():
        i, j = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}{int(bad.sum())} elements beyond the accumulation bound; "
                             f"worst at ({i}, {j}): |err| {err[i, j]:.3e} > {bound[i, j]:.3e}")

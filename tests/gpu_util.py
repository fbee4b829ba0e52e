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


def sample_rows(M: int, count: int, seed: int) -> list[int]:
    """Rows that cover the first and last tiles, tile boundaries and random rows."""
    fixed = [0, 1, 31, 32, 63, 64, 127, 128, 129, 255, 256, M // 2, M - 129, M - 128, M - 2, M - 1]
    rng = np.random.default_rng(seed)
    rand = rng.integers(0, M, size=max(0, count - len(fixed))).tolist()
    return sorted({r for r in fixed + rand if 0 <= r < M})

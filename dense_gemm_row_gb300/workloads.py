"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random matrices; it holds none of the GEMM arithmetic.
The CPU oracle and the GPU path both consume what it returns, so the same
seed always yields the same operands on both sides.

Every draw uses a CPU ``torch.Generator`` seeded explicitly, and the result is
moved to the requested device afterwards, so a workload is reproducible on any
host. The workloads follow the pages' own data:

* integer values uniform in [0, 99] stored as float32, as the tiled-multiply
  page ("使用CUDA和瓦片算法计算矩阵乘法") fills its matrices with
  ``rand() % 100``; with K = 128 every partial sum stays below 2^24, so any
  fp32 summation order is exact;
* the odd shapes of that page's harness (47 x 804 times 804 x 53) and the
  non-tile-multiple 1023 x 777 x 513 case;
* normal(0, 1) fp32, rounded to bf16 / fp16 with round-to-nearest-even for the
  tensor-core entry points (the warp-matrix-function page's half / bf16 rows);
* int8 uniform in [-128, 127] (the same page's signed-char row).

Leading dimensions larger than the row length are produced by allocating a
wider buffer and returning a view; the padding is filled with a poison value
(NaN for floats, 0x7f for int8) so that a kernel that reads it gives a visibly
wrong answer.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

FLOAT_POISON = float("nan")
INT8_POISON = 127


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def matrix(rows: int, cols: int, dtype: torch.dtype, dist: str, seed: int,
           ld: int | None = None, device="cpu") -> torch.Tensor:
    """A rows x cols matrix with row stride ``ld`` (>= cols), drawn from ``dist``.

    dist: "int0_99" (integers 0..99), "uniform_pm1" (U[-1, 1)), "normal"
    (N(0, 1)), "int8" (integers -128..127), "uint8" (integers 0..255), "zeros",
    "nan".
    Float draws are made in float32 and then rounded to ``dtype`` with
    round-to-nearest-even (``Tensor.to``).
    """
    ld = cols if ld is None else int(ld)
    if ld < cols:
        raise ValueError("ld must be >= cols")
    g = _gen(seed)
    shape = (rows, cols)
    if dist == "int0_99":
        v = torch.randint(0, 100, shape, generator=g, dtype=torch.int32).to(torch.float32)
    elif dist == "uniform_pm1":
        v = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        v = torch.randn(shape, generator=g, dtype=torch.float32)
    elif dist == "int8":
        v = torch.randint(-128, 128, shape, generator=g, dtype=torch.int32)
    elif dist == "uint8":
        v = torch.randint(0, 256, shape, generator=g, dtype=torch.int32)
    elif dist == "zeros":
        v = torch.zeros(shape, dtype=torch.float32)
    elif dist == "nan":
        v = torch.full(shape, float("nan"), dtype=torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    v = v.to(dtype)
    if ld == cols:
        return v.contiguous().to(device)
    poison = INT8_POISON if dtype in (torch.int8, torch.uint8) else (
        -2**31 if dtype == torch.int32 else FLOAT_POISON)
    store = torch.full((rows, ld), poison, dtype=dtype)
    store[:, :cols] = v
    return store.to(device)[:, :cols]


@dataclass
class Stack:
    """`batch` row-major rows x cols matrices in one flat buffer: matrix b
    starts at element b * stride, rows are ld apart. Everything outside the
    matrices (row padding, gaps between matrices) holds the poison value."""
    flat: torch.Tensor
    batch: int
    rows: int
    cols: int
    ld: int
    stride: int

    def mat(self, b: int) -> torch.Tensor:
        """View of matrix b (rows x cols, row stride ld)."""
        if self.rows == 0 or self.cols == 0:
            return torch.empty((self.rows, self.cols), dtype=self.flat.dtype)
        base = self.flat[b * self.stride:b * self.stride + (self.rows - 1) * self.ld + self.cols]
        return base.as_strided((self.rows, self.cols), (self.ld, 1))


def stack(batch: int, rows: int, cols: int, dtype: torch.dtype, dist: str, seed: int,
          ld: int | None = None, gap: int = 0) -> Stack:
    """A Stack of `batch` independent draws of matrix(rows, cols, dtype, dist,
    seed + b), with row stride ld (>= cols) and matrix stride rows * ld + gap."""
    ld = max(cols, 1) if ld is None else int(ld)
    if ld < cols:
        raise ValueError("ld must be >= cols")
    stride = rows * ld + int(gap)
    poison = INT8_POISON if dtype in (torch.int8, torch.uint8) else FLOAT_POISON
    flat = torch.full((max(batch * stride, 1),), poison, dtype=dtype)
    st = Stack(flat, batch, rows, cols, ld, stride)
    for b in range(batch):
        st.mat(b).copy_(matrix(rows, cols, dtype, dist, seed + b))
    return st


@dataclass
class Problem:
    """Operands of one GEMM call: C = alpha*A*B + beta*C0."""
    name: str
    A: torch.Tensor
    B: torch.Tensor
    C0: torch.Tensor
    alpha: float
    beta: float

    @property
    def shape(self):
        return self.A.shape[0], self.B.shape[1], self.A.shape[1]

    def to(self, device) -> "Problem":
        return Problem(self.name, self.A.to(device), self.B.to(device), self.C0.to(device),
                       self.alpha, self.beta)


def problem(M: int, N: int, K: int, in_dtype: torch.dtype, dist: str, seed: int,
            alpha=1.0, beta=0.0, c_dist: str = "zeros", lda=None, ldb=None,
            ldc=None, name: str = "custom") -> Problem:
    """Draw A (M x K), B (K x N) and C0 (M x N) with three seeds derived from ``seed``.

    C0 is float32 for float inputs and int32 for int8 inputs.
    """
    A = matrix(M, K, in_dtype, dist, seed * 3 + 0, lda)
    B = matrix(K, N, in_dtype, dist, seed * 3 + 1, ldb)
    if in_dtype == torch.int8:
        if c_dist == "zeros":
            C0 = matrix(M, N, torch.int32, "zeros", seed * 3 + 2, ldc)
        else:
            g = _gen(seed * 3 + 2)
            c = torch.randint(-2**31, 2**31 - 1, (M, N), generator=g, dtype=torch.int64)
            C0 = c.to(torch.int32)
            if ldc is not None and ldc > N:
                store = torch.full((M, ldc), -2**31, dtype=torch.int32)
                store[:, :N] = C0
                C0 = store[:, :N]
    else:
        C0 = matrix(M, N, torch.float32, c_dist, seed * 3 + 2, ldc)
    return Problem(name, A, B, C0, alpha, beta)


# The five workloads the library is measured and checked on.
def config(name: str) -> Problem:
    """Named workloads.

    f32_int128   fp32 128^3, integers 0..99, alpha=1, beta=0 (exact: bit-identical)
    f32_ragged   fp32 M=1023 N=777 K=513, U[-1,1) A, B and C0, alpha=1.5, beta=-0.5
    f32_4096     fp32 4096^3, N(0,1), alpha=1, beta=0
    bf16_8192    bf16 8192^3, N(0,1) rounded to bf16, fp32 C, alpha=1, beta=0
    f16_8192     fp16 8192^3, N(0,1) rounded to fp16, fp32 C, alpha=1, beta=0
    s8_8192      int8 8192^3, uniform -128..127, int32 C, alpha=1, beta=0
    f32_8192, bf16_4096, s8_4096: the same recipes at the other size the
                 throughput metric names
    """
    if name == "f32_int128":
        return problem(128, 128, 128, torch.float32, "int0_99", 1, name=name)
    if name == "f32_ragged":
        return problem(1023, 777, 513, torch.float32, "uniform_pm1", 2, alpha=1.5, beta=-0.5,
                       c_dist="uniform_pm1", name=name)
    if name == "f32_4096":
        return problem(4096, 4096, 4096, torch.float32, "normal", 3, name=name)
    if name == "bf16_8192":
        return problem(8192, 8192, 8192, torch.bfloat16, "normal", 4, name=name)
    if name == "f16_8192":
        return problem(8192, 8192, 8192, torch.float16, "normal", 4, name=name)
    if name == "s8_8192":
        return problem(8192, 8192, 8192, torch.int8, "int8", 5, alpha=1, beta=0, name=name)
    if name == "f32_8192":
        return problem(8192, 8192, 8192, torch.float32, "normal", 6, name=name)
    if name == "bf16_4096":
        return problem(4096, 4096, 4096, torch.bfloat16, "normal", 7, name=name)
    if name == "s8_4096":
        return problem(4096, 4096, 4096, torch.int8, "int8", 8, alpha=1, beta=0, name=name)
    raise KeyError(name)


CONFIG_NAMES = ("f32_int128", "f32_ragged", "f32_4096", "bf16_8192", "f16_8192", "s8_8192")

"""Time one C-ABI entry point on one problem shape.

    python -m dense_gemm_row_gb300.timing --dtype bf16 --shape 16,8192,8192 [--iters 20]
        [--ops NN|NT|TN|TT] [--batch B]

Draws seeded operands of the given shape (workloads.matrix: N(0,1) for floats,
uniform -128..127 for int8; alpha = 1, beta = 0), runs the entry point a few
times as warm-up, then times --iters back-to-back calls with CUDA events on
one stream and prints one JSON line: milliseconds per call, TFLOP/s (TOPS for
int8) and the GB/s of the algorithmic bytes (A and B read once, C written
once). Used for the per-shape measurements in profiles/. To profile it, run it
with a small --iters under an ncu that leaves the GPU clocks alone and captures
one kernel, e.g.
    ncu --clock-control none --metrics gpu__time_duration.sum -k regex:gemm_tc -c 3 \
        python -m dense_gemm_row_gb300.timing --dtype bf16 --shape 16,8192,8192 --iters 3
(without --clock-control none, ncu locks the clocks of a GPU others share).

--ops and --batch time the extended entry points (gemm_*_ex): a stack of B
problems, each operand stored as op says (T: the transpose is stored); the
figures are then totals over the stack.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import binding
from . import workloads as w

_DTYPES = {"f32": (torch.float32, torch.float32, binding.gemm_f32),
           "bf16": (torch.bfloat16, torch.float32, binding.gemm_bf16),
           "f16": (torch.float16, torch.float32, binding.gemm_f16),
           "s8": (torch.int8, torch.int32, binding.gemm_s8),
           "u8": (torch.uint8, torch.int32, binding.gemm_u8),
           "f16o": (torch.float16, torch.float16, binding.gemm_f16_f16),
           "bf16o": (torch.bfloat16, torch.bfloat16, binding.gemm_bf16_bf16),
           "tf32": (torch.float32, torch.float32, binding.gemm_tf32),
           "f64": (torch.float64, torch.float64, binding.gemm_f64)}
_EX = {"f32": binding.gemm_f32_ex, "bf16": binding.gemm_bf16_ex, "f16": binding.gemm_f16_ex,
       "s8": binding.gemm_s8_ex}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--dtype", choices=sorted(_DTYPES), required=True)
    ap.add_argument("--shape", required=True, help="M,N,K")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--ops", choices=["NN", "NT", "TN", "TT"], default="NN")
    ap.add_argument("--batch", type=int, default=1)
    a = ap.parse_args(argv)
    M, N, K = (int(x) for x in a.shape.split(","))
    in_dt, out_dt, fn = _DTYPES[a.dtype]
    dist = {"s8": "int8", "u8": "uint8"}.get(a.dtype, "normal")
    a_t, b_t = a.ops[0] == "T", a.ops[1] == "T"
    nb = a.batch
    A = w.stack(nb, *((K, M) if a_t else (M, K)), in_dt, dist, a.seed * 3).flat.cuda()
    B = w.stack(nb, *((N, K) if b_t else (K, N)), in_dt, dist, a.seed * 3 + 1000).flat.cuda()
    C = torch.zeros(nb * M * N, dtype=out_dt, device="cuda")
    one, zero = (1, 0) if a.dtype in ("s8", "u8") else (1.0, 0.0)
    stream = torch.cuda.current_stream()
    if (a.ops != "NN" or nb != 1) and a.dtype not in _EX:
        raise SystemExit(f"--ops/--batch: no extended entry point for {a.dtype}")
    if a.ops == "NN" and nb == 1:
        def call():
            fn(M, N, K, one, A, K, B, N, zero, C, N, stream)
    else:
        ex = _EX[a.dtype]
        ops = (binding.OP_T if a_t else binding.OP_N, binding.OP_T if b_t else binding.OP_N)

        def call():
            ex(*ops, M, N, K, one, A, M if a_t else K, M * K, B, K if b_t else N, K * N, zero, C,
               N, M * N, nb, stream)
    for _ in range(a.warmup):
        call()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(a.iters):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    binding.check_device_error()
    ms = e0.elapsed_time(e1) / a.iters
    nbytes = (A.numel() * A.element_size() + B.numel() * B.element_size()
              + C.numel() * C.element_size())
    print(json.dumps({"dtype": a.dtype, "M": M, "N": N, "K": K, "ops": a.ops, "batch": nb,
                      "iters": a.iters, "ms": ms,
                      "tflops": 2.0 * nb * M * N * K / (ms / 1e3) / 1e12,
                      "gbs": nbytes / (ms / 1e3) / 1e9}))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())

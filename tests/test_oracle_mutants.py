"""Planted mistakes: each mutant is a copy of the oracle's C source with one
plausible slip (a dropped term, a wrong sign or index, a transposed operand, a
wrong decoder constant, a lost epilogue term). It is compiled on the CPU into a
temporary library and run through the pins of ``test_oracle_pins``; every
mutant must fail at least one of them. This shows the pins are strong enough to
catch such mistakes in the real oracle."""
import os
import subprocess
import sys

import pytest

from oracle import oracle as oracle_module

SRC = os.path.join(os.path.dirname(oracle_module.__file__), "gemm_oracle.c")

# (name, [(old, new), ...]) -- each "old" must occur in the source.
MUTANTS = [
    ("sign_of_product", [("acc[j] += a * brow[j];", "acc[j] -= a * brow[j];")]),
    ("first_k_dropped", [("for (int64_t k = 0; k < K; k++) {\n                    double a",
                          "for (int64_t k = 1; k < K; k++) {\n                    double a")]),
    ("last_k_dropped", [("for (int64_t k = 0; k < K; k++) {\n                    double a",
                         "for (int64_t k = 0; k < K - 1; k++) {\n                    double a")]),
    ("A_transposed", [("double a = A[i * lda + k];", "double a = A[k * lda + i];")]),
    ("B_transposed", [("const double *brow = B + k * ldb;", "const double *brow = B + k;"),
                      ("acc[j] += a * brow[j];", "acc[j] += a * brow[j * ldb];")]),
    ("beta_not_applied", [("scaled + beta * crow[j]", "scaled + crow[j]")]),
    ("alpha_not_applied", [("double scaled = alpha * acc[j];", "double scaled = acc[j];")]),
    ("acc_not_reset", [("for (int64_t j = 0; j < N; j++) acc[j] = 0.0;", "")]),
    ("ldc_ignored", [("double *crow = C + i * ldc;", "double *crow = C + i * N;")]),
    ("lda_ignored_in_decode", [("a[i * K + k] = dec(A, i * lda + k);",
                                "a[i * K + k] = dec(A, i * K + k);")]),
    ("f16_exponent_bias", [("e - 25", "e - 24")]),
    ("f16_subnormal_scale", [("ldexp((double)m, -24)", "ldexp((double)m, -25)")]),
    ("bf16_shift", [("(uint32_t)h << 16", "(uint32_t)h << 15")]),
    ("s8_read_as_unsigned", [(": (int64_t)Bs[k * ldb + j];",
                              ": (int64_t)(uint8_t)Bs[k * ldb + j];")]),
    ("u8_read_as_signed", [("? (int64_t)Bu[k * ldb + j]", "? (int64_t)(int8_t)Bu[k * ldb + j]")]),
    ("u8_A_read_as_signed", [("? (int64_t)Au[i * lda + k]", "? (int64_t)(int8_t)Au[i * lda + k]")]),
    ("encode_ties_away_from_zero", [("(frac == 0.5 && fmod(r, 2.0) != 0.0)", "(frac == 0.5)")]),
    ("encode_truncates", [("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
                           "")]),
    ("encode_flushes_subnormals", [("if (ex < emin) ex = emin;",
                                    "if (ex < emin) return sign_bit;")]),
    ("encode_saturates_on_overflow", [("if (v > max_finite) return sign_bit | exp_all;",
                                       "if (v > max_finite) v = max_finite;")]),
    ("encode_drops_sign", [("const uint32_t sign = signbit(x) ? 1u : 0u;",
                            "const uint32_t sign = 0u;")]),
    ("tf32_clears_12_bits", [("u &= ~0x1fffu;", "u &= ~0xfffu;")]),
    ("tf32_rounds_up", [("u &= ~0x1fffu;", "u = (u + 0x1000u) & ~0x1fffu;")]),
    ("tf32_not_applied", [("return (double)oracle_round_tf32(((const float *)p)[i]);",
                           "return (double)((const float *)p)[i];")]),
    ("out16_c0_not_read", [("c[i * N + j] = (beta == 0.0) ? 0.0", "c[i * N + j] = 1 ? 0.0")]),
    ("out16_wrong_format", [("C[i * ldc + j] = is_bf16 ? oracle_encode_bf16",
                             "C[i * ldc + j] = !is_bf16 ? oracle_encode_bf16")]),
    ("s8_beta_dropped", [("v += (uint64_t)(int64_t)beta * (uint64_t)(int64_t)crow[j];",
                          "v += (uint64_t)(int64_t)crow[j];")]),
    ("s8_saturates_instead_of_wrapping",
     [("uint32_t low = (uint32_t)v; /* keep the low 32 bits */",
       "int64_t sv = (int64_t)v; if (sv > 2147483647) sv = 2147483647;"
       " if (sv < -2147483648LL) sv = -2147483648LL; uint32_t low = (uint32_t)sv;")]),
]


_CHILD = r"""
import inspect, sys
sys.path.insert(0, sys.argv[2])
import torch
from oracle import oracle as om
from tests import test_oracle_pins as pins
om._LIB = om.load(sys.argv[1])
caught = []
for name, fn in inspect.getmembers(pins, inspect.isfunction):
    if not name.startswith("test_"):
        continue
    params = list(inspect.signature(fn).parameters)
    if params == ["oracle_mod"]:
        calls = [()]
    elif params == ["oracle_mod", "seed"]:
        calls = [(s,) for s in range(4)]
    elif params == ["oracle_mod", "dtype"]:
        calls = [(torch.bfloat16,), (torch.float16,)]
    else:
        continue
    try:
        for extra in calls:
            fn(om, *extra)
    except Exception:
        caught.append(name)
print("CAUGHT", ",".join(caught))
sys.exit(0 if caught else 3)
"""


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, edits, tmp_path):
    src = open(SRC).read()
    for old, new in edits:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new, 1)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"{name}.so"
    c_path.write_text(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    str(c_path), "-o", str(so_path), "-lm"], check=True)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    # A mutant may read out of bounds and crash: run it in a child process, where
    # a crash (negative return code) also counts as caught.
    res = subprocess.run([sys.executable, "-c", _CHILD, str(so_path), root],
                         capture_output=True, text=True, timeout=600)
    assert res.returncode != 3, f"mutant {name} passed every pin"
    if res.returncode == 0:
        assert "CAUGHT" in res.stdout
    else:
        assert res.returncode < 0, res.stderr[-2000:]  # killed by a signal

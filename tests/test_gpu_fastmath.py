"""Exhaustive GPU check of the step kernel's correctly rounded square root and
reciprocal (scalar and paired FP32x2 forms), and a randomised check of its
reciprocal-based quotient.

The step kernel evaluates sqrt(v') and 1/d with a hardware approximation plus
FMA corrections (q4_fastmath.cuh).  Bit-identity with the oracle requires that
these equal IEEE round-to-nearest results, so they are compared with CUDA's
IEEE intrinsics (__fsqrt_rn, __frcp_rn, __fdiv_rn) on EVERY input of the
domain on which the kernel uses them: +0 and all positive normal floats for
the square root, every d in [2^-126, 2^126) for the reciprocal.  The quotient
(factored second moment) is checked on 2^31 random and adversarial pairs.
"""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "fastmath_check.cu")
OUT = os.path.join(HERE, "_build", "libfastmath_check.so")

# Variants the step kernel uses (template arguments in q4_step.cu).
SQRT_VARIANT = 0
RCP_VARIANT = 1


def build_checker() -> str:
    deps = [SRC, os.path.join(ROOT, "bit_quantized_adamw_q4adamw_b300", "csrc", "q4_fastmath.cuh")]
    if os.path.exists(OUT) and all(os.path.getmtime(OUT) >= os.path.getmtime(d) for d in deps):
        return OUT
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    tmp = OUT + f".tmp{os.getpid()}"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "bit_quantized_adamw_q4adamw_b300", "csrc"),
                    "-I", os.path.join(ROOT, "include"), "-fmad=false", "-prec-div=true", "-prec-sqrt=true",
                    "-ftz=false", "-Xcompiler", "-fPIC", "-shared", "-o", tmp, SRC], check=True)
    os.replace(tmp, OUT)
    return OUT


def run_check(which: int, variant: int, lo: int, hi: int):
    lib = ctypes.CDLL(build_checker())
    lib.fm_check.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p,
                             ctypes.c_void_p, ctypes.c_void_p]
    count = torch.zeros(1, dtype=torch.int64, device="cuda")
    first = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = lib.fm_check(which, variant, lo, hi, count.data_ptr(), first.data_ptr(),
                      torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    return int(count.item()), int(first.item()) & 0xFFFFFFFF


def test_sqrt_exhaustive_zero_and_positive_normals():
    n, first = run_check(0, SQRT_VARIANT, 0, 0x7F800000)
    assert n == 0, f"{n} mismatches, first input bits {first:#010x}"


def test_rcp_exhaustive_normal_range():
    n, first = run_check(1, RCP_VARIANT, 0x00800000, 0x7E800000)
    assert n == 0, f"{n} mismatches, first input bits {first:#010x}"


def test_paired_sqrt_exhaustive():
    n, first = run_check(3, 0, 0, 0x7F800000)
    assert n == 0, f"{n} mismatches, first input bits {first:#010x}"


def test_paired_rcp_exhaustive():
    n, first = run_check(3, 1, 0x00800000, 0x7E800000)
    assert n == 0, f"{n} mismatches, first input bits {first:#010x}"


def test_paired_patterns_round_like_scalar_ops():
    n, first = run_check(4, 0, 7, 1 << 28)
    assert n == 0, f"{n} mismatches, first sample {first}"


def test_quotient_random_and_adversarial_pairs():
    n, first = run_check(2, 0, 12345, 1 << 31)
    assert n == 0, f"{n} mismatches, first sample {first}"


def test_paired_quotient_random_and_adversarial_pairs():
    n, first = run_check(2, 1, 54321, 1 << 30)
    assert n == 0, f"{n} mismatches, first sample {first}"

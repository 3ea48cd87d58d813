"""The quantizers divide by the scale with Markstein's correction step instead of a
full IEEE division, and form the scale and its reciprocal the same way (a constant
divisor 448; a Newton-Raphson step plus the correction from a hardware reciprocal
approximation). tests/csrc/scale_fast_path.c checks the scale and the reciprocal for
every bf16 amax that takes that path and every binary32 significand of amax, for every
approximation within 8 units in the last place of 1 / s (the one significand of s for
which the reciprocal correction misses, all ones, is sent to division). tests/csrc/quotient_fast_path.c restates that formula on the CPU
(C99 binary32, fmaf) and compares it with IEEE division over every bf16 pair
(x, amax), |x| <= amax, whose scale the kernels send down that path, and over 2e8
random binary32 pairs (the GEMM epilogue quantizes FP32 values): bitwise equal wherever
the quotient can reach the E4M3 range, same sign and zero code elsewhere.
The GPU parity tests then check the kernels against the oracle on real data."""
import os
import shutil
import subprocess

import pytest

SRC = os.path.join(os.path.dirname(__file__), "csrc", "quotient_fast_path.c")
SRC_SCALE = os.path.join(os.path.dirname(__file__), "csrc", "scale_fast_path.c")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_fast_quotient_equals_ieee_division_on_all_bf16_pairs(tmp_path):
    exe = str(tmp_path / "qfp")
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-o", exe, SRC, "-lm"],
                   check=True)
    r = subprocess.run([exe, "1", "200"], capture_output=True, text=True, timeout=600)
    checked, bad = map(int, r.stdout.split())
    assert r.returncode == 0 and bad == 0, r.stderr[:2000]
    assert checked > 850_000_000 + 199_000_000


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_fast_scale_and_reciprocal_are_correctly_rounded(tmp_path):
    exe = str(tmp_path / "sfp")
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-o", exe, SRC_SCALE, "-lm"],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    checked, bad = map(int, r.stdout.split())
    assert r.returncode == 0 and bad == 0, r.stderr[:2000]
    assert checked > 300_000_000

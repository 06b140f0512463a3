"""CPU check of the method the fp8-cache kernels use for the quotient x / scale (a
correctly rounded reciprocal refined by two Markstein steps, for scales in [2^-64, 2^64]):
its e4m3 codes must equal those of the IEEE quotient.  tests/quotient_method.c restates
the method in C (with fmaf) and counts mismatching codes over every positive bf16 value
and random fp32 values, for fixed and random scales; then the form the kernels evaluate
(the same steps on the signed value with the negated reciprocal, each code's sign bit
flipped, NaN codes recomputed by the unsigned form) over every bf16 value of both signs,
infinities and zeros included, and random fp32 values of both signs.  The GPU parity
tests then compare the kernels with the oracle, which divides."""
from __future__ import annotations

import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent


def test_quotient_method_matches_ieee_division(tmp_path):
    exe = tmp_path / "quotient_method"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", str(exe),
                    str(HERE / "quotient_method.c"), "-lm"], check=True)
    out = subprocess.run([str(exe), "300", "20000"], capture_output=True, text=True,
                         check=True, timeout=600).stdout.split()
    pairs, bad = int(out[0]), int(out[1])
    assert pairs > 40_000_000
    assert bad == 0

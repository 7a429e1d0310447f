"""The integer-pipe binary64 addition and multiplication used by the FP64
kernels (finite_volume_field_gb300/csrc/fp64_emu.cuh) are bit-identical to
IEEE 754 round-to-nearest-even arithmetic: the same header, compiled for the
host, is checked against the host CPU's own addition and multiplication on
about 21 million operand pairs (random bit patterns, every exponent
difference up to 70, cancellations, ties, products from deep underflow to
overflow, exact and halfway products, subnormal operands, the ends of the
exponent range and special values; the complete algorithms and the fast
paths, including the fixed-factor product with either operand fixed), and
the fixed-point sum of four same-sign operands, ((a + b) + c) + d, on every
case its fast form accepts (about 5 million: spreads up to the 9-binade
limit, ties in each partial sum, all-ones significands, sums near
overflow, the diffusion's own value ranges; the written-out form and the
N-operand template must agree), the six-operand frame of the 3D update on
about 3.8 million accepted sets, and its forms that take a zero in the first
or second operand (the face-side neighbour of the cells next to a zero
face) on about 5.8 million accepted sets with that zero (and the four-operand
forms of the 2D update with such a zero, written-out and template, on about
7 million): partners at every
shift including the one the form must decline, zero and subnormal partners,
both zero signs, ties, and exponents near both limits."""
from __future__ import annotations

import re
import shutil
import subprocess
from pathlib import Path

import pytest

HERE = Path(__file__).resolve().parent


def test_emulated_add_and_mul_match_ieee(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "emu_check"
    subprocess.run([cxx, "-O2", "-ffp-contract=off", "-std=c++17", str(HERE / "emu_host_check.cpp"),
                    "-o", str(exe)], check=True, capture_output=True)
    r = subprocess.run([str(exe), "1000000"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0 " in r.stdout, r.stdout
    taken = int(re.search(r"sum4_taken (\d+)", r.stdout).group(1))
    assert taken > 4_000_000, r.stdout
    taken6 = int(re.search(r"sum6_taken (\d+)", r.stdout).group(1))
    assert taken6 > 3_000_000, r.stdout
    taken6z = int(re.search(r"sum6z_taken (\d+)", r.stdout).group(1))
    assert taken6z > 5_000_000, r.stdout
    taken4z = int(re.search(r"sum4z_taken (\d+)", r.stdout).group(1))
    assert taken4z > 6_000_000, r.stdout

"""The oracle's pins reject plausible mistakes.

Each case copies the oracle's C source, plants one mistake in the copy
(a reordered sum, a fused multiply-add, a flipped sign, a wrong neighbour
index, a missing edge write, a swapped ping-pong, a wrong ghost offset, a
swapped face, a copy of the wrong variable, swapped stage coefficients),
builds it with the oracle's flags, swaps it in for the real oracle library
and runs the named pin, which must fail.  Everything runs on the CPU; nothing here touches the GPU path.
"""
from __future__ import annotations

import contextlib
import ctypes
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

import oracle
import tests.test_oracle_diffusion as D
import tests.test_oracle_diffusion3d as D3
import tests.test_oracle_pack_flux as P
import tests.test_oracle_rk as R

SRC = Path(oracle.__file__).parent / "fvf_oracle.c"


@contextlib.contextmanager
def _mutant(tmp_path, old: str, new: str, count: int = 1):
    text = SRC.read_text()
    assert text.count(old) >= count, f"mutation anchor not found: {old!r}"
    mutated = text.replace(old, new, count)
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(mutated)
    cc = shutil.which("gcc") or "cc"
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11", str(c),
                    "-o", str(so), "-lm"], check=True, capture_output=True)
    real = oracle._load()
    lib = ctypes.CDLL(str(so))
    for name in ("oracle_diffuse2d_f64", "oracle_diffuse2d_f32", "oracle_diffuse3d_f64",
                 "oracle_diffuse3d_f32", "oracle_weno_pack",
                 "oracle_advect_rhs", "oracle_advect_rhs_add", "oracle_flux_unpack",
                 "oracle_fields_copy", "oracle_rk_axpby", "oracle_weno_pack_f32",
                 "oracle_advect_rhs_f32", "oracle_max_threads"):
        getattr(lib, name).argtypes = getattr(real, name).argtypes
        getattr(lib, name).restype = getattr(real, name).restype
    oracle._lib = lib
    try:
        yield
    finally:
        oracle._lib = real


STENCIL = ("src[c] + alpha * (src[c - 1] + src[c + 1] + src[c - nx]\n"
           "                                           + src[c + nx] - 4.0 * src[c])")
STENCIL32 = ("src[c] + alpha * (src[c - 1] + src[c + 1] + src[c - nx]\n"
             "                                           + src[c + nx] - 4.0f * src[c])")

STENCIL3D_32 = ("src[c] + alpha * (src[c - 1] + src[c + 1] + src[c - nx]\n"
                "                                               + src[c + nx] + src[c - sxy] + src[c + sxy]\n"
                "                                               - 6.0f * src[c])")

MUTANTS = [
    # (id, old, new, count, pin that must fail)
    ("sum-order-SNWE",
     STENCIL32,
     "src[c] + alpha * (src[c - nx] + src[c + nx] + src[c - 1]\n"
     "                                           + src[c + 1] - 4.0f * src[c])",
     1, lambda: D.test_printed_fp32_vs_fp64_table()),
    ("fused-multiply-add-fp32",
     STENCIL32,
     "fmaf(alpha, (src[c - 1] + src[c + 1] + src[c - nx] + src[c + nx] - 4.0f * src[c]), src[c])",
     1, lambda: D.test_printed_fp32_vs_fp64_table()),
    ("sign-of-centre-term",
     STENCIL, STENCIL.replace("- 4.0 * src[c]", "+ 4.0 * src[c]"),
     1, lambda: D.test_one_step_impulse(np.float64)),
    ("wrong-north-index",
     STENCIL, STENCIL.replace("src[c + nx] -", "src[c + nx + 1] -"),
     1, lambda: D.test_closed_form_fp64(31, 27, 8)),
    ("edges-not-zeroed",
     "dst[c] = 0.0;", "dst[c] = src[c];",
     1, lambda: D.test_brute_force_nonzero_initial_edges()),
    ("ping-pong-reversed",
     "if (s % 2 == 1)\n            step_f64(u, v",
     "if (s % 2 == 0)\n            step_f64(u, v",
     1, lambda: D.test_closed_form_centre_values()),
    ("pack-ghost-offset-dropped",
     "j = a; k = b + g2; l = c + g3;", "j = a; k = b; l = c + g3;",
     1, lambda: P.test_pack_coordinate_tags(0)),
    ("pack-y-axes-swapped",
     "j = b + g1; k = a; l = c + g3;", "j = a; k = b + g1; l = c + g3;",
     1, lambda: P.test_pack_coordinate_tags(1)),
    ("flux-faces-swapped",
     "w * (lo - hi)", "w * (hi - lo)",
     1, lambda: P.test_rhs_linear_flux_gives_minus_inv_d(0)),
    ("flux-z-spacing-index",
     "ll = l; lh = l + 1; w = inv_d[l];", "ll = l; lh = l + 1; w = inv_d[0];",
     1, lambda: P.test_rhs_linear_flux_gives_minus_inv_d(2)),
    ("rhs-add-faces-swapped",
     "const double term = inv_d[c] * (lo - hi);", "const double term = inv_d[c] * (hi - lo);",
     1, lambda: P.test_rhs_add_builds_two_direction_sum()),
    ("unpack-y-as-x",
     "src = k + F2 * (j + F1 * (l + F3 * (int64_t)i));",
     "src = j + F1 * (k + F2 * (l + F3 * (int64_t)i));",
     1, lambda: P.test_flux_unpack_coordinate_tags(1)),
    ("copy-wrong-variable",
     "dst[i][e] = src[i][e];", "dst[i][e] = src[0][e];",
     1, lambda: P.test_fields_copy_is_bitwise_identity()),
    ("copy-last-element-dropped",
     "for (int64_t e = 0; e < total; ++e)\n            dst[i][e]",
     "for (int64_t e = 0; e < total - 1; ++e)\n            dst[i][e]",
     1, lambda: P.test_fields_copy_is_bitwise_identity()),
    ("3d-centre-weight-4",
     "- 6.0 * src[c]", "- 4.0 * src[c]",
     1, lambda: D3.test_one_step_impulse_exact()),
    ("3d-z-neighbour-index",
     "src[c - sxy] + src[c + sxy]", "src[c - nx] + src[c + sxy]",
     1, lambda: D3.test_exact_on_dyadic_inputs_with_nonzero_edges()),
    ("3d-top-face-not-zeroed",
     "k == 0 || k == nz - 1) {\n                    dst[c] = 0.0;",
     "k == 0) {\n                    dst[c] = 0.0;",
     1, lambda: D3.test_exact_on_dyadic_inputs_with_nonzero_edges()),
    ("3d-sum-order-fp32",
     STENCIL3D_32,
     STENCIL3D_32.replace("src[c - 1] + src[c + 1] + src[c - nx]", "src[c - 1] + (src[c + 1] + src[c - nx])"),
     1, lambda: D3.test_summation_order_fp32_worked_value()),
    ("pack-f32-wrong-variable",
     "const float *f = fields[i];", "const float *f = fields[0];",
     1, lambda: P.test_pack_f32_coordinate_tags(1)),
    ("rhs-f32-faces-swapped",
     "const float term = inv_d[c] * (lo - hi);", "const float term = inv_d[c] * (hi - lo);",
     1, lambda: P.test_rhs_f32_linear_and_constant_flux(2)),
    ("stage-coefficients-swapped",
     "const double p = a * u0[e];\n        const double q = b * t;",
     "const double p = b * u0[e];\n        const double q = a * t;",
     1, lambda: R.test_ssprk3_closed_form_on_linear_equation(-0.5)),
    ("stage-from-un-not-u",
     "const double t = u[e] + dt * rhs[e];", "const double t = u0[e] + dt * rhs[e];",
     1, lambda: R.test_ssprk3_closed_form_on_linear_equation(-0.5)),
    ("stage-dt-dropped",
     "const double t = u[e] + dt * rhs[e];", "const double t = u[e] + rhs[e];",
     1, lambda: R.test_axpby_worked_values(1.0, 2.0, 4.0, 0.5, 0.75, 0.25, 1.75)),
]


@pytest.mark.parametrize("mid,old,new,count,pin", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_rejects_mutant(tmp_path, mid, old, new, count, pin):
    with _mutant(tmp_path, old, new, count):
        with pytest.raises(AssertionError):
            pin()


def test_unmutated_copy_passes_the_same_pins(tmp_path):
    """Sanity: a verbatim copy built the same way passes every pin above."""
    with _mutant(tmp_path, "int oracle_max_threads", "int oracle_max_threads"):
        for m in MUTANTS:
            m[4]()

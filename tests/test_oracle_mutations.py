"""Plants plausible mistakes in a copy of the oracle's C source and checks that the pins
in test_oracle_pins.py reject every one of them.

Each mutant is compiled from a temporary copy (the committed oracle is never touched),
the oracle module is pointed at it, and the pins run; at least one must fail.  This is
the evidence that the pins constrain the oracle rather than restate it.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle.build import SRC
import test_oracle_pins as pins

# (name, original text, mutated text)
MUTANTS = [
    ("mean divisor H-1", "double ms = ss / (double)H;", "double ms = ss / (double)(H - 1);"),
    ("eps outside sqrt", "1.0 / sqrt(ms + eps)", "1.0 / (sqrt(ms) + eps)"),
    ("y without w", "v_scratch[j] * rs * ld(w, w_kind, j)", "v_scratch[j] * rs"),
    ("dx drops xhat*c", "double d = rr * (g[j] - xhat[j] * c);", "double d = rr * g[j];"),
    ("dx sign", "double d = rr * (g[j] - xhat[j] * c);", "double d = rr * (g[j] + xhat[j] * c);"),
    ("dx without rstd", "double d = rr * (g[j] - xhat[j] * c);", "double d = (g[j] - xhat[j] * c);"),
    ("c not a mean", "double c = dot / (double)H;", "double c = dot;"),
    ("g without w", "g[j] = ld(dy, dy_kind, r * H + j) * ld(w, w_kind, j);",
     "g[j] = ld(dy, dy_kind, r * H + j);"),
    ("dh dropped", "if (dh) d += ld(dh, dh_kind, r * H + j);", ";"),
    ("dw without x", "dw[j] += ld(dy, dy_kind, r * H + j) * (ld(x, x_kind, base + j) * rr);",
     "dw[j] += ld(dy, dy_kind, r * H + j) * rr;"),
    ("dw one row's rstd", "double rr = r_all[r];\n    for (int32_t j = 0; j < H; ++j)\n      dw[j]",
     "double rr = r_all[0];\n    for (int32_t j = 0; j < H; ++j)\n      dw[j]"),
    ("strides swapped", "return t * s_tok + h * s_head;", "return h * s_tok + t * s_head;"),
    ("bf16 via fp32", "double q = ldexp(a, -qexp);", "double q = ldexp((double)(float)a, -qexp);"),
    ("bf16 ties away", "double n = rint(q);", "double n = round(q);"),
    ("residual unrounded", "v[j] = orc_bf16_to_f64(hb);", "v[j] = xv + ld(res, res_kind, base + j);"),
]

EPS = pins.EPS

PIN_CALLS = [
    pins.test_bf16_round_ties_and_single_rounding,
    pins.test_bf16_round_matches_torch_on_fp32_values,
    pins.test_fwd_zero_row,
    pins.test_fwd_constant_row,
    pins.test_fwd_pythagorean_row,
    pins.test_fwd_residual_sum_is_rounded_once_and_normalized,
    lambda: pins.test_bwd_finite_difference((3, 16), EPS),
    lambda: pins.test_bwd_finite_difference((2, 7), 0.3),
    pins.test_bwd_residual_combined_gradient_fd,
    lambda: pins.test_bwd_identity_x_dot_dx(0.1),
    pins.test_bwd_dw_single_row_and_constant_rows,
    pins.test_bwd_dh_is_added,
    pins.test_per_head_strided_view_matches_reshaped_plain,
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique/present"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(lib), str(path), "-lm"], check=True)
    return str(lib)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    lib = _build_mutant(tmp_path, name, old, new)
    failures = 0
    oracle.use_library(lib)
    try:
        for call in PIN_CALLS:
            try:
                with np.errstate(all="ignore"):
                    call()
            except AssertionError:
                failures += 1
    finally:
        oracle.use_library(None)
    assert failures > 0, f"no pin caught the planted mistake {name!r}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    lib = _build_mutant(tmp_path, "identity", "double ms = ss / (double)H;",
                        "double ms = ss / (double)H;")
    oracle.use_library(lib)
    try:
        for call in PIN_CALLS:
            call()
    finally:
        oracle.use_library(None)
    assert os.path.exists(lib)

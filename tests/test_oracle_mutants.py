"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle/oracle.c, builds it with gcc
into a temporary library and runs the pins of tests/test_oracle.py against it
(in place of the real oracle, through the same ctypes binding).  At least one
pin must fail for every planted mistake.  The committed oracle is untouched.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

# name -> (text in oracle.c, replacement): one plausible slip each.
MUTANTS = {
    "drops_the_last_k_term": ("  for (int64_t k = 0; k < p->K; k++) {\n    double a = p->lut[arow[k]];",
                              "  for (int64_t k = 0; k < p->K - 1; k++) {\n    double a = p->lut[arow[k]];"),
    "reads_tn_b_as_nn": ("(p->layout == OR_TN) ? p->lut[p->B[n * p->K + k]] : p->lut[p->B[k * p->N + n]]",
                         "(p->layout == OR_TN) ? p->lut[p->B[k * p->N + n]] : p->lut[p->B[k * p->N + n]]"),
    "reads_nn_b_as_tn": ("(p->layout == OR_TN) ? p->lut[p->B[n * p->K + k]] : p->lut[p->B[k * p->N + n]]",
                         "(p->layout == OR_TN) ? p->lut[p->B[n * p->K + k]] : p->lut[p->B[n * p->K + k]]"),
    "writes_c_transposed": ("      int64_t idx = m * p->N + n;", "      int64_t idx = n * p->M + m;"),
    "decode_drops_the_sign": ("  return sign ? -v : v;", "  return v;"),
    "subnormal_scale_off_by_one": ("    v = ldexp((double)frac, f->emin - f->frac_bits);",
                                   "    v = ldexp((double)frac, f->emin - f->frac_bits - 1);"),
    "ties_round_away_from_zero": ("  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "  return fl + 1.0;"),
    "truncates_instead_of_rounding": ("  double r = round_half_even(n);", "  double r = floor(n);"),
    "saturates_instead_of_overflowing": ("  if (v > maxfinite) return sign | exp_all;", "  if (v > maxfinite) v = maxfinite;"),
    "bf16_bias_wrong": ("static const fmt_t FMT_BF16 = {8, -126, 127, 127, 7, 8};",
                        "static const fmt_t FMT_BF16 = {8, -126, 127, 126, 7, 8};"),
    "abs_sum_keeps_signs": ("    sa += fabs(prod);", "    sa += prod;"),
}


def _pin_checks():
    """The pins, each with representative arguments (name, callable)."""
    checks = [
        ("decode f16 vs numpy", pins.test_decode_f16_all_patterns_matches_numpy),
        ("decode bf16 vs torch", pins.test_decode_bf16_all_patterns_matches_torch),
        ("encode f16 vs numpy", pins.test_encode_f16_matches_numpy_rne),
        ("tn and nn agree", pins.test_tn_and_nn_storage_agree),
    ]
    for case in pins.GOLDEN_CASES:
        checks.append(("golden " + case["name"], lambda c=case: pins.test_golden_products(c)))
    for fmt in ("f16", "bf16"):
        for layout in ("TN", "NN"):
            checks.append(("identity %s %s" % (fmt, layout), lambda f=fmt, l=layout: pins.test_identity_and_permutation(f, l)))
            checks.append(("integers %s %s" % (fmt, layout),
                           lambda f=fmt, l=layout: pins.test_small_integers_exact_vs_int64(f, l, (31, 8, 64))))
            checks.append(("torch %s %s" % (fmt, layout),
                           lambda f=fmt, l=layout: pins.test_float64_torch_matmul_third_opinion(f, l)))
    for layout in ("TN", "NN"):
        checks.append(("ones row %s" % layout, lambda l=layout: pins.test_ones_row_gives_column_sums(l)))
    checks.append(("all ones f16", lambda: pins.test_all_ones_gives_K("f16", 100)))
    return checks


def _build(tmp_path, old, new):
    with open(oracle._SRC) as f:
        src = f.read()
    assert src.count(old) == 1, "the planted mistake must name one place in oracle.c"
    path_c = tmp_path / "mutant.c"
    path_c.write_text(src.replace(old, new))
    path_so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", str(path_c),
                           "-o", str(path_so), "-lm"])
    return oracle._bind(str(path_so))


def test_the_real_oracle_passes_every_pin():
    for name, check in _pin_checks():
        check()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_a_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    monkeypatch.setattr(oracle, "_lib", _build(tmp_path, old, new))
    failed = []
    for check_name, check in _pin_checks():
        try:
            check()
        except (AssertionError, ValueError, RuntimeError, OverflowError):
            failed.append(check_name)
    assert failed, "no pin caught the planted mistake '%s'" % name

"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/tern_oracle.c (a dropped
factor, a wrong index, a flipped sign, eps under the root, truncation instead
of round-to-nearest, ...), builds it on the CPU, points the oracle at it and
runs the pins that cover that function: at least one of them must fail.  The
unmutated oracle passes the same pins (test_oracle_pins.py, test_oracle_sr4.py).
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as P
import test_oracle_sr4 as S
import test_oracle_split8 as S8

SRC = os.path.join(os.path.dirname(oracle.__file__), "tern_oracle.c")

# (name, text to find, replacement, occurrence (0-based), pins that must catch it)
MUTANTS = [
    ("ternary threshold off by one", "if (q >= theta) return 1;", "if (q > theta) return 1;", 0,
     [P.test_ternary_truth_table_theta2, lambda: P.test_ternary_exhaustive_int8(2)]),
    ("clamp rail one short", "if (q > clamp) return clamp;", "if (q > clamp) return clamp - 1;", 0,
     [lambda: P.test_clamp_exhaustive(7)]),
    ("bf16 rounding truncates", "double r = nearbyint(ldexp(m, 8));", "double r = floor(ldexp(m, 8));", 0,
     [P.test_bf16_round_matches_torch_rne, P.test_bf16_golden_values]),
    ("-1 packed as 10", "uint32_t code = w == 1 ? 1u : (w == -1 ? 3u : 0u);",
     "uint32_t code = w == 1 ? 1u : (w == -1 ? 2u : 0u);", 0, [P.test_pack_golden_words]),
    ("forward drops the scale", "a->out[m * a->N + c] = s * acc[c];", "a->out[m * a->N + c] = acc[c];", 0,
     [P.test_fwd_matches_library_matmul, P.test_fwd_all_positive_is_scaled_rowsum]),
    ("forward reads X transposed-ish", "double x = or_bf16_value(a->X[m * a->K + r]);",
     "double x = or_bf16_value(a->X[m * a->K + (a->K - 1 - r)]);", 0,
     [P.test_fwd_signed_permutation_is_exact, P.test_fwd_identity_weight_returns_x]),
    ("dX uses the wrong scale index", "double term = dy[c] * (double)a->scale[c] * (double)or_ternary(qrow[c], a->theta);",
     "double term = dy[c] * (double)a->scale[r % a->N] * (double)or_ternary(qrow[c], a->theta);", 0,
     [lambda: P.test_dx_is_the_gradient_of_the_loss((4, 8, 16))]),
    ("G reads the wrong X column", "double x = or_bf16_value(a->X[m * a->K + r]);",
     "double x = or_bf16_value(a->X[m * a->K + (a->K - 1 - r)]);", 1,
     [lambda: P.test_gq_is_the_straight_through_gradient((8, 16, 16)), P.test_gq_at_unit_scale_is_xt_dy]),
    ("gq drops the scale", "if (gq) gq[r * N + c] = G[r * N + c] * s;", "if (gq) gq[r * N + c] = G[r * N + c];", 0,
     [lambda: P.test_gq_is_the_straight_through_gradient((4, 8, 16))]),
    ("sgrad loses the sign of T", "s += G[r * N + c] * (double)w;", "s += G[r * N + c] * (double)abs(w);", 0,
     [lambda: P.test_sgrad_is_the_gradient_in_the_scale((4, 8, 16)), P.test_sgrad_through_the_forward]),
    ("AdamW eps under the root", "double step = lr * (mi / bc1) / (sqrt(vi / bc2) + eps);",
     "double step = lr * (mi / bc1) / sqrt(vi / bc2 + eps);", 0, [P.test_adamw_eps_sits_outside_the_root]),
    ("AdamW decay without lr", "double decay = decoupled ? lr * wd * wi : 0.0;",
     "double decay = decoupled ? wd * wi : 0.0;", 0,
     [P.test_adamw_first_step_closed_form, P.test_adamw_constant_gradient_closed_form]),
    ("AdamW bias correction of v uses beta1", "double bc2 = 1.0 - pow(b2, (double)t);",
     "double bc2 = 1.0 - pow(b1, (double)t);", 0,
     [P.test_adamw_first_step_closed_form, P.test_adamw_constant_gradient_closed_form]),
    ("SR4 steps up the gradient", "v = or_clamp(v - (int)d, clamp);", "v = or_clamp(v + (int)d, clamp);", 0,
     [S.test_round_half_up_without_dither, lambda: S.test_stochastic_rounding_is_unbiased(0.3)]),
    ("SR4 scale multiplies", "return target_step / mean;", "return target_step * mean;", 0,
     [S.test_scale_sets_the_mean_step]),
    # the tolerance denominators (sum of |term| of each output's dot product) made too large
    ("Y abs sum drops |T|", "aab[c] += fabs(term);", "aab[c] += fabs(x);", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31)]),
    ("dX abs sum drops |T|", "sa += fabs(term);",
     "sa += fabs(dy[c] * (double)a->scale[c]);", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31)]),
    ("dX abs sum counts each term twice", "sa += fabs(term);", "sa += 2.0 * fabs(term);", 0,
     [P.test_abs_sums_equal_the_outputs_when_every_term_has_one_sign]),
    ("gq abs sum drops |s|", "if (gqabs) gqabs[r * N + c] = Ga[r * N + c] * fabs(s);",
     "if (gqabs) gqabs[r * N + c] = Ga[r * N + c];", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31)]),
    ("gq abs sum uses the signed scale", "if (gqabs) gqabs[r * N + c] = Ga[r * N + c] * fabs(s);",
     "if (gqabs) gqabs[r * N + c] = Ga[r * N + c] * s;", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31)]),
    ("G abs sum without |.|", "ga[c] += fabs(term);", "ga[c] += term;", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31)]),
    ("sgrad abs sum drops |T|", "sa += Ga[r * N + c] * (double)abs(w);", "sa += Ga[r * N + c];", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31)]),
    ("sampled Y abs sum drops |s|", "*outabs = fabs((double)s) * aab;", "*outabs = aab;", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31), P.test_sampled_entries_equal_full_outputs]),
    ("sampled dX abs sum drops |T|", "aab += fabs(term);\n    }\n    *out = acc;",
     "aab += fabs(or_bf16_value(dyrow[c]) * (double)scale[c]);\n    }\n    *out = acc;", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31), P.test_sampled_entries_equal_full_outputs]),
    ("sampled gq abs sum drops |s|", "*outabs = aab * fabs((double)s);", "*outabs = aab;", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31), P.test_sampled_entries_equal_full_outputs]),
    ("sampled sgrad abs sum drops |T|", "sa += G[K + r] * (double)abs(w);", "sa += G[K + r];", 0,
     [lambda: P.test_abs_sums_are_products_of_absolute_values((12, 40, 32), 31), P.test_sampled_entries_equal_full_outputs]),
    # binary16 / E4M3 rounding and the fp16 + e4m3 split of the dX operands
    ("grid rounding ties away from zero", "double r = ldexp(nearbyint(ldexp(fabs(x), -lsb)), lsb);",
     "double r = ldexp(round(ldexp(fabs(x), -lsb)), lsb);", 0,
     [S8.test_f16_round_matches_numpy, S8.test_f16_golden_values, S8.test_e4m3_golden_values]),
    ("binary16 subnormals start one binade low", "if (e - 1 < -14) return sgn | (uint16_t)ldexp(r, 24);",
     "if (e - 1 < -15) return sgn | (uint16_t)ldexp(r, 24);", 0,
     [S8.test_f16_round_matches_numpy, S8.test_f16_golden_values]),
    ("e4m3 exponent bias 8", "return sgn | (uint8_t)((e - 1 + 7) << 3)", "return sgn | (uint8_t)((e - 1 + 8) << 3)", 0,
     [S8.test_e4m3_round_matches_torch_in_range, S8.test_e4m3_golden_values]),
    ("e4m3 without saturation", "if (r > 448.0) r = 448.0;", "if (r > 480.0) r = 480.0;", 0,
     [lambda: S8.test_e4m3_saturates(470.0)]),
    ("split mantissa in [0.5, 1)", "a = ldexp(s, -(e - 1));", "a = ldexp(s, -e);", 0,
     [S8.test_split_reconstructs_the_scale, S8.test_split_planes_match_library_conversions]),
    ("split low part scaled by 2^6", "or_e4m3_round(ldexp(a - or_f16_value(h), 7))",
     "or_e4m3_round(ldexp(a - or_f16_value(h), 6))", 0,
     [S8.test_split_reconstructs_the_scale, S8.test_split_planes_match_library_conversions]),
    ("split drops the sign of T", "(uint16_t)(w < 0 ? h ^ 0x8000u : h)", "(uint16_t)h", 0,
     [S8.test_split_reconstructs_the_scale, S8.test_split_planes_match_library_conversions]),
    ("clip inverted", "if (max_norm > 0.0 && norm > max_norm) return max_norm / norm;",
     "if (max_norm > 0.0 && norm > max_norm) return norm / max_norm;", 0,
     [P.test_sumsq_and_norm, P.test_clipped_gradient_has_the_clip_norm]),
]


def _mutant_lib(tmp, find, repl, occurrence):
    src = open(SRC).read()
    pos = -1
    for _ in range(occurrence + 1):
        pos = src.index(find, pos + 1)
    mutated = src[:pos] + repl + src[pos + len(find):]
    c = os.path.join(tmp, "mutant.c")
    so = os.path.join(tmp, "libmutant.so")
    open(c, "w").write(mutated)
    subprocess.check_call(["gcc", "-O1", "-shared", "-fPIC", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
                           "-o", so, c, "-lm", "-lpthread"])
    return so


@pytest.mark.parametrize("name,find,repl,occ,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_the_mutant(name, find, repl, occ, pins):
    with tempfile.TemporaryDirectory() as tmp:
        so = _mutant_lib(tmp, find, repl, occ)
        oracle.use_library(so)
        try:
            caught = 0
            for pin in pins:
                try:
                    pin()
                except (AssertionError, ValueError):
                    caught += 1
            assert caught >= 1, f"no pin caught the mutant: {name}"
        finally:
            oracle.use_library(None)

"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a temporary copy of oracle.c -- the
mistake lives only in that copy, compiled on the CPU -- and asserts that at
least one pin fails on it.  A pin set that let any of these through would not
be pinning the oracle.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "residual_added_first": [
        ("float acc = bf16_to_f32(partials[((int64_t)0 * T + t) * H + h]);",
         "float acc = (residual ? bf16_to_f32(residual[t * (int64_t)H + h]) : 0.0f) + "
         "bf16_to_f32(partials[((int64_t)0 * T + t) * H + h]);"),
        ("acc = acc + res;", "(void)res;"),
    ],
    "double_accumulator": [("float acc = bf16_to_f32(", "double acc = bf16_to_f32(")],
    "reversed_rank_order": [
        ("((int64_t)0 * T + t) * H + h]", "((int64_t)(R - 1) * T + t) * H + h]"),
        ("((int64_t)r * T + t) * H + h]", "((int64_t)(R - 1 - r) * T + t) * H + h]"),
    ],
    "transposed_partial_index": [("((int64_t)r * T + t) * H + h]", "((int64_t)t * R + r) * H + h]")],
    "eps_outside_sqrt": [("1.0 / sqrt(ss / (double)H + (double)eps)", "1.0 / sqrt(ss / (double)H) + (double)eps")],
    "mean_over_H_minus_1": [("ss / (double)H + (double)eps", "ss / (double)(H - 1) + (double)eps")],
    "gamma_dropped": [("x * rstd * g)", "x * rstd)")],
    "y_sign_dropped": [("oracle_bf16_from_double(x * rstd * g)", "oracle_bf16_from_double(fabs(x * rstd * g))")],
    "scale_divides_by_240": [("a / 448.0f", "a / 240.0f")],
    "absmax_without_abs": [("fabsf(bf16_to_f32(yg[i]))", "bf16_to_f32(yg[i])")],
    "zero_group_not_special": [("if (s == 0.0f) { qg[i] = 0; continue; }", "")],
    "truncating_rounding": [("nearbyint(a / ulp)", "floor(a / ulp)")],
    "rounding_ties_away": [("nearbyint(a / ulp)", "round(a / ulp)")],
    "bf16_subnormal_shift": [("ldexp(r, 133)", "ldexp(r, 132)")],
    "e4m3_subnormal_scale": [("ldexp((double)m, -6 - 3)", "ldexp((double)m, -6 - 2)")],
    "e4m3_no_saturation": [("if (r > 448.0) r = 448.0;", "")],
    "norm_without_square": [("ss += x * x;", "ss += fabs(x);")],
    "mx_emax_off_by_one": [("shared_exp = (ex - 1) - 2;", "shared_exp = (ex - 1) - 1;")],
    "mx_floor_log2_off": [("shared_exp = (ex - 1) - 2;", "shared_exp = ex - 2;")],
    "e2m1_no_saturation": [("if (r > 6.0) r = 6.0;", "")],
    "e2m1_subnormal_wrong": [("if (r < 1.0) return sign | 0x1;", "if (r < 1.0) return sign;")],
    "mx_nibble_order_swapped": [("qb[i] = (uint8_t)(lo | (hi << 4));", "qb[i] = (uint8_t)(hi | (lo << 4));")],
    "mx_no_lower_clamp": [("if (shared_exp < -127) shared_exp = -127;", "")],
    "mx_zero_block_code_one": [("int shared_exp = -127;", "int shared_exp = 0;")],
    "mx_scale_rounds_log2": [("(void)frexp(amax, &ex);", "(void)frexp(amax * 1.4142135623730951, &ex);")],
    "mx_divides_by_amax": [("ldexp(oracle_bf16_to_double(yb[2 * i]), -shared_exp)",
                            "oracle_bf16_to_double(yb[2 * i]) / amax * 6.0")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    mpath = tmp_path / "oracle_mutant.c"
    mpath.write_text(src)
    lib = oracle.load(oracle.build(str(tmp_path / "libmutant.so"), str(mpath)))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the {name} mutant"

"""The pins reject plausible mistakes in the oracle.

Each mutant is a copy of ``oracle/fp8_oracle.c`` with one planted mistake (a
dropped term, a wrong index, a wrong rounding rule ...), compiled on the CPU
into a temporary directory.  Every mutant must fail at least one of the pins
in ``test_oracle_pins.py``; the unmodified source must pass all of them.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "fp8_oracle.c")

MUTANTS = {
    "drops_a_scale": ("double scale = (double)sfa[(long)k * sfa_ld] * (double)sfb[k];",
                      "double scale = (double)sfb[k];"),
    "sfa_ignores_leading_dim": ("sfa[(long)k * sfa_ld]", "sfa[(long)k]"),
    "sfb_indexed_by_row_block": ("SFB + (long)(n / 128) * kb", "SFB + (long)(m / 128) * kb"),
    "sfb_block_of_64": ("SFB + (long)(n / 128) * kb", "SFB + (long)(n / 64 % ((N + 127) / 128)) * kb"),
    "drops_last_k_block": ("for (int k = 0; k < kb; ++k) {", "for (int k = 0; k + 1 < kb; ++k) {"),
    "ties_away_from_zero": ("r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "r = fl + 1.0;"),
    "rounds_through_fp32": ("double a = fabs(x);", "double a = fabs((double)(float)x);"),
    "truncates": ("if (frac > 0.5)\n        r = fl + 1.0;", "if (frac > 2.0)\n        r = fl + 1.0;"),
    "exponent_bias_8": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "subnormals_as_normals": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp(1.0 + (double)m / 8.0, -7);"),
    "sign_bit_ignored": ("return s ? -v : v;", "return v;"),
    "masked_count_off_by_one": ("if (m < 0 || m >= count || m >= M_max)", "if (m < 0 || m > count || m >= M_max)"),
    "acc_drops_addend": ("double v = (double)C[(long)m * N + n] +", "double v = 0.0 * (double)C[(long)m * N + n] +"),
    "acc_addend_transposed": ("C[(long)m * N + n]", "C[(long)n * M + m]"),
    "acc_addend_subtracted": ("double v = (double)C[(long)m * N + n] +", "double v = -(double)C[(long)m * N + n] +"),
    "acc_addend_rounded_to_bf16_first": ("double v = (double)C[(long)m * N + n] +",
                                         "double v = oracle_bf16_to_f64(oracle_f64_to_bf16_rne((double)C[(long)m * N + n])) +"),
    "ue8m0_bias_126": ("return ldexp(1.0, (int)e - 127);", "return ldexp(1.0, (int)e - 126);"),
    "ue8m0_sfb_by_row_block": ("oracle_ue8m0_to_f64(SFB_e[(long)(n / 128) * kb + k])",
                               "oracle_ue8m0_to_f64(SFB_e[(long)(m / 128 % ((N + 127) / 128)) * kb + k])"),
    "ue8m0_max_not_nan": ("    if (e == 0xFF)\n        return NAN;\n    return ldexp", "    return ldexp"),
    "contiguous_ignores_group": ("const uint8_t *Bg = B + (long)g * N * K;\n        const float *SFBg = SFB + (long)g * nb * kb;",
                                 "const uint8_t *Bg = B;\n        const float *SFBg = SFB;"),
}


def _pins():
    cases = pins._parse_hand_cases()
    return [
        ("decode_vs_library", lambda lib: pins.test_e4m3_decode_exhaustive_matches_library(lib)),
        ("special_values", lambda lib: pins.test_e4m3_special_values_golden(lib)),
        ("e4m3_round_trips", lambda lib: pins.test_e4m3_quantise_dequantise_round_trips(lib)),
        ("bf16_vs_library", lambda lib: pins.test_bf16_rne_matches_library_on_f32_values(lib)),
        ("bf16_fp64_cases", lambda lib: pins.test_bf16_rne_fp64_only_cases(lib)),
        ("hand_worked", lambda lib: [pins.test_hand_worked_elements(c, lib) for c in cases]),
        ("brute_force", lambda lib: pins.test_brute_force_against_dequant_matmul(5, 200, 256, lib)),
        ("exact_integer", lambda lib: pins.test_exact_integer_closed_form(6, 256, 512, lib)),
        ("double_b_scale", lambda lib: pins.test_doubling_one_b_scale_changes_exactly_its_block(lib)),
        ("double_a_scale", lambda lib: pins.test_doubling_one_a_scale_changes_exactly_its_row(lib)),
        ("contig_own_group", lambda lib: pins.test_contiguous_rows_use_their_own_group(lib)),
        ("masked_untouched", lambda lib: pins.test_masked_rows_beyond_count_untouched(lib)),
        ("masked_full", lambda lib: pins.test_masked_full_counts_equal_per_group_dense(lib)),
        ("acc_zero_addend", lambda lib: pins.test_acc_zero_addend_equals_plain(lib)),
        ("acc_zero_product", lambda lib: pins.test_acc_zero_product_rounds_the_addend_like_library(lib)),
        ("acc_exact_integer", lambda lib: pins.test_acc_exact_integer_closed_form(6, 256, 512, lib)),
        ("ue8m0_decode", lambda lib: pins.test_ue8m0_decode_exhaustive(lib)),
        ("ue8m0_vs_fp32", lambda lib: pins.test_ue8m0_reduces_to_fp32_scales(lib)),
        ("ue8m0_exact", lambda lib: pins.test_ue8m0_exact_integer_closed_form(6, 256, 512, lib)),
    ]


def _build_variant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutant {name}: pattern not found in the oracle source"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    out = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(path), "-o", str(out), "-lm"], check=True)
    return oracle.load_variant(str(out))


def _failing_pins(lib):
    failed = []
    for pname, fn in _pins():
        try:
            fn(lib)
        except AssertionError:
            failed.append(pname)
    return failed


def test_unmodified_source_passes_every_pin(tmp_path):
    src = open(SRC).read()
    lib = _build_variant(tmp_path, "unmodified", src[:20], src[:20])
    assert _failing_pins(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_variant(tmp_path, name, old, new)
    failed = _failing_pins(lib)
    assert failed, f"mutant {name} passed every pin"

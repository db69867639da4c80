"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle/gqa_oracle.c, applies one plausible mistake as a text
substitution (a wrong head map, a dropped or inverted scale, a flipped sign, an
off-by-one length, swapped planes or scales, a wrong exponent bias, rounding
ties away from zero, ...), compiles the copy into a temporary library on the
CPU, and re-runs the pin tests of test_oracle_attention.py and
test_oracle_formats.py against it.  At least one pin must fail for every
mutant; the real oracle passes them all (those tests, run normally).
"""
import os
import shutil

import pytest

import oracle
import test_oracle_append as P
import test_oracle_attention as A
import test_oracle_formats as F

SRC = os.path.join(os.path.dirname(oracle.__file__), "gqa_oracle.c")

MUTANTS = {
    "head map h%8": ("const int g = h / (ORC_HQ / ORC_HKV);", "const int g = h % ORC_HKV;"),
    "scale without 1/sqrt(d)": ("j->q_scale / sqrt((double)ORC_D)", "j->q_scale"),
    "scale times sqrt(d)": ("j->q_scale / sqrt((double)ORC_D)", "j->q_scale * sqrt((double)ORC_D)"),
    "softmax sign flipped": ("double w = exp(s[t] - m);", "double w = exp(m - s[t]);"),
    "no max subtraction": ("double w = exp(s[t] - m);", "double w = exp(s[t]);"),
    "score pass reads slot L when it exists": (
        "for (int t = 0; t < L; ++t) {\n    const double row_k",
        "for (int t = 0; t < L + (L < j->capacity); ++t) {\n    const double row_k"),
    "value pass drops the last slot": ("for (int t = 0; t < L; ++t) {\n    double w",
                                       "for (int t = 0; t < L - 1; ++t) {\n    double w"),
    "K and V planes swapped": ("(((size_t)b * 2 + 0) * ORC_HKV + g) * C * ORC_D",
                               "(((size_t)b * 2 + 1) * ORC_HKV + g) * C * ORC_D"),
    "int8 K rows scaled by the V-plane scale": ("const size_t ks_off = (((size_t)b * 2 + 0)",
                                                "const size_t ks_off = (((size_t)b * 2 + 1)"),
    "int8 scale of the next row": ("orc_decode_bf16(j->kv_scales[vs_off + t])",
                                   "orc_decode_bf16(j->kv_scales[vs_off + (t + 1) % L])"),
    "verify window shifted by one slot": ("const int L = len - j->q_len + 1 + qt;",
                                          "const int L = len - j->q_len + qt + (qt == 0);"),
    "RoPE pairs interleaved": ("    z[i] = y[i] * c - y[i + half] * s;\n    z[i + half] = y[i + half] * c + y[i] * s;",
                               "    z[2 * (i % 64)] = y[2 * (i % 64)] * c - y[2 * (i % 64) + 1] * s;\n"
                               "    z[2 * (i % 64) + 1] = y[2 * (i % 64) + 1] * c + y[2 * (i % 64)] * s;"),
    "RoPE rotation sign flipped": ("z[i + half] = y[i + half] * c + y[i] * s;", "z[i + half] = y[i + half] * c - y[i] * s;"),
    "RoPE frequency doubled": ("pow(theta, -(double)i / half)", "pow(theta, -2.0 * (double)i / half)"),
    "RMS over the sum, not the mean": ("sqrt(ss / ORC_D + eps)", "sqrt(ss + eps)"),
    "RMS eps dropped": ("sqrt(ss / ORC_D + eps)", "sqrt(ss / ORC_D)"),
    "int8 codes read as unsigned": ("if (type == ORC_I8) return (double)((const int8_t*)base)[i];",
                                    "if (type == ORC_I8) return (double)((const uint8_t*)base)[i];"),
    "k_scale applied to V": ("* j->v_scale;\n      acc", "* j->k_scale;\n      acc"),
    "v_scale dropped": ("* j->v_scale;\n      acc", ";\n      acc"),
    "f16 exponent bias off by one": ("ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    "bf16 fraction width": ("ldexp((double)(128 + m), e - 134)", "ldexp((double)(128 + m), e - 133)"),
    "e4m3 subnormal scale": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "e4m3 NaN rule": ("if (e == 0xf && m == 0x7) v = NAN;", "if (e == 0xf) v = NAN;"),
    "rounding ties away from zero": ("double r = rint(a / quantum) * quantum;",
                                     "double r = floor(a / quantum + 0.5) * quantum;"),
    "normalise by length": ("double o = acc[d] / denom;", "double o = acc[d] / L;"),
    "q element offset": ("q_off + d)", "q_off + (d ^ 1))"),
}

PINS = [
    A.test_golden_worked_examples,
    lambda lib: [A.test_length_one_returns_first_value_row(lib, k) for k in ("f16", "bf16", "e4m3")],
    lambda lib: [A.test_zero_q_scale_gives_mean_of_values(lib, k) for k in ("f16", "e4m3")],
    A.test_equal_keys_give_mean_of_values,
    A.test_large_q_scale_selects_largest_score,
    A.test_grouped_head_map,
    A.test_slots_past_length_are_never_read,
    A.test_v_scale_is_linear_and_k_scale_folds_into_q_scale,
    lambda lib: A.test_matches_torch_sdpa_on_small_workloads(lib, 1),
    A.test_matches_torch_sdpa_fp8_with_distinct_scales,
    F.test_decode_f16_all_patterns,
    F.test_decode_bf16_all_patterns,
    F.test_decode_e4m3_all_patterns,
    F.test_round_f16_matches_numpy_single_step,
    F.test_round_exact_ties_to_even,
    A.test_int8_length_one_returns_scaled_first_row,
    A.test_int8_matches_torch_sdpa_on_dequantised_rows,
    A.test_int8_scales_act_per_row,
    A.test_window_2,
    P.test_constant_vector_normalises_to_the_weight,
    P.test_position_zero_is_the_plain_rms_norm,
    lambda lib: [P.test_one_hot_rotates_into_its_rotate_half_partner(lib, i) for i in (0, 17, 63)],
    P.test_exact_one_radian_example,
    P.test_relative_position_property,
]


def _caught(lib) -> bool:
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    oracle.build(force=True, src=str(src), out=lib_path)
    lib = oracle.load(lib_path)
    assert _caught(lib), f"no pin caught the planted mistake: {name}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    src = tmp_path / "copy.c"
    shutil.copy(SRC, src)
    lib_path = str(tmp_path / "libcopy.so")
    oracle.build(force=True, src=str(src), out=lib_path)
    assert not _caught(oracle.load(lib_path))

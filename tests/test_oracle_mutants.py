"""The oracle pins must catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake (a flipped sign, a
wrong nibble or group index, a dropped term, a transposed operand, a wrong
rounding rule), builds the copy with gcc into a temporary directory, swaps it
in for the real oracle and checks that at least one pin of
``test_oracle_pins`` fails.  The mistake is planted in the oracle, on the CPU.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "w4a16_oracle.c")

MUTANTS = {
    "nibble_order_reversed": ("return (row_words[idx / 8] >> (4 * (idx % 8))) & 0xfu;",
                              "return (row_words[idx / 8] >> (4 * (7 - idx % 8))) & 0xfu;"),
    "sign_flipped": ("double w = (double)(qv - zv) * dec(s_row[g]);",
                     "double w = (double)(zv - qv) * dec(s_row[g]);"),
    "scale_group_ignored": ("double w = (double)(qv - zv) * dec(s_row[g]);",
                            "double w = (double)(qv - zv) * dec(s_row[0]);"),
    "zero_group_off_by_one": ("int zv = (int)nibble_at(z_row, g);",
                              "int zv = (int)nibble_at(z_row, g ? g - 1 : 0);"),
    "last_term_dropped": ("for (long k = 0; k < K; k++) {\n        long g = k / group;\n        int qv = (int)nibble_at(q_row, k);\n        int zv",
                          "for (long k = 0; k < K - 1; k++) {\n        long g = k / group;\n        int qv = (int)nibble_at(q_row, k);\n        int zv"),
    "operands_transposed": ("linear_one(j->x + m * (long)j->K, j->qweight + n * KW,",
                            "linear_one(j->x + (n % j->M) * (long)j->K, j->qweight + (m % j->N) * KW,"),
    "subnormal_exponent": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "ties_away_from_zero": ("if (frac > 0.5 || (frac == 0.5 && (m & 1u))) m++;\n    if (m == 0) return sign;\n    if (m < 1024)",
                            "if (frac >= 0.5) m++;\n    if (m == 0) return sign;\n    if (m < 1024)"),
    "silu_sign": ("out[(long)m * I + n] = g / (1.0 + exp(-g)) * u;",
                  "out[(long)m * I + n] = g / (1.0 + exp(g)) * u;"),
    "silu_halves_swapped": ("const double g = y[(long)m * 2 * I + n];\n            const double u = y[(long)m * 2 * I + I + n];",
                            "const double u = y[(long)m * 2 * I + n];\n            const double g = y[(long)m * 2 * I + I + n];"),
    "residual_dropped": ("out[i] = y[i] + dec(r[i]);", "out[i] = y[i];"),
    "transpose_order_inverted": ("const unsigned pos = (order >> (4 * (c % 8))) & 7u;",
                                 "unsigned pos = 0;\n            while (((order >> (4 * pos)) & 7u) != (unsigned)(c % 8) && pos < 7) ++pos;"),
    "transpose_dst_word_index": ("dst[c * dw + r / 8] |= (uint32_t)v << (4 * (r % 8));",
                                 "dst[c * dw + r / 8] |= (uint32_t)v << (4 * (7 - r % 8));"),
    "bf16_bias_off_by_one": ("v = ldexp((double)(128 + f), e - 134);", "v = ldexp((double)(128 + f), e - 133);"),
    "bf16_subnormal_exponent": ("v = ldexp((double)f, -133);", "v = ldexp((double)f, -132);"),
    "bf16_truncates": ("    if (frac > 0.5 || (frac == 0.5 && (m & 1u))) m++;\n    if (m == 0) return sign;\n    if (m < 128)",
                       "    if (m == 0) return sign;\n    if (m < 128)"),
    "bf16_read_as_half": ("return dtype == 1 ? w4o_bf16_to_double : w4o_half_to_double;",
                          "return w4o_half_to_double;"),
    "dense_transposed_weight": ("for (long k = 0; k < K; ++k) acc += dec(x[m * K + k]) * dec(w[n * K + k]);\n            y[m * N + n] = acc;",
                                "for (long k = 0; k < K; ++k) acc += dec(x[m * K + k]) * dec(w[(k % N) * K + n % K]);\n            y[m * N + n] = acc;"),
    "dense_last_term_dropped": ("for (long k = 0; k < K; ++k) acc += dec(x[m * K + k]) * dec(w[n * K + k]);\n            y[m * N + n] = acc;",
                                "for (long k = 0; k < K - 1; ++k) acc += dec(x[m * K + k]) * dec(w[n * K + k]);\n            y[m * N + n] = acc;"),
    "moe_align_unstable": ("    for (int s = 0; s < n_slots; ++s) {\n        const int p = fill[ids[s]]++;",
                           "    for (int s = n_slots - 1; s >= 0; --s) {\n        const int p = fill[ids[s]]++;"),
    "moe_token_of_slot": ("const long e = ids[s], m = per_slot ? s : s / k;",
                          "const long e = ids[s], m = per_slot ? s : s % T;"),
    "moe_expert_offset": ("const long row = e * N + n;", "const long row = n;"),
    "moe_sum_weight_index": ("acc += wts[t * k + j] * y[(t * k + j) * N + n];",
                             "acc += wts[t * k] * y[(t * k + j) * N + n];"),
    "pack_zero_pad_dirty": ("if (g < G) word |= (uint32_t)(z[n * G + g] & 0xfu) << (4 * j);",
                            "word |= (uint32_t)(z[n * G + (g < G ? g : G - 1)] & 0xfu) << (4 * j);"),
}


def _pin_calls():
    return [
        pins.test_half_to_double_every_pattern,
        pins.test_double_to_half_round_to_nearest_even,
        pins.test_double_to_half_ties_closed_form,
        pins.test_pack_closed_form_words,
        pins.test_pack_unpack_round_trip_every_nibble_everywhere,
        pins.test_unpack_pack_round_trip_random_words,
        pins.test_dequant_all_q_z_pairs_exact,
        pins.test_dequant_group_index,
        lambda: pins.test_linear_matches_exact_rationals(2, 3, 256, 128),
        lambda: pins.test_linear_matches_exact_rationals(2, 5, 384, 128),
        pins.test_q_equal_z_gives_zero,
        pins.test_single_nonzero_group_closed_form,
        pins.test_linearity_in_x,
        lambda: pins.test_integer_case_equals_int64_matmul(0x2C00, 1 / 16),
        pins.test_hand_worked_example,
        pins.test_silu_mul_closed_forms,
        pins.test_silu_mul_odd_part_identity,
        pins.test_silu_mul_column_split_and_rows,
        pins.test_add_residual_exact,
        pins.test_transpose_u4_hand_block,
        pins.test_transpose_u4_against_pinned_pack_unpack,
        pins.test_transpose_u4_ragged_rows_pad_with_zero,
        pins.test_transpose_u4_nibble_order,
        pins.test_bf16_to_double_every_pattern,
        pins.test_double_to_bf16_neighbours_and_ties,
        pins.test_double_to_bf16_closed_form,
        lambda: pins.test_linear_bf16_matches_exact_rationals(2, 3, 256),
        pins.test_linear_bf16_integer_case_equals_int64_matmul,
        pins.test_add_residual_bf16_exact,
        lambda: pins.test_dense_linear_matches_exact_rationals("f16"),
        lambda: pins.test_dense_linear_matches_exact_rationals("bf16"),
        pins.test_dense_linear_equals_the_4bit_linear_on_its_dequantised_weights,
        pins.test_dense_linear_integer_case_equals_int64_matmul,
        pins.test_moe_align_is_a_stable_sort_by_expert,
        pins.test_moe_linear_is_the_pinned_linear_of_each_slots_expert,
        pins.test_moe_sum_selects_and_is_exact,
    ]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(so), str(mutated), "-lm", "-lpthread"], check=True)
    real = oracle._load()
    oracle._lib = oracle._bind(ctypes.CDLL(str(so)))
    failed = []
    try:
        for call in _pin_calls():
            try:
                with np.errstate(all="ignore"):
                    call()
            except (AssertionError, ValueError, IndexError):
                failed.append(getattr(call, "__name__", "lambda"))
    finally:
        oracle._lib = real
    assert failed, f"no pin caught the planted mistake {name}"

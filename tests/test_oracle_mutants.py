"""Planted mistakes in the oracle must fail its pins (no GPU needed).

Each case copies the oracle's C source, plants one plausible slip -- a dropped
term, a flipped sign, a wrong block / slot / head index, a missing
normalisation, a wrong rounding -- builds the copy, and runs the pins of
test_oracle_pins.py against it.  At least one pin must fail for every mutant;
otherwise the pins would not be able to tell that mistake from the right answer.
The mistakes are planted on the CPU only, in a temporary copy.  The pins are those of
test_oracle_pins.py, test_oracle_fp8_pins.py and test_oracle_fp4_pins.py.
"""
import os

import pytest

import test_oracle_fp4_pins as fp4
import test_oracle_fp8_pins as fp8
import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
F32, BF16 = 0, 1

MUTANTS = {
    "no_max_subtraction": ("x[t] = exp(x[t] - xmax);", "x[t] = exp(x[t]);"),
    "score_sign": ("x[t] = scale * acc;", "x[t] = -scale * acc;"),
    "scale_dropped": ("x[t] = scale * acc;", "x[t] = acc;"),
    "no_normalisation": ("double p = x[t] / denom;", "double p = x[t];"),
    "context_short_by_one": ("    for (int t = 0; t < L; ++t) {\n        int64_t blk;\n        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);\n        if (rc != OR_OK) goto done;\n        for (int d",
                             "    for (int t = 0; t < L - 1; ++t) {\n        int64_t blk;\n        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);\n        if (rc != OR_OK) goto done;\n        for (int d"),
    "fp8_context_short_by_one": ("    for (int t = 0; t < L; ++t) {\n        int64_t blk;\n        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);\n        if (rc != OR_OK) goto done;\n        int slot",
                                 "    for (int t = 0; t < L - 1; ++t) {\n        int64_t blk;\n        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);\n        if (rc != OR_OK) goto done;\n        int slot"),
    "wrong_slot": ("size_t e = pool_elem(blk, g, t % ORACLE_BLOCK, d, Hkv, D, X);",
                   "size_t e = pool_elem(blk, g, (t + 1) % ORACLE_BLOCK, d, Hkv, D, X);"),
    "wrong_block": ("int32_t b = tables[(size_t)s * (size_t)max_blocks + (size_t)lb];",
                    "int32_t b = tables[(size_t)s * (size_t)max_blocks];"),
    "gqa_modulo_map": ("int X = 16 / elem_bytes_of(dtype);\n    int g = h / (Hq / Hkv);",
                       "int X = 16 / elem_bytes_of(dtype);\n    int g = h % Hkv;"),
    "fp8_gqa_modulo_map": ("D % 16 != 0 || Hq <= 0 || Hq % Hkv != 0) return OR_BAD_ARG;\n    int g = h / (Hq / Hkv);",
                           "D % 16 != 0 || Hq <= 0 || Hq % Hkv != 0) return OR_BAD_ARG;\n    int g = h % Hkv;"),
    "query_of_wrong_head": ("qv[d] = load_elem(q, ((size_t)s * Hq + h) * (size_t)D + d, dtype);",
                            "qv[d] = load_elem(q, ((size_t)s * Hq + g) * (size_t)D + d, dtype);"),
    "round_down": ("double r = rint(m / ulp) * ulp;\n    if (r >= ldexp(1.0, 128))",
                   "double r = floor(m / ulp) * ulp;\n    if (r >= ldexp(1.0, 128))"),
    "no_subnormal_spacing": ("    if (ex < -126) ex = -126;     /* subnormal range keeps the fixed spacing */\n", ""),
    "widen_shift": ("uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;"),
    "append_wrong_slot": ("size_t dst = pool_elem(blk, h, p % ORACLE_BLOCK, d, Hkv, D, X);",
                          "size_t dst = pool_elem(blk, h, (p + 1) % ORACLE_BLOCK, d, Hkv, D, X);"),
    "append_first_row_only": ("size_t row = (size_t)(cu_new[s] + i);\n            for (int h = 0; h < Hkv; ++h) {\n                for (int d",
                              "size_t row = (size_t)(cu_new[s]);\n            for (int h = 0; h < Hkv; ++h) {\n                for (int d"),
    "e4m3_round_down": ("    double r = rint(m / ulp) * ulp;\n    if (r > 448.0) r = 448.0;",
                        "    double r = floor(m / ulp) * ulp;\n    if (r > 448.0) r = 448.0;"),
    "e4m3_no_saturation": ("    if (r > 448.0) r = 448.0;\n", ""),
    "e4m3_exponent_bias": ("int E = re - 1 + 7;", "int E = re - 1 + 8;"),
    "fp8_scale_not_applied": ("Kc[(size_t)t * D + d] = oracle_e4m3_to_double(krec[((size_t)(d / 16) * 16 + slot) * 16 + d % 16]) * ks;",
                              "Kc[(size_t)t * D + d] = oracle_e4m3_to_double(krec[((size_t)(d / 16) * 16 + slot) * 16 + d % 16]);"),
    "fp8_v_layout_untransposed": ("for (int d = 0; d < D; ++d) vrec[(size_t)d * 16 + t] = codes[d];",
                                  "for (int d = 0; d < D; ++d) vrec[((size_t)(d / 16) * 16 + t) * 16 + d % 16] = codes[d];"),
    "fp8_scale_from_first_value": ("        if (f > amax) amax = f;\n", "        if (d == 0) amax = f;\n"),
    "e2m1_round_down": ("double r = rint(m / ulp) * ulp;                /* half-way cases to the even multiple */",
                        "double r = floor(m / ulp) * ulp;               /* half-way cases to the even multiple */"),
    "e2m1_no_saturation": ("    if (r > 6.0) r = 6.0;\n", ""),
    "e2m1_exponent_bias": ("int E = re;                                /* bias 1", "int E = re - 1;                            /* bias 1"),
    "mx_scale_emax_3": ("int code = 127 + (e - 1) - 2;", "int code = 127 + (e - 1) - 3;"),
    "mx_scale_from_first_block": ("for (int d = 32 * b; d < 32 * b + 32; ++d) {\n            double v = fabs",
                                  "for (int d = 0; d < 32; ++d) {\n            double v = fabs"),
    "fp4_k_nibbles_swapped": ("put_nibble(krec, fp4_k_byte(t, d, D), d & 1, codes[d]);",
                              "put_nibble(krec, fp4_k_byte(t, d, D), !(d & 1), codes[d]);"),
    "fp4_v_untransposed": ("put_nibble(vrec, fp4_v_byte(t, d, D), t & 1, codes[d]);",
                           "put_nibble(vrec, fp4_k_byte(t, d, D), d & 1, codes[d]);"),
    "fp4_scale_not_applied": ("return ldexp(oracle_e2m1_to_double(code), (int)sc - 127);",
                              "return oracle_e2m1_to_double(code);"),
    "fp4_context_short_by_one": ("    for (int t = 0; t < L; ++t) {\n        int64_t blk;\n        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);\n        if (rc != OR_OK) goto done;\n        int t16",
                                 "    for (int t = 0; t < L - 1; ++t) {\n        int64_t blk;\n        rc = lookup_block(tables, max_blocks, s, t, num_blocks, &blk);\n        if (rc != OR_OK) goto done;\n        int t16"),
    "fp4_gqa_modulo_map": ("D % 32 != 0 || Hq <= 0 || Hq % Hkv != 0) return OR_BAD_ARG;\n    int g = h / (Hq / Hkv);",
                           "D % 32 != 0 || Hq <= 0 || Hq % Hkv != 0) return OR_BAD_ARG;\n    int g = h % Hkv;"),
    "copy_keys_only": ("        memmove((char*)v_pool + (size_t)dst * block_bytes, (char*)v_pool + (size_t)src * block_bytes, block_bytes);\n", ""),
}


def _pins():
    yield "bf16_cases", lambda o: pins.test_bf16_rounding_hand_worked_cases(o)
    yield "bf16_torch", lambda o: pins.test_bf16_rounding_matches_torch_on_fp32_values(o)
    yield "bf16_widen", lambda o: pins.test_bf16_widening_is_exact(o)
    for dt in (F32, BF16):
        yield f"single_token_{dt}", lambda o, dt=dt: pins.test_single_token_context_returns_its_value_row(o, dt)
        yield f"zero_query_{dt}", lambda o, dt=dt: pins.test_zero_query_gives_mean_of_values(o, dt)
        yield f"paged_contig_{dt}", lambda o, dt=dt: pins.test_paged_equals_contiguous_and_batched_equals_alone(o, dt)
    yield "two_token", lambda o: pins.test_two_token_closed_form(o)
    for hot in (0, 37):
        yield f"dominant_{hot}", lambda o, hot=hot: pins.test_dominant_key_selects_its_value(o, hot)
    yield "positions", lambda o: pins.test_positions_reach_the_right_block_and_slot(o)
    yield "gqa", lambda o: pins.test_gqa_query_head_reads_kv_head_h_div_group(o)
    yield "zero_len", lambda o: pins.test_zero_length_context_is_zero(o)
    yield "large_scores", lambda o: pins.test_large_scores_do_not_overflow(o)
    yield "sdpa", lambda o: pins.test_matches_torch_sdpa_on_contiguous_rows(o, BF16, 14, 2, 64)
    yield "append", lambda o: pins.test_append_writes_only_its_slots_and_reads_back(o)
    yield "append_bad", lambda o: pins.test_append_rejects_bad_block_and_position(o)
    yield "copy", lambda o: pins.test_copy_block_copies_every_byte_of_both_pools(o)
    yield "e4m3_cases", lambda o: fp8.test_e4m3_hand_worked_cases(o)
    yield "e4m3_torch", lambda o: fp8.test_e4m3_matches_torch_in_range(o)
    yield "e4m3_bijection", lambda o: fp8.test_e4m3_codes_and_values_are_a_bijection(o)
    yield "fp8_append", lambda o: fp8.test_quantised_append_scales_and_codes(o)
    yield "fp8_decode", lambda o: fp8.test_fp8_decode_closed_forms_and_library_routine(o)
    yield "e2m1_table", lambda o: fp4.test_e2m1_value_table(o)
    yield "e2m1_cases", lambda o: fp4.test_e2m1_hand_worked_cases(o)
    yield "e2m1_brute", lambda o: fp4.test_e2m1_matches_brute_force_nearest(o)
    yield "e2m1_bijection", lambda o: fp4.test_e2m1_codes_and_values_are_a_bijection(o)
    yield "mx_scale", lambda o: fp4.test_mx_scale_hand_worked_and_library(o)
    yield "fp4_append", lambda o: fp4.test_quantised_append_scales_values_and_error_bound(o)
    yield "fp4_layout", lambda o: fp4.test_record_layout_positions(o)
    yield "fp4_decode", lambda o: fp4.test_fp4_decode_closed_forms_and_library_routine(o)


def test_every_pin_passes_on_the_unmutated_source(oracle_mod, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "pa_oracle.c")).read()
    path = tmp_path / "same.c"
    path.write_text(src)
    so = oracle_mod.compile_source(str(path), str(tmp_path / "same.so"))
    with oracle_mod.use_library(so):
        for name, pin in _pins():
            pin(oracle_mod)


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(oracle_mod, tmp_path, mutant):
    old, new = MUTANTS[mutant]
    src = open(os.path.join(ROOT, "oracle", "pa_oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {mutant} not found exactly once"
    path = tmp_path / f"{mutant}.c"
    path.write_text(src.replace(old, new))
    so = oracle_mod.compile_source(str(path), str(tmp_path / f"{mutant}.so"))
    caught = []
    with oracle_mod.use_library(so):
        for name, pin in _pins():
            try:
                pin(oracle_mod)
            except (AssertionError, ValueError):
                caught.append(name)
    assert caught, f"no pin fails when the oracle has the mistake '{mutant}'"

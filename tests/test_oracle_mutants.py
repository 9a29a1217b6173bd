"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign or index, a transposed operand, a wrong rounding rule),
compiles it on the CPU, swaps it in, and checks that at least one pin fails.
The committed oracle is untouched.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
import oracle.oracle as OM
import test_oracle_codecs as C
import test_oracle_fused as Fz

SRC = os.path.join(os.path.dirname(OM.__file__), "ar_oracle.c")

MUTANTS = {
    "drop_residual": ("dec_d(dtype, a) + dec_d(dtype, residual_in[t * H + h]));\n            if (residual_out)",
                      "dec_d(dtype, a) + 0.0f);\n            if (residual_out)"),
    "skip_last_rank": ("for (int r = 1; r < R; ++r) {\n        s = s + dec_d(dtype, p[(int64_t)r * stride]);",
                       "for (int r = 1; r < R - 1; ++r) {\n        s = s + dec_d(dtype, p[(int64_t)r * stride]);"),
    "subtract_rank": ("s = s + dec_d(dtype, p[(int64_t)r * stride]);", "s = s - dec_d(dtype, p[(int64_t)r * stride]);"),
    "no_sum_rounding": ("uint16_t y = rnd_d(dtype, dec_d(dtype, a) + dec_d(dtype, residual_in[t * H + h]));\n            if (residual_out)",
                        "uint16_t y = rnd_d(dtype, s + dec_d(dtype, residual_in[t * H + h])); (void)a;\n            if (residual_out)"),
    "fp64_rank_sum": ("    float s = dec_d(dtype, p[0]);\n    for (int r = 1; r < R; ++r) {\n        s = s + dec_d(dtype, p[(int64_t)r * stride]);\n        if (acc)\n            s = dec_d(dtype, rnd_d(dtype, s));\n    }\n    return s;",
                      "    double s = dec_d(dtype, p[0]);\n    for (int r = 1; r < R; ++r) {\n        s = s + dec_d(dtype, p[(int64_t)r * stride]);\n        if (acc)\n            s = dec_d(dtype, rnd_d(dtype, (float)s));\n    }\n    return (float)s;"),
    "acc_rounding_dropped": ("        if (acc)\n            s = dec_d(dtype, rnd_d(dtype, s));", "        if (0)\n            s = dec_d(dtype, rnd_d(dtype, s));"),
    "acc_rounding_always": ("        if (acc)\n            s = dec_d(dtype, rnd_d(dtype, s));", "        if (1)\n            s = dec_d(dtype, rnd_d(dtype, s));"),
    "mean_over_H_minus_1": ("float ms = ss32 / (float)H;", "float ms = ss32 / (float)(H - 1);", 0),
    "eps_dropped": ("float v = ms + eps;", "float v = ms;", 0),
    "eps_outside_sqrt": ("float v = ms + eps;\n        float rstd = 1.0f / sqrtf(v);",
                         "float v = ms;\n        float rstd = 1.0f / (sqrtf(v) + eps);", 0),
    "gamma_reversed": ("float n = ny * dec_d(dtype, gamma[h]);", "float n = ny * dec_d(dtype, gamma[H - 1 - h]);"),
    "norm_uses_unrounded_sum": ("float ny = dec_d(dtype, y) * rstd;", "float ny = (dec_d(dtype, a) + dec_d(dtype, residual_in[t * H + h])) * rstd;"),
    "bf16_ties_away": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))",
                       "if (dropped >= 0x8000u)"),
    "f16_truncate": ("if (dropped > 0x1000u || (dropped == 0x1000u && (kept & 1u)))", "if (0)"),
    "e4m3_ties_away": ("if (frac > 0.5f || (frac == 0.5f && (n & 1u)))\n        n += 1u;\n    if (e == -6",
                       "if (frac >= 0.5f)\n        n += 1u;\n    if (e == -6"),
    "e4m3_no_subnormal": ("e = -6;                                       /* subnormal band: step 2^-9 */",
                          "e = -7;"),
    "e4m3_saturate_low": ("return s | 0x7e;\n    int e;", "return s | 0x7d;\n    int e;"),
    "e2m1_ties_away": ("if (frac > 0.5f || (frac == 0.5f && (n & 1u)))\n        n += 1u;\n    if (ax < 1.0f && n < 2u)",
                       "if (frac >= 0.5f)\n        n += 1u;\n    if (ax < 1.0f && n < 2u)"),
    "e2m1_saturate_low": ("return s | 0x7;\n    int e;", "return s | 0x6;\n    int e;"),
    "nvfp4_no_div6": ("float per_block = bmax / 6.0f;", "float per_block = bmax;", 0),
    "nvfp4_nibbles_swapped": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))", 0),
    "nvfp4_enc_inverted": ("float enc = (dec == 0.0f) ? 0.0f : gs / dec;", "float enc = (dec == 0.0f) ? 0.0f : dec / gs;", 0),
    "fp8_scale_not_inverted": ("return 1.0f / scale;", "return scale;"),
    "flip_wrong_word": ("if (words[i] == 0x80000000u)", "if (words[i] == 0x00008000u)"),
    "sum_without_rounding": ("out[i] = rnd_d(dtype, rank_sum(dtype, acc, in + i, rank_stride, R));",
                             "out[i] = (uint16_t)rank_sum(dtype, acc, in + i, rank_stride, R);"),
    "lamport_clear_wrong_slot": ("io[3] = (flag + 2) % 3;", "io[3] = (flag + 1) % 3;"),
    # fp32 element type
    "f32_drop_residual": ("float y = s + residual_in[t * H + h];\n            if (residual_out)",
                          "float y = s + 0.0f;\n            if (residual_out)"),
    "f32_skip_last_rank": ("for (int r = 1; r < R; ++r)\n                s = s + partials[",
                           "for (int r = 1; r < R - 1; ++r)\n                s = s + partials[", 0),
    "f32_norm_skips_last_rank": ("for (int r = 1; r < R; ++r)\n                s = s + partials[",
                                 "for (int r = 1; r < R - 1; ++r)\n                s = s + partials[", 1),
    "f32_fp64_rank_sum": ("            float s = partials[t * H + h];\n            for (int r = 1; r < R; ++r)",
                          "            double s = partials[t * H + h];\n            for (int r = 1; r < R; ++r)", 0),
    "f32_mean_over_H_minus_1": ("float ms = ss32 / (float)H;", "float ms = ss32 / (float)(H - 1);", 1),
    "f32_eps_dropped": ("float v = ms + eps;", "float v = ms;", 1),
    "f32_eps_outside_sqrt": ("float v = ms + eps;\n        float rstd = 1.0f / sqrtf(v);",
                             "float v = ms;\n        float rstd = 1.0f / (sqrtf(v) + eps);", 1),
    "f32_gamma_reversed": ("norm_out[t * H + h] = ny * gamma[h];", "norm_out[t * H + h] = ny * gamma[H - 1 - h];"),
    "f32_amax_no_abs": ("m = fmaxf(m, fabsf(x[i]));", "m = fmaxf(m, x[i]);"),
    "f32_fp8_scale_ignored": ("q[i] = oracle_f32_to_e4m3(n_in[i] * inv_scale);", "q[i] = oracle_f32_to_e4m3(n_in[i]);"),
    "f32_nvfp4_no_div6": ("float per_block = bmax / 6.0f;", "float per_block = bmax;", 1),
    "f32_nvfp4_nibbles_swapped": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))", 1),
    "f32_nvfp4_enc_inverted": ("float enc = (dec == 0.0f) ? 0.0f : gs / dec;",
                               "float enc = (dec == 0.0f) ? 0.0f : dec / gs;", 1),
    "f32_sum_subtract": ("s = s + in[(int64_t)r * rank_stride + i];", "s = s - in[(int64_t)r * rank_stride + i];"),
    "buffer_size_missing_R": ("out[0] = (int64_t)R * max_tokens * H * elem_bytes;", "out[0] = max_tokens * H * elem_bytes;"),
    "f16_subnormal_decode_scale": ("mag = (float)m * 0x1p-24f;", "mag = (float)m * 0x1p-25f;"),
    "e4m3_decode_bias": ("mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);",
                         "mag = ldexpf(1.0f + (float)m / 8.0f, e - 8);"),
    "amax_no_abs": ("m = fmaxf(m, fabsf(dec_d(dtype, x[i])));", "m = fmaxf(m, dec_d(dtype, x[i]));"),
    "nvfp4_block_max_no_abs": ("bmax = fmaxf(bmax, fabsf(dec_d(dtype, blk[i])));",
                               "bmax = fmaxf(bmax, dec_d(dtype, blk[i]));"),
    "sum_of_abs_not_squares": ("ss += yd * yd;", "ss += fabs(yd);"),
    "swizzle_row_major_inside_tile": ("int64_t within = (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4;",
                                      "int64_t within = (m % 32) * 4 + ((m / 32) % 4) * 128 + k % 4;"),
    "norm_gamma_before_rstd": ("float ny = dec_d(dtype, y) * rstd;\n            float n = ny * dec_d(dtype, gamma[h]);",
                               "float ny = dec_d(dtype, y) * dec_d(dtype, gamma[h]);\n            float n = ny * rstd;"),
    "mean_in_fp64": ("float ms = ss32 / (float)H;", "float ms = (float)(ss / (double)H);", 0),
    "mean_by_reciprocal": ("float ms = ss32 / (float)H;", "float ms = ss32 * (1.0f / (float)H);", 0),
    "nvfp4_enc_unrounded_scale": ("float enc = (dec == 0.0f) ? 0.0f : gs / dec;",
                                  "float enc = (dec == 0.0f) ? 0.0f : 6.0f / bmax;", 0),
    "f32_norm_gamma_before_rstd": ("float ny = y * rstd;\n            norm_out[t * H + h] = ny * gamma[h];",
                                   "float ny = y * gamma[h];\n            norm_out[t * H + h] = ny * rstd;"),
    "f32_mean_in_fp64": ("float ms = ss32 / (float)H;", "float ms = (float)(ss / (double)H);", 1),
    "f32_mean_by_reciprocal": ("float ms = ss32 / (float)H;", "float ms = ss32 * (1.0f / (float)H);", 1),
    "nvfp4_global_scale_448": ("return 2688.0f / amax;", "return 448.0f / amax;"),
    "nvfp4_sf_index_transposed": ("scale_out[t * (H / 16) + b] = sf;",
                                  "scale_out[(b * T + t) % (T * (H / 16))] = sf;", 0),
    "nvfp4_block_max_of_8": ("for (int i = 0; i < 16; ++i)\n                bmax = fmaxf(bmax, fabsf(dec_d(dtype, blk[i])));",
                             "for (int i = 0; i < 8; ++i)\n                bmax = fmaxf(bmax, fabsf(dec_d(dtype, blk[i])));"),
    "fp8_divides_by_inverse_scale": ("q[i] = oracle_f32_to_e4m3(dec_d(dtype, n_in[i]) * inv_scale);",
                                     "q[i] = oracle_f32_to_e4m3(dec_d(dtype, n_in[i]) / inv_scale);"),
    "flip_any_negative_zero_half": ("if (words[i] == 0x80000000u)",
                                    "if ((words[i] & 0xffffu) == 0x8000u || (words[i] >> 16) == 0x8000u)"),
    "fp8_inv_scale_one_division": ("return 1.0f / scale;", "return 448.0f / amax;"),
    "e4m3_binade_carry_missing": ("if (n == 16u) { n = 8u; e += 1; }", "if (n == 16u) { n = 15u; }"),
    "e2m1_binade_carry_missing": ("if (n == 4u) { n = 2u; e += 1; }", "if (n == 4u) { n = 3u; }"),
    "e4m3_sign_of_zero_lost": ("uint8_t s = (uint8_t)((f2u(x) >> 24) & 0x80u);",
                               "uint8_t s = (uint8_t)(x < 0.0f ? 0x80u : 0u);"),
    "lamport_clear_size_missing_R": ("io[1] = (int64_t)R * T * H;", "io[1] = (int64_t)T * H;"),
    "slot_ignores_oneshot_floor": ("int64_t tok = max_tokens > oneshot_max ? max_tokens : oneshot_max;",
                                   "int64_t tok = max_tokens;"),
    "flag_bytes_without_R": ("out[1] = (int64_t)R * flag_count * 4;", "out[1] = flag_count * 4;"),
    "two_lamport_slots": ("out[3] = 3 * out[2];", "out[3] = 2 * out[2];"),
    "lamport_reads_wrong_slot": ("io[2] = flag % 3;", "io[2] = (flag + 1) % 3;"),
    "f32_sf_index_transposed": ("scale_out[t * (H / 16) + b] = sf;",
                                "scale_out[(b * T + t) % (T * (H / 16))] = sf;", 1),
    "swizzle_tiles_column_major": ("int64_t tile = (m / 128) * ktiles + k / 4;",
                                   "int64_t tile = (k / 4) * ((T + 127) / 128) + m / 128;"),
}

PINS = [
    C.test_bf16_round_matches_torch, C.test_f16_round_matches_numpy,
    C.test_bf16_decode_matches_torch, C.test_f16_decode_matches_numpy,
    C.test_e4m3_decode_facts, C.test_e4m3_decode_matches_torch, C.test_e2m1_decode_table,
    C.test_e4m3_encode_matches_torch_below_saturation, C.test_e4m3_saturates_and_keeps_nan,
    C.test_e4m3_ties_to_even_examples,
    C.test_e2m1_encode_brute_force, C.test_e2m1_ties_to_even_examples,
    lambda: C.test_e2m1_saturation_and_sign(100.0, 0x7),
    lambda: [Fz.test_identical_partials_sum_equals_R_times_x(R) for R in (2, 3, 8)],
    Fz.test_zero_partials_leave_residual_unchanged_and_norm_is_textbook,
    lambda: Fz.test_single_rank_is_textbook_residual_rmsnorm(oracle.BF16),
    Fz.test_rank_order_fp32_accumulation_worked_value,
    Fz.test_rank_sum_is_rounded_before_residual_add_worked_value,
    lambda: Fz.test_constant_power_of_two_row_normalises_to_signed_gamma_exactly(512, -0.25),
    Fz.test_constant_row_with_eps_closed_form,
    Fz.test_exact_rational_brute_force_tiny,
    Fz.test_norm_invariant_locates_eps_and_mean,
    lambda: Fz.test_rows_follow_the_pages_rounding_order_exactly(oracle.FP16),
    Fz.test_normalisation_multiplies_rstd_before_gamma,
    Fz.test_lamport_flip_only_touches_negative_zero_words,
    Fz.test_fp8_amax_element_maps_to_448_and_roundtrip_bound,
    Fz.test_fp8_multiplier_is_the_reciprocal_of_the_rounded_scale,
    lambda: Fz.test_amax_is_the_largest_magnitude_on_either_side(oracle.BF16),
    Fz.test_nvfp4_zero_block_and_max_element,
    lambda: Fz.test_nvfp4_global_scale_puts_the_amax_block_on_the_largest_scale(oracle.BF16),
    Fz.test_nvfp4_nibble_order_convention,
    Fz.test_nvfp4_roundtrip_bound_random,
    Fz.test_vector_sum_closed_form_and_fp64,
    Fz.test_element_type_accumulation_worked_value,
    lambda: Fz.test_element_type_accumulation_is_chained_library_adds(oracle.BF16),
    Fz.test_vector_sum_element_type_accumulation,
    lambda: Fz.test_vector_sum_element_type_special_values_are_chained_library_adds(oracle.FP16),
    Fz.test_scales_of_an_all_zero_tensor_are_finite,
    Fz.test_swizzled_scales_worked_positions,
    lambda: [Fz.test_swizzled_scales_are_a_tile_permutation(T, KB)
             for T, KB in ((128, 4), (257, 448), (300, 5))],
    Fz.test_workspace_sizes_match_page_formula_golden,
    Fz.test_lamport_state_cycles,
    lambda: [Fz.test_f32_identical_partials_power_of_two_ranks(R) for R in (2, 8)],
    Fz.test_f32_zero_partials_and_textbook_rmsnorm,
    Fz.test_f32_rank_order_worked_value,
    Fz.test_f32_constant_power_of_two_row,
    Fz.test_f32_constant_row_with_eps_closed_form,
    Fz.test_f32_norm_is_rmsnorm_of_residual_out,
    Fz.test_f32_rows_follow_the_pages_rounding_order_exactly,
    Fz.test_f32_quantisers_match_the_16_bit_ones_on_representable_values,
    Fz.test_f32_vector_sum,
]


def _build_mutant(tmp_path, name):
    src = open(SRC).read()
    old, new, *which = MUTANTS[name]
    if which:
        # the k-th of several identical lines (the 16-bit function comes first,
        # its fp32 counterpart second)
        k = which[0]
        assert src.count(old) > k, f"mutation anchor for {name} has no occurrence {k}"
        at = -1
        for _ in range(k + 1):
            at = src.index(old, at + 1)
        src = src[:at] + new + src[at + len(old):]
    else:
        assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
        src = src.replace(old, new)
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", str(path), "-o", str(so), "-lm"])
    return OM.load_library(str(so))


def test_pins_pass_on_committed_oracle():
    for pin in PINS:
        pin()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    mutant = _build_mutant(tmp_path, name)
    monkeypatch.setattr(OM, "_lib", mutant)
    caught = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught.append(getattr(pin, "__name__", "lambda"))
    assert caught, f"no pin caught mutant {name}"


def test_pins_catch_a_dropped_row_in_the_thread_split(monkeypatch):
    # the Python layer splits rows (elements) over threads; a split that
    # loses the last row of a span must fail a pin
    orig = OM._chunks

    def drop_last(n, parts):
        spans = orig(n, parts)
        if spans and spans[-1][1] > spans[-1][0]:
            spans[-1] = (spans[-1][0], spans[-1][1] - 1)
        return spans

    monkeypatch.setattr(OM, "_chunks", drop_last)
    caught = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin)
    assert caught


def test_results_do_not_depend_on_the_thread_count():
    from allreduce_residual_rmsnorm_gb300 import workloads as W
    w = W.FusedWorkload("threads", R=3, T=37, H=1024, pattern=W.RES_NORM_NVFP4, heavy_frac=0.01)
    inp = W.make_fused_inputs(w)
    args = (oracle.BF16, W.bits(inp.partials), W.bits(inp.residual), W.bits(inp.gamma), w.eps)
    ref = oracle.fused(*args, threads=1)
    for k in (2, 5, 16):
        got = oracle.fused(*args, threads=k)
        assert all(np.array_equal(a, b) for a, b in zip(ref, got)), k
    x = W.make_sum_inputs(W.SumWorkload("s", R=4, N=10_007))
    s1 = oracle.vector_sum(oracle.FP16, W.bits(x), threads=1)
    assert np.array_equal(s1, oracle.vector_sum(oracle.FP16, W.bits(x), threads=7))

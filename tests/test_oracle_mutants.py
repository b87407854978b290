"""The oracle's pins must catch plausible mistakes.

Each case compiles a copy of ``oracle/oracle.c`` with one planted mistake
(a dropped term, a wrong sign, a wrong index or bias, a swapped operand)
into a temporary directory, points the oracle module at it, and requires
at least one pin of ``test_oracle_pins`` to fail.  Only the CPU runs here.
"""
import os
import subprocess

import pytest

import oracle
import tests.test_oracle_append as apins
import tests.test_oracle_pins as pins
import tests.test_oracle_sparse as spins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "nibble_order_swapped": ("(d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xf)",
                             "(d & 1) ? (uint8_t)(byte & 0xf) : (uint8_t)(byte >> 4)"),
    "e4m3_bias_off_by_one": ("v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 9);"),
    "e2m1_mantissa_dropped": ("ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0, e - 1)"),
    "gqa_head_mapping_strided": ("int h = kvh * G + g, r = i * G + g;",
                                 "int h = g * c->num_kv_heads + kvh, r = i * G + g;"),
    "causal_offset_off_by_one": ("int lim = L - Q + 1 + i;", "int lim = L - Q + i;"),
    "softmax_sign_flipped": ("double w = exp(scores[(int64_t)r * tmax + t] - mx[r]);",
                             "double w = exp(mx[r] - scores[(int64_t)r * tmax + t]);"),
    "softmax_scale_dropped": ("scores[(int64_t)r * tmax + t] = J->scale * dot;",
                              "scores[(int64_t)r * tmax + t] = dot;"),
    "int8_scale_dropped": ("return code * s;", "return code;"),
    "nvfp4_global_scale_dropped": ("return prod * g;", "return prod;"),
    "slot_index_shifted": ("token_row(const oracle_cache *c, int which, const int32_t *tables, int32_t stride,\n"
                           "                     int b, int t, int head, float *out) {\n"
                           "  int32_t blk = tables[(int64_t)b * stride + t / c->block_size];",
                           "token_row(const oracle_cache *c, int which, const int32_t *tables, int32_t stride,\n"
                           "                     int b, int t, int head, float *out) {\n"
                           "  t = t ^ 1;\n"
                           "  int32_t blk = tables[(int64_t)b * stride + t / c->block_size];"),
    "lse_log_dropped": ("J->lse[o] = mx[r] + log(sum[r]);", "J->lse[o] = mx[r] + sum[r];"),
    "merge_weight_dropped": ("+= w * part_o[((int64_t)p * R + r) * D + d];",
                             "+= part_o[((int64_t)p * R + r) * D + d];"),
    "fp16_subnormal_exponent": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "fp8_global_scale_dropped": ("return e * g;", "return e;"),
    # quantise-on-write (KV append)
    "grid_ties_away_from_zero": ("return (lo & 1) ? lo + 1 : lo;", "return lo + 1;"),
    "int8_scale_divisor": ("float ratio = amax / 127.0f;", "float ratio = amax / 128.0f;"),
    "nvfp4_scale_denominator": ("float denom = g * 6.0f;", "float denom = g * 4.0f;"),
    "append_nibble_order": ("(uint8_t)(nib[0] | (nib[1] << 4))", "(uint8_t)(nib[1] | (nib[0] << 4))"),
    "fp8_append_sign_dropped": ("(uint8_t)(mag | ((y < 0.0f && mag != 0) ? 0x80 : 0))",
                                "(uint8_t)mag"),
    # the pages' incident: a padded row's K/V lands in another request's slot
    "padded_row_written": ("if (slot == -1) continue;", "if (slot == -1) slot = 0;"),
    "append_offset_reversed": ("int64_t row = (blk * H + h) * bs + off;",
                               "int64_t row = (blk * H + h) * bs + (bs - 1 - off);"),
    "int8_round_half_up": ("return fmod(f, 2.0) == 0.0 ? f : f + 1.0;", "return f + 1.0;"),
    # block-sparse decode
    "sparse_score_summed_over_heads": ("if (dot > sc[j]) sc[j] = dot;",
                                       "sc[j] = (sc[j] == -INFINITY ? 0.0 : sc[j]) + dot;"),
    "sparse_ties_to_higher_index": ("(best < 0 || sc[j] > sc[best])",
                                    "(best < 0 || sc[j] >= sc[best])"),
    "block_mean_over_full_block": ("m[d] /= (double)(hi - lo);", "m[d] /= (double)sb;"),
    "sparse_token_range_shifted": ("for (int t = j * sb; t < (j + 1) * sb && t < L; ++t) keep[t] = 1;",
                                   "for (int t = j * sb + 1; t <= (j + 1) * sb && t < L; ++t) keep[t] = 1;"),
}


def _checks():
    yield pins.test_fp16_decoder_exhaustive, ()
    yield pins.test_e4m3_decoder_exhaustive, ()
    yield pins.test_e2m1_decoder_table, ()
    for dt in ("bf16", "int8", "nvfp4", "fp8"):
        yield pins.test_gather_bit_exact_vs_numpy_decode, (dt,)
        for Q in (1, 3):
            yield pins.test_attention_matches_dense_brute_force, (dt, Q)
    yield pins.test_merge_ignores_empty_partials_and_handles_all_empty, ()
    yield pins.test_golden_closed_form_examples, ()
    yield apins.test_fp8_encoder_matches_torch_float8_over_all_bf16_in_range, ()
    yield apins.test_int8_scale_matches_numpy_float16_over_all_bf16_maxima, ()
    yield apins.test_e2m1_ties_saturation_and_signed_zero, ()
    yield apins.test_e4m3_ties_subnormals_saturation_and_sign, ()
    yield apins.test_int8_ties_round_half_even, ()
    for dt in ("bf16", "int8", "fp8", "nvfp4"):
        yield apins.test_append_matches_generator_encoders, (dt,)
        yield apins.test_padded_rows_write_nothing_bad_slots_counted, (dt,)
    yield apins.test_on_grid_values_round_trip, ()
    for dt in ("int8", "nvfp4"):
        yield spins.test_block_means_match_numpy_mean_of_gathered_keys, (dt,)
        yield spins.test_sparse_attention_matches_numpy_softmax_over_selected_tokens, (dt,)
    yield spins.test_select_matches_numpy_brute_force, ()
    yield spins.test_select_ties_go_to_the_lower_index, ()
    yield spins.test_block_aligned_with_the_query_is_selected, ()
    yield spins.test_sparse_attention_with_every_block_equals_dense, ("int8",)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-pthread", str(c), "-o", str(so), "-lm"], check=True)
    oracle.use_library(str(so))
    caught = []
    try:
        for fn, args in _checks():
            try:
                fn(*args)
            except AssertionError:
                caught.append(fn.__name__)
                break
    finally:
        oracle.use_library(None)
    assert caught, f"no pin failed for planted mistake {name}"

"""Plant plausible mistakes in copies of the oracle and check the pins catch them.

Each mutant is the oracle's C source with one small textual change (a dropped
term, a wrong sign, a wrong index, a missing scale ...), compiled with gcc into
a temporary directory.  The committed oracle itself is never modified.  A
mutant that no pin rejects would mean the pins leave that part of the oracle
unchecked.
"""
import os

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sda_oracle.c")

MUTANTS = {
    # decode
    "drop_sink_term": ("double Z = exp(sink - M);", "double Z = 0.0;", pins.DECODE_PINS),
    "sink_times_scale": ("const double sink = (double)attn_sink[h];",
                         "const double sink = (double)attn_sink[h] * (double)softmax_scale;",
                         pins.DECODE_PINS),
    "missing_scale": ("x[j] = scale * dot;", "x[j] = dot;", pins.DECODE_PINS),
    "wrong_exp_sign": ("const double w = exp(x[j] - M) / Z;", "const double w = exp(M - x[j]) / Z;",
                       pins.DECODE_PINS),
    "reversed_value_row": ("o[d] += w * pool_value(pool, s, d, D);",
                           "o[d] += w * pool_value(pool, s, D - 1 - d, D);", pins.DECODE_PINS),
    "wrong_head_of_q": ("const uint16_t* qh = q + ((size_t)t * H + h) * D;",
                        "const uint16_t* qh = q + ((size_t)t * H + (H - 1 - h)) * D;",
                        pins.DECODE_PINS),
    "slice_off_by_one": ("const int32_t len = kv_indptr[t + 1] - begin;",
                         "const int32_t len = kv_indptr[t + 1] - begin - (kv_indptr[t + 1] > begin + 1);",
                         pins.DECODE_PINS),
    "max_ignores_logits": ("if (x[j] > M) M = x[j];", "(void)0;", pins.DECODE_PINS),
    # FP8 pool
    "e4m3_bias_8": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);",
                    "else v = ldexp(1.0 + (double)m / 8.0, e - 8);", pins.FP8_PINS),
    "e4m3_subnormal_scale": ("if (e == 0) v = ldexp((double)m / 8.0, -6);",
                             "if (e == 0) v = ldexp((double)m / 8.0, -7);", pins.FP8_PINS),
    "e4m3_mantissa_quarters": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);",
                               "else v = ldexp(1.0 + (double)m / 4.0, e - 7);", pins.FP8_PINS),
    "fp8_scale_ignored": ("return oracle_e4m3_to_double(p->fp8[(size_t)s * D + d]) * (double)p->scale[s];",
                          "return oracle_e4m3_to_double(p->fp8[(size_t)s * D + d]);", pins.FP8_PINS),
    "fp8_scale_of_wrong_row": ("return oracle_e4m3_to_double(p->fp8[(size_t)s * D + d]) * (double)p->scale[s];",
                               "return oracle_e4m3_to_double(p->fp8[(size_t)s * D + d]) * (double)p->scale[0];",
                               pins.FP8_PINS),
    # q/kv norm + RoPE + store
    "rms_drops_eps": ("sqrt(ss / D + (double)eps)", "sqrt(ss / D)", pins.STORE_PINS),
    "rms_sum_not_mean": ("sqrt(ss / D + (double)eps)", "sqrt(ss + (double)eps)", pins.STORE_PINS),
    "rms_wrong_weight": ("const uint16_t* w = r < H ? q_norm_w : kv_norm_w;",
                         "const uint16_t* w = q_norm_w;", pins.STORE_PINS),
    "rope_sign": ("y[d] = a * c - b * s;", "y[d] = a * c + b * s;", pins.STORE_PINS),
    "rope_leading_dims": ("const int d = D - R + 2 * i;", "const int d = 2 * i;", pins.STORE_PINS),
    "rope_neox_pairs": ("const double a = y[d], b = y[d + 1];\n        y[d] = a * c - b * s;\n        y[d + 1] = b * c + a * s;",
                        "const double a = y[D - R + i], b = y[D - R / 2 + i];\n        y[D - R + i] = a * c - b * s;\n        y[D - R / 2 + i] = b * c + a * s;",
                        pins.STORE_PINS),
    "rope_cos_sin_swapped": ("const double c = cos_cache[", "const double c = sin_cache[", pins.STORE_PINS),
    "rope_wrong_position": ("cos_cache[(size_t)pos * (R / 2) + i]", "cos_cache[(size_t)0 * (R / 2) + i]",
                            pins.STORE_PINS),
    "ring_without_mod": ("state_slot[t] * win + pos % win;", "state_slot[t] * win + pos;",
                         pins.STORE_PINS),
    "bf16_truncates": ("const double r = rint(a / quantum) * quantum;",
                       "const double r = trunc(a / quantum) * quantum;", pins.ROUNDING_PINS),
    "bf16_ties_away": ("const double r = rint(a / quantum) * quantum;",
                       "const double r = round(a / quantum) * quantum;", pins.ROUNDING_PINS),
    "e4m3_ties_away": ("double r = rint(a / quantum) * quantum;\n  if (r > 448.0)",
                       "double r = round(a / quantum) * quantum;\n  if (r > 448.0)", pins.ROUNDING_PINS),
    "e4m3_no_saturation": ("if (r > 448.0) r = 448.0;", "(void)0;", pins.ROUNDING_PINS),
    "e4m3_subnormal_binade": ("if (E < -6) E = -6;", "if (E < -7) E = -7;", pins.ROUNDING_PINS),
    "fp8_scale_floor": ("int e = (int)ceil(log2(amax / 448.0));\n  while (ldexp(448.0, e) < amax) ++e;",
                        "int e = (int)floor(log2(amax / 448.0));", pins.ROUNDING_PINS),
    "fp8_scale_one_too_big": ("while (ldexp(448.0, e - 1) >= amax) --e;\n  return e",
                              "while (ldexp(448.0, e - 1) >= amax) --e;\n  ++e;\n  return e",
                              pins.ROUNDING_PINS),
    # top-k -> slot lists
    "topk_ties_larger_position_first": ("return (x->pos > y->pos) - (x->pos < y->pos);",
                                        "return (x->pos < y->pos) - (x->pos > y->pos);",
                                        pins.TOPK_PINS),
    "topk_nan_ranks_first": ("if (isnan(f)) return 0;", "if (isnan(f)) return 0xFFFFFFFFu;",
                             pins.TOPK_PINS),
    "topk_minus_zero_below_zero": ("if (u == 0x80000000u) u = 0;", "(void)0;", pins.TOPK_PINS),
    "topk_smallest_scores": ("return x->key > y->key ? -1 : 1;", "return x->key > y->key ? 1 : -1;",
                             pins.TOPK_PINS),
    "topk_not_in_position_order": ("qsort(sel, (size_t)kk, sizeof(int32_t), int_order);", "(void)0;",
                                   pins.TOPK_PINS),
    "topk_block_slot_swapped": ("block_table[(size_t)t * bt_stride + p / k_per_block];",
                                "block_table[(size_t)t * bt_stride + p % k_per_block];",
                                pins.TOPK_PINS),
    "topk_reads_padding": ("int64_t n = lengths[t];", "int64_t n = score_stride;", pins.TOPK_PINS),
    "topk_bad_length_unflagged": ("flags |= 1;\n      n = 0;", "n = 0;", pins.TOPK_PINS),
    # builder
    "ring_newest_first": ("(int64_t)swa_head[t] - n_swa + 1 + j", "(int64_t)swa_head[t] - j",
                          pins.BUILDER_PINS),
    "no_swa_offset": ("kv_indices[pos++] = (int32_t)(swa_pages + (int64_t)comp_block[e]",
                      "kv_indices[pos++] = (int32_t)((int64_t)comp_block[e]", pins.BUILDER_PINS),
    "block_slot_swapped": ("(int64_t)comp_block[e] * k_per_block + comp_slot[e]);\n    }\n    kv_indptr",
                           "(int64_t)comp_slot[e] * k_per_block + comp_block[e]);\n    }\n    kv_indptr",
                           pins.BUILDER_PINS),
    "padded_not_empty": ("if (state_slot[t] < 0) continue;", "if (state_slot[t] < -1) continue;",
                         pins.BUILDER_PINS),
    "swa_head_unchecked": ("else if (n_swa > 0 && (swa_head[t] < 0 || swa_head[t] >= win)) bad |= 2;",
                           "else if (0) bad |= 2;", pins.BUILDER_PINS),
    "comp_indptr_decrease_unchecked": ("if (c0 < 0 || c1 < c0 || (int64_t)c1 > comp_total) bad |= 4;",
                                       "if (c0 < 0 || (int64_t)c1 > comp_total) bad |= 4;",
                                       pins.BUILDER_PINS),
    # validation
    "validate_off_by_one": ("(int64_t)kv_indices[e] >= total_pages) ++n_bad;",
                            "(int64_t)kv_indices[e] > total_pages) ++n_bad;", pins.VALIDATE_PINS),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new, pin_set = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    csrc = tmp_path / "mutant.c"
    csrc.write_text(mutated)
    so = oracle.build(force=True, src=str(csrc), dst=str(tmp_path / "libmutant.so"))
    lib = oracle.load(so)
    failed = pins.failing_pins(lib, pin_set)
    assert failed, f"no pin catches mutant {name}"


def test_unmutated_copy_passes(tmp_path):
    csrc = tmp_path / "copy.c"
    csrc.write_text(open(SRC).read())
    lib = oracle.load(oracle.build(force=True, src=str(csrc), dst=str(tmp_path / "libcopy.so")))
    assert pins.failing_pins(lib) == []

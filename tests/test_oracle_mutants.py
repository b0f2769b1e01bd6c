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

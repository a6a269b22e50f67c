"""The pins catch plausible slips: each mutant is a copy of the oracle source with one
planted mistake, compiled on the CPU into a temporary library; at least one pin must
fail for every mutant.  (Mistakes are planted only in these CPU copies.)"""
import os
import re

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "fd_oracle.c")

# (name, exact text in the oracle, replacement of its first occurrence).  Every mutant
# stays in bounds.
MUTANTS = [
    ("dropped_scale", "s[t] = dot * scale;", "s[t] = dot;"),
    ("wrong_exp_sign", "double p = exp(s[t] - m);", "double p = exp(m - s[t]);"),
    ("no_max_shift", "double p = exp(s[t] - m);", "double p = exp(s[t]);"),
    ("log2_lse", "lse[row] = m + log(l);", "lse[row] = m + log2(l);"),
    ("missing_normalisation", "for (int j = 0; j < d; ++j) o[j] /= l;", ";"),
    ("gqa_modulo_map", "const int g = h / G;", "const int g = h % Hkv;"),
    ("q_transposed", "double qj = fdo_load(q, dtype, row * d + j);",
     "double qj = fdo_load(q, dtype, ((int64_t)h * B + b) * d + j);"),
    ("dropped_last_key", "    for (int64_t t = 0; t < L; ++t) {\n      double p",
     "    for (int64_t t = 0; t + 1 < L; ++t) {\n      double p"),
    ("dropped_first_key", "    for (int64_t t = 0; t < L; ++t) {\n      double p",
     "    for (int64_t t = 1; t < L; ++t) {\n      double p"),
    ("page_id_from_logical_slot", "int64_t page = block_table[(int64_t)b * max_pages + t / page_size];",
     "int64_t page = (int64_t)b * max_pages + t / page_size;"),
    ("empty_row_fake_block", "lse[row] = -INFINITY;", "lse[row] = 0.0;"),
    ("v_reads_k", "o[j] += p * fdo_load(v, dtype,", "o[j] += p * fdo_load(k, dtype,"),
    # The multi-token (causal) oracle.
    ("causal_off_by_one", "const int64_t visible = (int64_t)seq_lens[b] - Q + 1 + j;",
     "const int64_t visible = (int64_t)seq_lens[b] - Q + j;"),
    ("causal_reversed", "const int64_t visible = (int64_t)seq_lens[b] - Q + 1 + j;",
     "const int64_t visible = (int64_t)seq_lens[b] - j;"),
    ("causal_token_index", "const int j = (int)((row / Hq) % Q);", "const int j = (int)(row % Q);"),
    # The FP8 decoder and the scaled decode.
    ("e4m3_bias", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3_subnormal", "mag = ldexp((double)m / 8.0, -6);", "mag = ldexp((double)m / 8.0, -7);"),
    ("kv8_v_scale_from_k", "const double ks = (double)k_scale[g], vs = (double)v_scale[g];",
     "const double ks = (double)k_scale[g], vs = (double)k_scale[g];"),
    ("causal_drops_scale", "      s[t] = dot * scale;\n    }\n    double m = s[0];\n    for (int64_t t = 1; t < visible;",
     "      s[t] = dot;\n    }\n    double m = s[0];\n    for (int64_t t = 1; t < visible;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, "mutation anchor not found: %r" % old
    src = tmp_path / ("mutant_%s.c" % name)
    src.write_text(text.replace(old, new, 1))   # the first occurrence: the single-token
                                                # oracle, unless the anchor is causal-only
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / ("libmutant_%s.so" % name)))
    lib = oracle.load_library(so)
    failed = oracle_pins.failing_pins(lib)
    assert failed, "mutant %s passed every pin" % name


def test_unmutated_oracle_passes_every_pin():
    assert oracle_pins.failing_pins(oracle.load_library()) == []

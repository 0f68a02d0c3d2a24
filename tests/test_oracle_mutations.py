"""The pins must catch plausible mistakes in the oracle.

Each case compiles a copy of oracle.c with one planted mistake (on the CPU,
into a temporary directory), swaps it in as the oracle, and checks that at
least one pin of tests/test_oracle_pins.py fails.
"""
import os
import subprocess
import sys

import pytest

import oracle
from oracle import build as obuild

MUTANTS = {
    # wrong grouped-query mapping: modulo instead of integer division
    "head_map": ("h / G, Hkv, bs, d, scale, &m,\n                         &l, o);",
                 "h % Hkv, Hkv, bs, d, scale, &m,\n                         &l, o);"),
    # context off by one: attends one token past the context (within the last block)
    "ctx_off_by_one": ("for (int t = t0; t < t1; ++t)", "for (int t = t0; t < t1 + (t1 % bs != 0); ++t)"),
    # scale dropped from the scores
    "no_scale": ("        x *= scale;\n        double w = exp(x - m);", "        double w = exp(x - m);"),
    # block offset wrong: next slot in the page
    "offset": ("static int64_t cache_index(int64_t block, int h, int off, int i, int Hkv, int bs, int d) {\n    return (((block * Hkv) + h) * (int64_t)bs + off) * d + i;",
               "static int64_t cache_index(int64_t block, int h, int off, int i, int Hkv, int bs, int d) {\n    return (((block * Hkv) + h) * (int64_t)bs + (off + 1) % bs) * d + i;"),
    # K and V swapped in the weighted sum
    "kv_swap": ("acc[i] += w * elem(v_cache,", "acc[i] += w * elem(k_cache,"),
    # causal rule excludes the query's own position
    "causal_exclusive": ("row, 0, p + 1, h / G", "row, 0, p, h / G"),
    # merge forgets the rescaling of partial sums
    "merge_no_rescale": ("L += w * l[j];", "L += l[j];"),
    # bf16 decoded as if it were fp16
    "dtype_swap": ("return dtype == ORACLE_BF16 ? bf16_bits_to_double(p[i]) : half_bits_to_double(p[i]);",
                   "return dtype == ORACLE_BF16 ? half_bits_to_double(p[i]) : half_bits_to_double(p[i]);"),
}

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert old in src, "mutation site moved: " + name
    mutant = tmp_path / ("oracle_%s.c" % name)
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / ("liboracle_%s.so" % name)
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-o", str(lib), str(mutant), "-lm"],
                   check=True)
    monkeypatch.setattr(oracle, "_lib", oracle._open(str(lib)))
    import test_oracle_pins as pins
    failures = 0
    cases = [
        lambda: pins.test_fp16_decode_matches_numpy_for_every_pattern(),
        lambda: pins.test_bf16_decode_matches_torch_for_every_pattern(),
        lambda: pins.test_dense_matches_torch_sdpa("bf16", 32, 8, 64, 40),
        lambda: pins.test_paged_decode_equals_dense_on_random_tables(17),
        lambda: pins.test_one_hot_selects_exactly_one_value_row("bf16", 16, 2, 64),
        lambda: pins.test_uniform_weights_give_the_mean_of_values(17),
        lambda: pins.test_two_token_logistic_weight_pins_the_scale(64),
        lambda: pins.test_split_ranges_merged_by_lse_equal_unsplit(0),
        lambda: pins.test_prefill_matches_sdpa_lower_right_causal(23, 17),
        lambda: pins.test_append_then_read_back_through_the_table(),
    ]
    for case in cases:
        try:
            case()
        except Exception:
            failures += 1
    assert failures >= 1, "no pin caught mutant " + name

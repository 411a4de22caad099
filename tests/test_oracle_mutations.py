"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies the oracle's C source, changes one expression into a
plausible mistake, builds the copy, and checks that at least one pin fails.
"""
import os
import shutil

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, planted mistake)
MUTATIONS = [
    ("causal_diagonal_excluded", "if (pos + 1 < n) n = pos + 1;\n    }\n    return n;",
     "if (pos < n) n = pos;\n    }\n    return n;"),
    ("new_tokens_at_suffix_start", "int32_t pos = pb->P + pb->S[b] - pb->T[b] + t;\n        if (pos + 1 < n) n = pos + 1;\n    }\n    return n;",
     "int32_t pos = pb->P + t;\n        if (pos + 1 < n) n = pos + 1;\n    }\n    return n;"),
    ("gqa_head_modulo", "int32_t hk = h / G;", "int32_t hk = h % pb->H_kv;"),
    ("scale_dropped", "s[j - lo] = pb->scale * acc;", "s[j - lo] = acc;"),
    ("page_offset_shifted", "(j % page)", "((j + 1) % page)"),
    ("lse_without_max", "lse[(int64_t)i * H_q + h] = m + log(l);",
     "lse[(int64_t)i * H_q + h] = log(l);"),
    ("merge_weight_dropped", "l = l * sa + lb * sb;", "l = l * sa + lb;"),
    ("fork_reuses_pages", "free_pages[next_free++]", "free_pages[i]"),
    ("v_used_as_k", "const uint16_t *kr = kv_row(pb->k,", "const uint16_t *kr = kv_row(pb->v,"),
    ("softmax_denominator_dropped", "dst[c] = o[c] / l;", "dst[c] = o[c];"),
    ("append_position_shifted", "int32_t j = prefix_len + suffix_lens[b] + t;",
     "int32_t j = prefix_len + suffix_lens[b] + t + 1;"),
    ("cow_copy_skipped", "if (partial) {\n            cow[2 * b] = prefix_pages[n_full];",
     "if (0) {\n            cow[2 * b] = prefix_pages[n_full];"),
    ("extend_floor_pages", "int64_t have = (len0 + page_size - 1) / page_size;",
     "int64_t have = len0 / page_size;"),
]


@pytest.mark.parametrize("name,orig,bad", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, orig, bad, tmp_path):
    text = open(SRC).read()
    assert text.count(orig) >= 1, f"mutation target for {name} not found"
    src = tmp_path / "oracle_mut.c"
    src.write_text(text.replace(orig, bad, 1))
    lib = oracle.load(oracle.build(str(src), str(tmp_path / "liboracle_mut.so")))
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, IndexError) as e:
            failures.append(pin.__name__)
    assert failures, f"planted mistake {name} passed every pin"

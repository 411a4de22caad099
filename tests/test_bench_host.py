"""The benchmark's work accounting against the oracle's visible-pair count (CPU only)."""
import numpy as np
import pytest

import bench
import oracle
from shared_prefix_fan_gb300.workloads import WORKLOADS, draw, small_spec


@pytest.mark.parametrize("name", ["tiny", "decode", "batching", "wide"])
def test_visible_pairs_match_oracle(name):
    w = draw(WORKLOADS[name])
    s = w.spec
    assert bench.visible_pairs(w) == oracle.count_pairs(s.prefix_len, w.suffix_lens, w.q_rows,
                                                        s.h_q, s.causal)


def test_noncausal_pairs():
    w = draw(small_spec(causal=False, q_rows=[3, 0, 5], suffix_lens=[1, 4, 9]))
    s = w.spec
    assert bench.visible_pairs(w) == oracle.count_pairs(s.prefix_len, w.suffix_lens, w.q_rows,
                                                        s.h_q, False)


def test_decode_bytes():
    w = draw(WORKLOADS["decode"])
    work = bench.algorithmic_work(w)
    assert work["kv_bytes"] == (32768 + 8 * 512) * 8 * 128 * 2 * 2
    assert work["flops"] == 4 * 128 * 64 * 8 * (32768 + 512)


def test_kernel_fingerprint_ignores_comments_only():
    """The ncu traffic stays attached to a kernel whose comments changed, and
    is dropped as soon as its code changes."""
    code = "int f(int a) {\n  return a + 1;  // add one\n}\n/* block\n comment */\n"
    assert bench.source_code_text(code) == bench.source_code_text(
        "int f(int a) { return a + 1; }  // other words\n")
    assert bench.source_code_text(code) != bench.source_code_text("int f(int a) { return a + 2; }")
    assert bench.source_code_text('asm("ld.global.v4.s32 {%0}, [%1];");') == \
        'asm("ld.global.v4.s32 {%0}, [%1];");'

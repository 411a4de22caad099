"""Consecutive fanout_attn calls whose suffix lengths grow between calls (decode
steps) on one stream: the library keeps the cached work plan when no key range
gains a 128-key tile and only re-uploads the moved range ends and causal
positions (fanout_plan_step describes that plan). Every step is checked
against the fp64 oracle on the same inputs and page table, through the C ABI."""
import dataclasses

import numpy as np
import pytest

import oracle
from shared_prefix_fan_gb300 import binding
from shared_prefix_fan_gb300.workloads import draw, small_spec
from tests.gpu_helpers import DevWorkload, compare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("q_rows", [[1, 1, 1, 1], [20, 20, 20, 20]], ids=["one_tile", "two_tiles"])
def test_decode_steps_match_oracle(q_rows):
    S0 = np.array([100, 90, 110, 100], dtype=np.int32)
    grows = [0, 1, 2, 7, 40]
    # pages for the longest step; every step reads its keys through that table
    spec = small_spec(h_q=64, h_kv=8, page_size=64, prefix_len=2048, q_rows=q_rows,
                      suffix_lens=[int(x) for x in S0 + max(grows)], permute_prefix=True,
                      permute_suffix=True, seed=77)
    w_max = draw(spec)
    dw = DevWorkload(w_max)
    s = spec
    prev = None
    for step, grow in enumerate(grows):
        S = S0 + grow
        w = dataclasses.replace(w_max, suffix_lens=S)
        if prev is not None:
            _, _, _, reused = binding.plan_step(prev, S, w.q_rows, s.prefix_len, s.h_q, s.h_kv,
                                                s.page_size, s.causal)
            assert reused == (grow < 40)   # +40 keys reach a new 128-key tile
        dw.w = w
        out, lse = dw.run()
        ref = oracle.attn(w.q, w.k_pool, w.v_pool, dw.table_host, s.prefix_len, S, w.q_rows,
                          s.h_q, s.h_kv, s.page_size, s.scale, s.causal)
        compare(out, lse, *ref, what=f"step {step} (+{grow})")
        prev = S

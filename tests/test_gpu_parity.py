"""GPU parity: fanout_attn (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element. Five workloads at full size (the two
largest checked on sampled rows the oracle computes one by one), a sweep of
small shapes spanning several tiles and ragged tails, and edge cases."""
import numpy as np
import pytest
import torch

import oracle
from shared_prefix_fan_gb300 import binding
from shared_prefix_fan_gb300.workloads import WORKLOADS, draw, small_spec
from tests.gpu_helpers import DevWorkload, compare, oracle_ref, sample_rows

pytestmark = pytest.mark.gpu


def test_wait_timeout_reports_and_context_survives():
    DevWorkload(draw(WORKLOADS["tiny"]))  # builds/loads the library
    assert binding.selftest_wait_timeout(20_000_000) == binding.ETIMEOUT
    assert binding.last_error() == binding.OK  # cleared
    w = draw(WORKLOADS["tiny"])
    out, lse = DevWorkload(w).run()
    compare(out, lse, *oracle_ref(w), what="tiny after timeout")


@pytest.mark.parametrize("name", ["tiny", "decode", "batching"])
def test_full_workload(name):
    w = draw(WORKLOADS[name])
    out, lse = DevWorkload(w).run()
    compare(out, lse, *oracle_ref(w), what=name)


def partial_unit_tokens(w):
    """Tokens of every unit of the plan the call runs that writes a partial
    (merged later), and the units themselves, planned for this device."""
    s = w.spec
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    units, _, _ = binding.plan(w.suffix_lens, w.q_rows, s.prefix_len, s.h_q, s.h_kv,
                               s.page_size, s.causal, sms)
    parts = units[units[:, 7] >= 0]
    toks = set()
    for u in parts:
        toks.update(range(int(u[2]), int(u[2] + u[3])))
    return parts, toks


@pytest.mark.parametrize("name,every", [("wide", 16), ("prefill", 64)])
def test_large_workload_sampled(name, every):
    """Full-size workloads on sampled tokens: every `every`-th token, each
    branch's first and last, and -- where only some tokens have partials (the
    long prefill's tail cuts, merged through the sparse key list) -- every
    token of every partial unit, so each merge path the plan takes is checked."""
    w = draw(WORKLOADS[name])
    rows = set(sample_rows(w, every).tolist())
    parts, part_toks = partial_unit_tokens(w)
    if len(part_toks) < w.total_rows:   # a sparse merge: cover all of it
        rows |= part_toks
    rows = np.array(sorted(rows), dtype=np.int32)
    for u in parts:   # every partial unit has sampled tokens
        assert ((rows >= u[2]) & (rows < u[2] + u[3])).any(), u
    out, lse = DevWorkload(w).run()
    ref_o, ref_l = oracle_ref(w, rows=rows)
    compare(out, lse, ref_o, ref_l, rows=rows, what=name)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()


SWEEP = [
    # (q_rows, suffix_lens, prefix, page, h_q, h_kv, causal)
    ([1], [1], 0, 16, 8, 8, True),
    ([2, 7], [9, 40], 32, 16, 8, 2, True),
    ([16, 33, 1], [100, 33, 500], 256, 64, 16, 2, True),
    ([33], [300], 0, 64, 4, 1, True),
    ([7, 7, 7, 7], [7, 90, 129, 128], 128, 32, 32, 4, True),
    ([5, 3], [17, 3], 16, 16, 8, 1, False),
    ([40, 0, 12], [600, 10, 12], 1024, 128, 64, 8, True),
    ([1] * 9, [200] * 9, 2048, 16, 64, 8, True),
    ([20, 20], [256, 256], 512, 64, 128, 1, True),   # G = 128: one token per tile
    ([3, 4], [0, 4], 64, 16, 8, 2, False),            # a branch with no private suffix
]


@pytest.mark.parametrize("case", range(len(SWEEP)))
def test_small_sweep(case):
    tq, sl, P, ps, hq, hkv, causal = SWEEP[case]
    spec = small_spec(h_q=hq, h_kv=hkv, page_size=ps, prefix_len=P, causal=causal,
                      q_rows=tq, suffix_lens=sl, permute_prefix=True, permute_suffix=True,
                      seed=100 + case)
    w = draw(spec)
    out, lse = DevWorkload(w).run()
    compare(out, lse, *oracle_ref(w), what=f"sweep {case}")


@pytest.mark.parametrize("splits", [1, 2, 3, 32])
def test_forced_splits(splits):
    spec = small_spec(h_q=16, h_kv=2, page_size=16, prefix_len=1024, q_rows=[3, 9, 1],
                      suffix_lens=[200, 45, 700], seed=55)
    w = draw(spec)
    dw = DevWorkload(w)
    ref = oracle_ref(w)
    try:
        binding.set_option(binding.OPT_SPLITS, splits)
        out, lse = dw.run()
    finally:
        binding.set_option(binding.OPT_SPLITS, 0)
    compare(out, lse, *ref, what=f"splits={splits}")


def test_bf16_output():
    w = draw(WORKLOADS["batching"])
    out, lse = DevWorkload(w).run(out_dtype="bf16")
    ref_o, ref_l = oracle_ref(w)
    # the oracle rounded to bf16 (round to nearest even) is what a perfect kernel writes
    ref_bf = torch.from_numpy(ref_o).float().to(torch.bfloat16).double().numpy()
    o = out.double().cpu().numpy()
    ulp = np.abs(ref_bf) * 2.0 ** -8 + 1e-30
    assert (np.abs(o - ref_bf) <= ulp + 2e-3).all()
    compare(out, lse, ref_o, ref_l, what="bf16 out")


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes(seed):
    """Seeded random problems (branch count, new tokens and private suffix per
    branch, prefix length, page size, GQA group, causal or not, page placement,
    output dtype) through the C ABI against the fp64 oracle: planner paths the
    fixed cases may not reach (ragged tails, a single branch, empty branches,
    G from 1 to 16, one- and two-query-tile units)."""
    rng = np.random.default_rng(9000 + seed)
    B = int(rng.integers(1, 7))
    ps = int(rng.choice([16, 32, 64, 128]))
    P = ps * int(rng.integers(0, 24))
    causal = bool(rng.integers(0, 2))
    T = rng.integers(0, 40, size=B)
    if T.sum() == 0:
        T[0] = 1
    S = T + rng.integers(0 if P else 1, 700, size=B)
    h_kv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    spec = small_spec(h_q=h_kv * G, h_kv=h_kv, page_size=ps, prefix_len=P, causal=causal,
                      q_rows=[int(x) for x in T], suffix_lens=[int(x) for x in S],
                      permute_prefix=bool(rng.integers(0, 2)), permute_suffix=True,
                      seed=9500 + seed)
    w = draw(spec)
    out_dtype = "bf16" if seed % 4 == 3 else "f32"
    out, lse = DevWorkload(w).run(out_dtype=out_dtype)
    ref_o, ref_l = oracle_ref(w)
    if out_dtype == "bf16":
        # a perfect kernel writes the oracle rounded to bf16 (half an ulp away)
        ref_bf = torch.from_numpy(ref_o).float().to(torch.bfloat16).double().numpy()
        o = out.double().cpu().numpy()
        assert (np.abs(o - ref_bf) <= np.abs(ref_bf) * 2.0 ** -8 + 2e-3).all(), f"seed {seed}"
        return
    compare(out, lse, ref_o, ref_l, what=f"random {seed}: B={B} T={T.tolist()} "
            f"S={S.tolist()} P={P} page={ps} G={G} H_kv={h_kv} causal={causal}")


@pytest.mark.parametrize("n_branches,prefix,page,h_q,h_kv,tmax,smax", [
    (200, 2048, 16, 16, 2, 4, 200),
    (1024, 512, 16, 8, 1, 1, 64),
], ids=["200_branches", "1024_branches"])
def test_many_branches(n_branches, prefix, page, h_q, h_kv, tmax, smax):
    """Fan-out to many sub-agents (up to fanout_kv_append's 1024 branches):
    hundreds of private suffix ranges per KV head, many units per CTA, a large
    merge index; every row against the fp64 oracle."""
    rng = np.random.default_rng(n_branches)
    T = rng.integers(1, tmax + 1, size=n_branches)
    S = T + rng.integers(0, smax, size=n_branches)
    spec = small_spec(h_q=h_q, h_kv=h_kv, page_size=page, prefix_len=prefix, causal=True,
                      q_rows=[int(x) for x in T], suffix_lens=[int(x) for x in S],
                      permute_prefix=True, permute_suffix=True, seed=n_branches + 7)
    w = draw(spec)
    out, lse = DevWorkload(w).run()
    compare(out, lse, *oracle_ref(w), what=f"{n_branches} branches")


def test_pools_beyond_4gb():
    """K/V pools of 7.9 GB each (60000 pages of 8 KV heads x 64 tokens) with
    the problem's pages scattered over their last 8000 ids, so that page
    offsets pass 32-bit byte offsets: attention (the kernel's TMA rows) against
    the oracle on a compact copy of the same pages, then an append of one row
    per branch read back through the high page ids."""
    spec = small_spec(h_q=64, h_kv=8, page_size=64, prefix_len=1024, q_rows=[1, 3, 2, 1],
                      suffix_lens=[100, 90, 130, 64], permute_prefix=True, permute_suffix=True,
                      seed=321)
    w = draw(spec)
    s = w.spec
    dw = DevWorkload(w)
    n_big = 60000
    remap = (n_big - 8000 + np.random.default_rng(4).permutation(8000)[:w.num_pages])
    kb = torch.empty((n_big, s.h_kv, s.page_size, s.d), dtype=torch.bfloat16, device="cuda")
    vb = torch.empty_like(kb)
    idx = torch.from_numpy(remap.astype(np.int64)).cuda()
    kb[idx] = dw.k
    vb[idx] = dw.v
    tb = dw.table_host.copy()
    tb[tb >= 0] = remap[tb[tb >= 0]]
    assert int(tb.max()) * s.h_kv * s.page_size * s.d * 2 > 2**32
    t_big = torch.from_numpy(tb.astype(np.int32)).cuda()
    out, lse = dw.run(table=t_big, k=kb, v=vb)
    compare(out, lse, *oracle_ref(w), what="pools beyond 4 GB")
    # one new row per branch over its last token (its page is allocated)
    before = (np.asarray(w.suffix_lens) - 1).astype(np.int32)
    add = np.ones(len(before), dtype=np.int32)
    g = torch.Generator().manual_seed(5)
    k_new = torch.randn((len(before), s.h_kv, s.d), generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn((len(before), s.h_kv, s.d), generator=g).to(torch.bfloat16).cuda()
    binding.kv_append(k_new, v_new, kb, vb, t_big, s.prefix_len, before, add, s.page_size)
    assert binding.last_error() == binding.OK
    for b in range(len(before)):
        pos = s.prefix_len + int(before[b])
        page = int(tb[b, pos // s.page_size])
        assert page >= n_big - 8000
        assert torch.equal(kb[page, :, pos % s.page_size], k_new[b])
        assert torch.equal(vb[page, :, pos % s.page_size], v_new[b])
    del kb, vb
    torch.cuda.empty_cache()


@pytest.mark.parametrize("scale", [1e-3, 0.5, 2.0])
def test_softmax_scale(scale):
    """Softmax scales other than 1/sqrt(d): nearly uniform weights (1e-3) and
    sharply peaked ones (2.0, scores up to ~100 in base-2 units), on a split
    problem with causal suffixes, against the oracle with the same scale."""
    spec = small_spec(h_q=16, h_kv=2, page_size=32, prefix_len=768, q_rows=[4, 7, 1],
                      suffix_lens=[150, 60, 400], permute_prefix=True, permute_suffix=True,
                      seed=88)
    w = draw(spec)
    s = w.spec
    dw = DevWorkload(w)
    out, lse = binding.attn(dw.q, dw.k, dw.v, dw.table, s.prefix_len, w.suffix_lens, w.q_rows,
                            s.h_q, s.h_kv, s.page_size, scale, s.causal)
    assert binding.last_error() == binding.OK
    ref = oracle.attn(w.q, w.k_pool, w.v_pool, dw.table_host, s.prefix_len, w.suffix_lens,
                      w.q_rows, s.h_q, s.h_kv, s.page_size, scale, s.causal)
    compare(out, lse, *ref, what=f"scale {scale}")

"""The host work planner: every visible key of every (token, query head) is
covered by exactly one unit, partial slots are consistent, and the planned
work equals the visible-pair count (the pages' compute identity) (CPU only)."""
import numpy as np
import pytest

import oracle
from shared_prefix_fan_gb300 import binding, build
from shared_prefix_fan_gb300.workloads import WORKLOADS, draw

NO_CAUSAL = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def check_plan(S, T, P, h_q, h_kv, ps, causal, sms=148):
    units, cta_first, n_parts = binding.plan(list(map(int, S)), list(map(int, T)), P, h_q, h_kv,
                                             ps, causal, sms)
    return check_units(units, cta_first, n_parts, S, T, P, h_q, h_kv, ps, causal, sms)


def check_units(units, cta_first, n_parts, S, T, P, h_q, h_kv, ps, causal, sms=148):
    S, T = list(map(int, S)), list(map(int, T))
    G = h_q // h_kv
    R = sum(T)
    n_cta = len(cta_first) - 1
    assert 1 <= n_cta <= max(1, sms)
    assert cta_first[0] == 0 and cta_first[-1] == len(units)
    assert (np.diff(cta_first) >= 1).all(), "a CTA without work"
    parts = units[:, 7]
    assert sorted(parts[parts >= 0].tolist()) == list(range(n_parts)), "partial blocks not 0..n-1"
    tok_branch = np.repeat(np.arange(len(T)), T)
    tok0 = np.concatenate([[0], np.cumsum(T)])
    vis = np.zeros(R, dtype=np.int64)
    pos = np.zeros(R, dtype=np.int64)
    for r in range(R):
        b = tok_branch[r]
        pos[r] = P + S[b] - T[b] + (r - tok0[b])
        vis[r] = min(P + S[b], pos[r] + 1) if causal else P + S[b]
    covered = {}   # (r, h) -> list of (lo, hi, part)
    total_pairs = 0
    for row in units:
        h, br, tb, nt, k0, k1, pb, part = (int(x) for x in row)
        assert k1 > k0 >= 0 and nt >= 1 and nt * G <= 256 and 0 <= h < h_kv  # one or two 128-row tiles
        assert k0 % ps == 0, "chunk start not page aligned"
        for r in range(tb, tb + nt):
            b = int(tok_branch[r])
            if k1 > P:   # touches private keys: single-branch unit, through its own table
                assert br == b
            if pb != NO_CAUSAL:
                assert pb + r == pos[r], "causal position mismatch"
            else:
                assert not causal or k1 <= P, "an unmasked unit reaches past the prefix"
            hi = min(k1, int(vis[r]))
            covered.setdefault((r, h), []).append((k0, max(hi, k0), part))
            total_pairs += max(0, hi - k0) * G
    for r in range(R):
        for h in range(h_kv):
            segs = sorted(covered.get((r, h), []))
            assert segs, f"token {r} head {h} uncovered"
            # contiguous, disjoint cover of [0, vis)
            cur = 0
            for lo, hi, _ in segs:
                if hi <= lo:
                    continue  # a chunk entirely in this token's causal future
                assert lo == cur, (r, h, segs)
                cur = hi
            assert cur == vis[r], (r, h, segs, vis[r])
            ps_ = [p_ for _, _, p_ in segs]
            if -1 in ps_:
                assert ps_ == [-1], "a direct unit shares its rows with another unit"
            else:
                assert len(set(ps_)) == len(ps_)
    assert total_pairs == oracle.count_pairs(P, S, T, h_q, causal)
    return units, cta_first, n_parts


@pytest.mark.parametrize("name", ["tiny", "decode", "batching", "wide"])
def test_plan_workloads(name):
    w = draw(WORKLOADS[name]) if name != "wide" else draw(WORKLOADS[name])
    s = w.spec
    check_plan(w.suffix_lens, w.q_rows, s.prefix_len, s.h_q, s.h_kv, s.page_size, s.causal)


def test_plan_prefill_tail_cut():
    """Long prefill: whole query blocks (two 128-row tiles: 32 tokens x 8 heads)
    are written directly; only the blocks cut to even out the last wave become
    partials, and every CTA ends up with the same number of tiles."""
    s = WORKLOADS["prefill"]
    units, cta, n_parts = check_plan(s.suffix_lens, s.q_rows, s.prefix_len, s.h_q, s.h_kv,
                                     s.page_size, s.causal, sms=152)
    assert len(cta) == 153
    assert set((units[:, 3]).tolist()) == {32}
    blocks = {(int(u[0]), int(u[2])) for u in units}
    assert len(blocks) == 8 * 8192 // 32
    assert (units[:, 7] == -1).sum() >= 0.85 * len(units)
    assert n_parts <= 2 * 152
    mk, total = _makespan(units, cta)
    assert mk <= 1.01 * total / 152, (mk, total / 152)


def _makespan(units, cta):
    work = -(-(units[:, 5] - units[:, 4]) // 128) + 2
    return max(work[cta[c]:cta[c + 1]].sum() for c in range(len(cta) - 1)), work.sum()


@pytest.mark.parametrize("name", ["decode", "batching", "wide", "prefill"])
def test_plan_balance(name):
    """Persistent CTAs get nearly equal work (longest-first assignment)."""
    w = draw(WORKLOADS[name])
    s = w.spec
    units, cta, _ = binding.plan(w.suffix_lens, w.q_rows, s.prefix_len, s.h_q, s.h_kv,
                                 s.page_size, s.causal, 152)
    mk, total = _makespan(units, cta)
    assert mk <= 1.25 * total / (len(cta) - 1) + 40, (mk, total / (len(cta) - 1))


@pytest.mark.parametrize("seed", range(16))
def test_plan_random(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 6))
    ps = int(rng.choice([16, 32, 64, 128]))
    P = ps * int(rng.integers(0, 12))
    if seed % 4 == 3:  # a prefix that ends inside a page
        P += int(rng.integers(1, ps))
    causal = bool(rng.integers(0, 2))
    T = rng.integers(0, 40, size=B)
    S = np.array([int(t) + int(rng.integers(0 if P else 1, 300)) for t in T])
    if not causal:
        S = rng.integers(0 if P else 1, 300, size=B)
    hkv = int(rng.choice([1, 2, 8]))
    hq = hkv * int(rng.choice([1, 3, 8, 16]))
    sms = int(rng.choice([1, 7, 148]))
    try:
        binding.set_option(binding.OPT_SPLITS, int(rng.choice([0, 0, 1, 3])))
        check_plan(S, T, P, hq, hkv, ps, causal, sms)
    finally:
        binding.set_option(binding.OPT_SPLITS, 0)


def test_plan_decode_unit_counts():
    """Decode (one query tile per unit): a unit boundary costs about three
    HBM-bound tile times, so no CTA is given more than two units (measured:
    CTAs with three 4-tile suffix units finished last)."""
    w = draw(WORKLOADS["decode"])
    s = w.spec
    units, cta, _ = check_plan(w.suffix_lens, w.q_rows, s.prefix_len, s.h_q, s.h_kv,
                               s.page_size, s.causal, sms=152)
    assert np.diff(cta).max() <= 2



def test_plan_step_keeps_plan_for_a_decode_step():
    """A decode step (every suffix one token longer, no key range gaining a
    128-key tile) keeps the previous plan's chunks and CTA assignment; only
    the range ends and causal positions move, and the plan stays a complete,
    disjoint cover of every visible key."""
    w = draw(WORKLOADS["decode"])
    s = w.spec
    S0 = [500] * 8                      # 4 tiles of suffix keys per branch
    S1 = [501] * 8
    prev, prev_cta, prev_parts = binding.plan(S0, w.q_rows, s.prefix_len, s.h_q, s.h_kv,
                                              s.page_size, s.causal, 152)
    units, cta, n_parts, reused = binding.plan_step(S0, S1, w.q_rows, s.prefix_len, s.h_q, s.h_kv,
                                                    s.page_size, s.causal, 152)
    assert reused
    assert (cta == prev_cta).all() and n_parts == prev_parts
    same = [0, 1, 2, 3, 4, 7]           # kv_head, branch, tok_begin, n_tok, key_begin, part
    assert (units[:, same] == prev[:, same]).all()
    check_units(units, cta, n_parts, S1, w.q_rows, s.prefix_len, s.h_q, s.h_kv, s.page_size,
                s.causal, 152)


def test_plan_step_replans_when_a_range_gains_a_tile():
    w = draw(WORKLOADS["decode"])
    s = w.spec
    S0, S1 = [512] * 8, [513] * 8        # 4 -> 5 tiles of suffix keys
    units, cta, n_parts, reused = binding.plan_step(S0, S1, w.q_rows, s.prefix_len, s.h_q, s.h_kv,
                                                    s.page_size, s.causal, 152)
    assert not reused
    fresh, fresh_cta, fresh_parts = binding.plan(S1, w.q_rows, s.prefix_len, s.h_q, s.h_kv,
                                                 s.page_size, s.causal, 152)
    assert (units == fresh).all() and (cta == fresh_cta).all() and n_parts == fresh_parts


@pytest.mark.parametrize("seed", range(12))
def test_plan_step_random(seed):
    """Random problems and random suffix growth: a kept plan is a valid plan of
    the new problem with the old structure; a rebuilt one is the fresh plan."""
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 6))
    ps = int(rng.choice([16, 32, 64, 128]))
    P = ps * int(rng.integers(0, 12)) + (int(rng.integers(1, ps)) if seed % 3 == 2 else 0)
    causal = bool(rng.integers(0, 2))
    T = rng.integers(0, 30, size=B)
    S0 = np.array([int(t) + int(rng.integers(0 if P else 1, 400)) for t in T])
    S1 = S0 + rng.integers(0, 3 if seed % 2 == 0 else 300, size=B)
    hkv = int(rng.choice([1, 2, 8]))
    hq = hkv * int(rng.choice([1, 4, 8, 16]))
    sms = int(rng.choice([7, 148]))
    units, cta, n_parts, reused = binding.plan_step(S0, S1, T, P, hq, hkv, ps, causal, sms)
    check_units(units, cta, n_parts, S1, T, P, hq, hkv, ps, causal, sms)
    if reused:
        prev, prev_cta, _ = binding.plan(S0, T, P, hq, hkv, ps, causal, sms)
        assert (cta == prev_cta).all()
        assert (units[:, [0, 1, 2, 3, 4, 7]] == prev[:, [0, 1, 2, 3, 4, 7]]).all()
    else:
        fresh, fresh_cta, _ = binding.plan(S1, T, P, hq, hkv, ps, causal, sms)
        assert (units == fresh).all() and (cta == fresh_cta).all()


def test_planning_from_two_threads_at_once():
    """Two host threads plan (and set options) concurrently through the C ABI:
    each gets exactly the plan a lone call gives (ctypes releases the GIL for
    the duration of each call, so the library's planning really overlaps)."""
    import threading

    cases = []
    for name in ("decode", "batching", "wide"):
        w = draw(WORKLOADS[name])
        s = w.spec
        args = (w.suffix_lens, w.q_rows, s.prefix_len, s.h_q, s.h_kv, s.page_size, s.causal, 152)
        cases.append((args, binding.plan(*args)))
    errors = []

    def worker(k):
        try:
            for i in range(8):
                args, (units, cta, n_parts) = cases[(k + i) % len(cases)]
                binding.set_option(binding.OPT_VALIDATE_TABLE, 0)
                got_u, got_c, got_n = binding.plan(*args)
                assert (got_u == units).all() and (got_c == cta).all() and got_n == n_parts
        except Exception as e:  # noqa: BLE001 -- reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors

"""Pins of the fp64 oracle: checks against facts fixed by the pages and by
mathematics, not against the oracle itself.

Each pin takes the oracle library handle, so the same checks can run against a
build of the oracle with a planted mistake (see test_oracle_mutations.py):
every planted mistake must make at least one pin fail.

Facts used:
  * brute force: full score matrix, library softmax / logsumexp, textbook GQA
    head repeat and a bottom-right-aligned causal mask (new tokens are the tail
    of the context) -- "AHBM Agentic Runtime Architecture" section 1.1 (branch
    = shared prefix + private instruction + private continuation) and ADR-0060
    section 5.4 (causal tile rules);
  * closed forms: identical keys give the mean of the visible V rows and
    lse = s + ln n; a single visible key gives that key's V row;
  * batching invariance ("batching changes the execution shape, not the
    attention semantics", Agentic_Runtime_Architecture section 3.2);
  * merge invariance: partial states over a split of the keys merged with the
    pairwise log-sum-exp rule equal the unsplit result (ADR-0060 section 4;
    Agentic_Runtime_Architecture section 3.4);
  * GQA invariance: folding G query heads onto one KV head equals a plain
    multi-head problem with each KV head repeated G times (ADR-0060 section 5.2);
  * fork invariance: physical page placement, and sharing vs duplicating the
    prefix pages, do not change the result (Agentic_Runtime_Architecture 3.1);
  * causal reductions: one new token sees the whole context; a single
    sequence with no cached prefix is plain causal self-attention;
  * the pages' work identity (Agentic_Runtime_Architecture section 3.7): the
    visible-pair count does not depend on how keys are split.
"""
from __future__ import annotations

import numpy as np
import scipy.special
import torch

import oracle
from shared_prefix_fan_gb300.workloads import _bf16_bits, bf16_bits_to_f32


def bf16(x: np.ndarray) -> np.ndarray:
    return _bf16_bits(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)))


def f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


class Problem:
    """A problem built from LOGICAL per-branch K/V, scattered into a paged pool.

    The scatter is written here, independently of the oracle's gather.
    """

    def __init__(self, rng, B, P, S, T, h_q, h_kv, d, page, causal, scale=None,
                 permute=True, k_mult=1.0, same_keys=False):
        self.B, self.P, self.S, self.T = B, P, list(S), list(T)
        self.h_q, self.h_kv, self.d, self.page, self.causal = h_q, h_kv, d, page, causal
        self.scale = 1.0 / np.sqrt(d) if scale is None else scale
        kp = rng.standard_normal((P, h_kv, d)) * k_mult
        ks = [rng.standard_normal((s, h_kv, d)) * k_mult for s in self.S]
        if same_keys:
            row = rng.standard_normal((1, h_kv, d))
            kp = np.broadcast_to(row, kp.shape).copy()
            ks = [np.broadcast_to(row, k.shape).copy() for k in ks]
        vp = rng.standard_normal((P, h_kv, d))
        vs = [rng.standard_normal((s, h_kv, d)) for s in self.S]
        self.k_log = [bf16(np.concatenate([kp, k], 0)) for k in ks]
        # prefix rows must be bit-identical across branches
        for b in range(B):
            self.k_log[b][:P] = self.k_log[0][:P]
        self.v_log = [bf16(np.concatenate([vp, v], 0)) for v in vs]
        for b in range(B):
            self.v_log[b][:P] = self.v_log[0][:P]
        self.q = bf16(rng.standard_normal((sum(self.T), h_q, d)))
        n_pre = P // page
        n_priv = [(s + page - 1) // page for s in self.S]
        num_pages = n_pre + sum(n_priv)
        ids = rng.permutation(num_pages).astype(np.int32) if permute else \
            np.arange(num_pages, dtype=np.int32)
        self.prefix_pages = ids[:n_pre].copy()
        self.free_pages = ids[n_pre:].copy()
        self.max_pages = n_pre + max(n_priv + [0]) + 1  # one spare column
        self.table = np.full((B, self.max_pages), -1, dtype=np.int32)
        nxt = 0
        for b in range(B):
            self.table[b, :n_pre] = self.prefix_pages
            self.table[b, n_pre:n_pre + n_priv[b]] = self.free_pages[nxt:nxt + n_priv[b]]
            nxt += n_priv[b]
        # pool filled with garbage first: slots outside every sequence must not be read
        garbage = bf16(rng.standard_normal((num_pages, h_kv, page, d)) * 1e4)
        self.k_pool = garbage.copy()
        self.v_pool = garbage.copy()
        for b in range(B):
            for j in range(P + self.S[b]):
                pg = self.table[b, j // page]
                self.k_pool[pg, :, j % page, :] = self.k_log[b][j]
                self.v_pool[pg, :, j % page, :] = self.v_log[b][j]

    def run(self, lib, rows=None, table=None, k_pool=None, v_pool=None, h_kv=None, causal=None):
        return oracle.attn(self.q, self.k_pool if k_pool is None else k_pool,
                           self.v_pool if v_pool is None else v_pool,
                           self.table if table is None else table, self.P, self.S, self.T,
                           self.h_q, self.h_kv if h_kv is None else h_kv, self.page, self.scale,
                           self.causal if causal is None else causal, rows=rows, lib=lib)

    def brute(self, causal=None):
        """Full score matrix per branch, textbook GQA repeat, library softmax."""
        causal = self.causal if causal is None else causal
        G = self.h_q // self.h_kv
        outs, lses, r0 = [], [], 0
        for b in range(self.B):
            T, n = self.T[b], self.P + self.S[b]
            qb = f64(self.q[r0:r0 + T])  # [T, H_q, d]
            kb = np.repeat(f64(self.k_log[b]), G, axis=1)  # [n, H_q, d]
            vb = np.repeat(f64(self.v_log[b]), G, axis=1)
            s = self.scale * np.einsum("thd,nhd->htn", qb, kb)
            if causal:
                allowed = np.tril(np.ones((T, n), dtype=bool), k=n - T)
                s = np.where(allowed[None], s, -np.inf)
            w = scipy.special.softmax(s, axis=-1)
            outs.append(np.einsum("htn,nhd->thd", w, vb))
            lses.append(scipy.special.logsumexp(s, axis=-1).T)
            r0 += T
        return np.concatenate(outs, 0), np.concatenate(lses, 0)


def _close(a, b, tol):
    assert a.shape == b.shape, (a.shape, b.shape)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"max abs diff {err:.3e} > {tol:.1e}"


def _shapes():
    # (B, P, S, T, h_q, h_kv, d, page, causal)
    return [
        (3, 32, [5, 16, 9], [2, 4, 3], 8, 2, 16, 8, True),
        (2, 0, [12, 7], [12, 7], 4, 4, 8, 4, True),
        (2, 16, [4, 11], [1, 5], 6, 3, 4, 4, False),
        (1, 64, [24], [6], 8, 1, 128, 16, True),
    ]


def pin_brute_force(lib, seed=0):
    rng = np.random.default_rng(seed)
    for shp in _shapes():
        pb = Problem(rng, *shp)
        out, lse = pb.run(lib)
        bo, bl = pb.brute()
        _close(out, bo, 1e-12)
        _close(lse, bl, 1e-12)


def pin_identical_keys(lib, seed=1):
    rng = np.random.default_rng(seed)
    pb = Problem(rng, 2, 32, [9, 20], [3, 6], 8, 2, 16, 8, True, same_keys=True)
    out, lse = pb.run(lib)
    G = pb.h_q // pb.h_kv
    r = 0
    for b in range(pb.B):
        n_all = pb.P + pb.S[b]
        for t in range(pb.T[b]):
            n_vis = n_all - pb.T[b] + t + 1  # the new token sees itself and all before it
            for h in range(pb.h_q):
                kv = h // G
                v = f64(pb.v_log[b][:n_vis, kv])
                _close(out[r, h], v.mean(0), 1e-12)
                s0 = pb.scale * float(f64(pb.q[r, h]) @ f64(pb.k_log[b][0, kv]))
                assert abs(lse[r, h] - (s0 + np.log(n_vis))) <= 1e-12
            r += 1


def pin_single_key(lib, seed=2):
    rng = np.random.default_rng(seed)
    # no prefix, the first new token of a causal branch sees only key 0
    pb = Problem(rng, 1, 0, [5], [5], 4, 2, 8, 4, True)
    out, lse = pb.run(lib)
    G = pb.h_q // pb.h_kv
    for h in range(pb.h_q):
        _close(out[0, h], f64(pb.v_log[0][0, h // G]), 0.0)
        s0 = pb.scale * float(f64(pb.q[0, h]) @ f64(pb.k_log[0][0, h // G]))
        assert abs(lse[0, h] - s0) <= 1e-12
    # a context of exactly one key, non-causal
    pb = Problem(rng, 2, 0, [1, 1], [1, 1], 4, 1, 8, 4, False)
    out, _ = pb.run(lib)
    for b in range(2):
        for h in range(pb.h_q):
            _close(out[b, h], f64(pb.v_log[b][0, 0]), 0.0)


def pin_batching_invariance(lib, seed=3):
    rng = np.random.default_rng(seed)
    pb = Problem(rng, 3, 48, [10, 3, 17], [4, 2, 5], 8, 2, 16, 16, True)
    out, lse = pb.run(lib)
    r0 = 0
    for b in range(pb.B):
        T = pb.T[b]
        q_b = pb.q[r0:r0 + T]
        o_b, l_b = oracle.attn(q_b, pb.k_pool, pb.v_pool, pb.table[b:b + 1], pb.P, [pb.S[b]],
                               [T], pb.h_q, pb.h_kv, pb.page, pb.scale, pb.causal, lib=lib)
        _close(out[r0:r0 + T], o_b, 0.0)
        _close(lse[r0:r0 + T], l_b, 0.0)
        r0 += T


def pin_merge_invariance(lib, seed=4):
    rng = np.random.default_rng(seed)
    pb = Problem(rng, 2, 64, [30, 45], [5, 7], 8, 2, 16, 8, True)
    out, lse = pb.run(lib)
    n_max = pb.P + max(pb.S)
    for cuts in ([0, n_max], [0, 64, n_max], [0, 8, 24, 64, 72, n_max], [0, 40, 48, n_max]):
        parts = [oracle.attn_partial(pb.q, pb.k_pool, pb.v_pool, pb.table, pb.P, pb.S, pb.T,
                                     pb.h_q, pb.h_kv, pb.page, pb.scale, pb.causal, lo, hi,
                                     lib=lib) for lo, hi in zip(cuts[:-1], cuts[1:])]
        pm = np.stack([p[0] for p in parts])
        pl = np.stack([p[1] for p in parts])
        po = np.stack([p[2] for p in parts])
        mo, ml = oracle.merge(pm, pl, po, lib=lib)
        _close(mo, out, 1e-12)
        _close(ml, lse, 1e-12)
        # the merge is order-free (associative and commutative)
        rev = oracle.merge(pm[::-1], pl[::-1], po[::-1], lib=lib)
        _close(rev[0], out, 1e-12)


def pin_gqa_invariance(lib, seed=5):
    rng = np.random.default_rng(seed)
    pb = Problem(rng, 2, 16, [7, 12], [3, 4], 8, 2, 16, 8, True)
    out, lse = pb.run(lib)
    G = pb.h_q // pb.h_kv
    k_mha = np.repeat(pb.k_pool, G, axis=1)
    v_mha = np.repeat(pb.v_pool, G, axis=1)
    o2, l2 = pb.run(lib, k_pool=k_mha, v_pool=v_mha, h_kv=pb.h_q)
    _close(out, o2, 0.0)
    _close(lse, l2, 0.0)


def pin_fork_invariance(lib, seed=6):
    rng = np.random.default_rng(seed)
    pb = Problem(rng, 3, 32, [5, 9, 1], [2, 3, 1], 4, 2, 8, 8, True)
    out, lse = pb.run(lib)
    # (a) move every physical page somewhere else
    perm = rng.permutation(pb.k_pool.shape[0])
    inv = np.argsort(perm)
    k2, v2 = pb.k_pool[perm], pb.v_pool[perm]
    t2 = np.where(pb.table >= 0, inv[np.maximum(pb.table, 0)], -1).astype(np.int32)
    o2, l2 = pb.run(lib, table=t2, k_pool=k2, v_pool=v2)
    _close(out, o2, 0.0)
    _close(lse, l2, 0.0)
    # (b) give every branch its own copy of the prefix pages
    n_pre = pb.P // pb.page
    k3, v3, t3 = [pb.k_pool], [pb.v_pool], pb.table.copy()
    base = pb.k_pool.shape[0]
    for b in range(1, pb.B):
        k3.append(pb.k_pool[pb.prefix_pages])
        v3.append(pb.v_pool[pb.prefix_pages])
        t3[b, :n_pre] = np.arange(base, base + n_pre, dtype=np.int32)
        base += n_pre
    o3, l3 = pb.run(lib, table=t3, k_pool=np.concatenate(k3), v_pool=np.concatenate(v3))
    _close(out, o3, 0.0)
    _close(lse, l3, 0.0)


def pin_causal_reductions(lib, seed=7):
    rng = np.random.default_rng(seed)
    pb = Problem(rng, 3, 24, [6, 1, 13], [1, 1, 1], 8, 4, 16, 8, True)
    oc, lc = pb.run(lib, causal=True)
    on, ln = pb.run(lib, causal=False)
    _close(oc, on, 0.0)
    _close(lc, ln, 0.0)
    # one sequence, nothing cached: standard causal self-attention (library SDPA)
    pb = Problem(rng, 1, 0, [11], [11], 4, 2, 16, 4, True)
    out, _ = pb.run(lib)
    G = pb.h_q // pb.h_kv
    q = torch.from_numpy(f64(pb.q)).permute(1, 0, 2)  # [H, T, d]
    k = torch.from_numpy(np.repeat(f64(pb.k_log[0]), G, axis=1)).permute(1, 0, 2)
    v = torch.from_numpy(np.repeat(f64(pb.v_log[0]), G, axis=1)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=pb.scale)
    _close(out, ref.permute(1, 0, 2).numpy(), 1e-12)


def pin_fork(lib, seed=8):
    rng = np.random.default_rng(seed)
    pb = Problem(rng, 4, 48, [17, 0, 33, 16], [1, 0, 2, 3], 4, 2, 8, 16, True)
    table = oracle.fork(pb.prefix_pages, pb.S, pb.page, pb.free_pages, pb.max_pages, lib=lib)
    assert np.array_equal(table, pb.table), "fork differs from prefix + private pages in order"
    n_pre = pb.P // pb.page
    assert (table[:, :n_pre] == pb.prefix_pages[None]).all()
    priv = table[:, n_pre:]
    used = priv[priv >= 0]
    assert len(np.unique(used)) == len(used), "a private page is shared"
    assert not np.isin(used, pb.prefix_pages).any()


def pin_work_identity(lib):
    """The pages' printed example (tests/golden/pages_work_identity.json)."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "pages_work_identity.json")))
    n_agents, t_new = g["agents"], g["new_tokens_per_agent"]
    assert n_agents * t_new == g["combined_q_rows"]
    assert g["pes"] * g["local_kv_columns"] == g["total_kv_columns"]
    n_cols = g["total_kv_columns"]
    # a context of n_cols keys per agent, the last t_new of them new, non-causal:
    # every row sees every column
    P, T, S = n_cols - t_new, [t_new] * n_agents, [t_new] * n_agents
    full = oracle.count_pairs(P, S, T, 1, causal=False, lib=lib)
    assert full == g["combined_q_rows"] * n_cols
    assert full == g["pes"] * g["combined_q_rows"] * g["local_kv_columns"]
    assert full == (g["temporal_q_groups"] * g["pes"] * g["rows_per_temporal_group"]
                    * g["local_kv_columns"])
    # causal: token t of a branch sees P + S - T + t + 1 keys
    c = oracle.count_pairs(P, S, T, 1, causal=True, lib=lib)
    assert c == n_agents * sum(P + 1 + t for t in range(t_new))
    assert oracle.count_pairs(P, S, T, 64, causal=True, lib=lib) == 64 * c


def pin_append(lib, seed=9):
    """Fork for the current suffixes, then grow the tables and append the new
    tokens' K/V: every logical key of every branch must then read back its own
    row (checked by a gather written here), and attention must match brute
    force on the grown contexts (ADR-0060 section 0.5.1, precondition P3).
    The last case has a prefix ending inside a page (forked with copy-on-write
    of that page): the growth continues from the branch's last token wherever
    the prefix ended."""
    rng = np.random.default_rng(seed)
    for (P, S_old, T, page) in ((32, [5, 16, 0], [3, 1, 4], 8), (0, [7, 1], [2, 9], 4),
                                (21, [5, 0, 11], [3, 9, 1], 8)):
        S_new = [a + b for a, b in zip(S_old, T)]
        pb = Problem(rng, len(T), P, S_new, T, 8, 2, 16, page, True)
        # the state before the append: a pool holding only the old tokens
        max_pages = max(-(-(P + s) // page) for s in S_new) + 1
        free = rng.permutation(np.arange(2000, 2000 + 200, dtype=np.int32))
        n_pre = -(-P // page)
        pre_ids = np.arange(1000, 1000 + n_pre, dtype=np.int32)
        if P % page == 0:
            table0 = oracle.fork(pre_ids, S_old, page, free, max_pages, lib=lib)
            n_used0 = sum((s + page - 1) // page for s in S_old)
        else:
            table0, _, n_used0 = oracle.fork_cow(pre_ids, P, S_old, page, free, max_pages,
                                                 lib=lib)
        pool_pages = 2200
        kp = np.zeros((pool_pages, pb.h_kv, page, pb.d), np.uint16)
        vp = np.zeros_like(kp)
        for b in range(pb.B):
            for j in range(P + S_old[b]):
                pg = table0[b, j // page]
                kp[pg, :, j % page] = pb.k_log[b][j]
                vp[pg, :, j % page] = pb.v_log[b][j]
        table1, used = oracle.extend(table0, P, S_old, T, page, free[n_used0:], lib=lib)
        # pages a branch holds: one per page_size of its logical positions
        assert used == sum(-(-(P + s + t) // page) - -(-(P + s) // page)
                           for s, t in zip(S_old, T))
        assert (table1[table0 >= 0] == table0[table0 >= 0]).all()
        grown = table1[table1 >= 0]
        assert len(np.unique(grown[grown >= 2000])) == len(grown[grown >= 2000])
        k_new = np.concatenate([pb.k_log[b][P + S_old[b]:] for b in range(pb.B)])
        v_new = np.concatenate([pb.v_log[b][P + S_old[b]:] for b in range(pb.B)])
        kp1, vp1 = oracle.kv_append(k_new, v_new, kp, vp, table1, P, S_old, T, lib=lib)
        for b in range(pb.B):
            for j in range(P + S_new[b]):
                pg = table1[b, j // page]
                assert (kp1[pg, :, j % page] == pb.k_log[b][j]).all(), (b, j)
                assert (vp1[pg, :, j % page] == pb.v_log[b][j]).all(), (b, j)
        out, lse = oracle.attn(pb.q, kp1, vp1, table1, P, S_new, T, pb.h_q, pb.h_kv, page,
                               pb.scale, True, lib=lib)
        bo, bl = pb.brute()
        _close(out, bo, 1e-12)
        _close(lse, bl, 1e-12)


def pin_partial_prefix(lib, seed=10):
    """A prefix ending inside a page: fork with copy-on-write of the partial
    page, copy it, then every branch reads back its own logical sequence
    through its table (a gather written here) and attention equals brute force
    ("AHBM Agentic Runtime Architecture" section 3.1: shared pages referenced,
    the partial one copied so branches can extend it)."""
    rng = np.random.default_rng(seed)
    for (P, S, T, page) in ((21, [6, 0, 13], [2, 0, 5], 8), (3, [9, 4], [9, 1], 4)):
        pb = Problem(rng, len(S), P, S, T, 8, 2, 16, page, True)
        n_pre = -(-P // page)
        pre_ids = np.arange(500, 500 + n_pre, dtype=np.int32)
        free = rng.permutation(np.arange(1000, 1100, dtype=np.int32))
        mp = n_pre + max(-(-(P + s) // page) for s in S) + 1
        table, cow, used = oracle.fork_cow(pre_ids, P, S, page, free, mp, lib=lib)
        assert (table[:, :P // page] == pre_ids[None, :P // page]).all()
        assert len(np.unique(table[table >= 1000])) == (table >= 1000).sum()
        kp = np.zeros((1100, pb.h_kv, page, pb.d), np.uint16)
        vp = np.zeros_like(kp)
        for j in range(P):  # the shared prefix, in the shared pages
            kp[pre_ids[j // page], :, j % page] = pb.k_log[0][j]
            vp[pre_ids[j // page], :, j % page] = pb.v_log[0][j]
        kp, vp = oracle.copy_pages(kp, vp, cow, P % page, lib=lib)
        for b in range(pb.B):  # each branch's suffix, in its own pages
            for j in range(P, P + S[b]):
                kp[table[b, j // page], :, j % page] = pb.k_log[b][j]
                vp[table[b, j // page], :, j % page] = pb.v_log[b][j]
        for b in range(pb.B):
            for j in range(P + S[b]):
                assert (kp[table[b, j // page], :, j % page] == pb.k_log[b][j]).all(), (b, j)
        out, lse = oracle.attn(pb.q, kp, vp, table, P, S, T, pb.h_q, pb.h_kv, page, pb.scale,
                               True, lib=lib)
        bo, bl = pb.brute()
        _close(out, bo, 1e-12)
        _close(lse, bl, 1e-12)


ALL_PINS = [pin_brute_force, pin_identical_keys, pin_single_key, pin_batching_invariance,
            pin_merge_invariance, pin_gqa_invariance, pin_fork_invariance,
            pin_causal_reductions, pin_fork, pin_work_identity, pin_append,
            pin_partial_prefix]

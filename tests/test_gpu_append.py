"""fanout_kv_append on the GPU against the oracle's append (bit-exact pools), and
the whole step a decoding fan-out runs -- fork, grow the tables, append the
new tokens' K/V, attend -- against the oracle doing the same."""
import numpy as np
import pytest
import torch

import oracle
from shared_prefix_fan_gb300 import binding
from shared_prefix_fan_gb300.workloads import _bf16_bits, draw, small_spec
from tests.gpu_helpers import compare, ensure_lib, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", range(3))
def test_fork_extend_append_attend(case):
    ensure_lib()
    tq, s_old, P, ps, hq, hkv = [
        ([1] * 8, [500] * 8, 1024, 64, 64, 8),
        ([3, 0, 17, 5], [13, 40, 0, 77], 256, 16, 16, 2),
        ([20, 20], [236, 100], 512, 32, 32, 4),
    ][case]
    s_new = [a + b for a, b in zip(s_old, tq)]
    spec = small_spec(h_q=hq, h_kv=hkv, page_size=ps, prefix_len=P, q_rows=tq,
                      suffix_lens=s_new, permute_prefix=True, permute_suffix=True, seed=300 + case)
    w = draw(spec)  # pool sized for the grown suffixes; the drawn values are the "old" cache
    rng = np.random.default_rng(case)
    R = int(sum(tq))
    k_new = _bf16_bits(torch.from_numpy(rng.standard_normal((R, hkv, 128)).astype(np.float32)))
    v_new = _bf16_bits(torch.from_numpy(rng.standard_normal((R, hkv, 128)).astype(np.float32)))
    n_pre = P // ps
    mp = w.max_pages_per_branch
    n_old = sum((s + ps - 1) // ps for s in s_old)
    # product: fork for the old suffixes, grow, append on the device
    t0 = binding.fork(w.prefix_pages, s_old, ps, w.free_pages, mp)
    t1, used = binding.extend(t0, P, s_old, tq, ps, w.free_pages[n_old:])
    k_pool, v_pool = to_dev_bf16(w.k_pool), to_dev_bf16(w.v_pool)
    dt1 = torch.from_numpy(t1).cuda()
    binding.kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), k_pool, v_pool, dt1, P, s_old, tq,
                      ps)
    assert binding.last_error() == binding.OK
    # oracle: the same steps on the host
    r0 = oracle.fork(w.prefix_pages, s_old, ps, w.free_pages, mp)
    r1, used_ref = oracle.extend(r0, P, s_old, tq, ps, w.free_pages[n_old:])
    assert np.array_equal(t1, r1) and used == used_ref
    rk, rv = oracle.kv_append(k_new, v_new, w.k_pool, w.v_pool, r1, P, s_old, tq)
    gk = k_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    gv = v_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
    # attention over the grown contexts, the new tokens attending as the suffix tail
    q = to_dev_bf16(w.q)
    out, lse = binding.attn(q, k_pool, v_pool, dt1, P, s_new, tq, hq, hkv, ps, spec.scale, True)
    assert binding.last_error() == binding.OK
    ro, rl = oracle.attn(w.q, rk, rv, r1, P, s_new, tq, hq, hkv, ps, spec.scale, True)
    compare(out, lse, ro, rl, what=f"append case {case}")


def test_kv_append_skips_bad_page_ids():
    ensure_lib()
    k_pool = torch.zeros((4, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    table = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")  # page 99 does not exist
    k_new = torch.ones((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    binding.kv_append(k_new, k_new.clone(), k_pool, v_pool, table, 0, [16], [1], 16)
    assert binding.last_error() == binding.EINVAL
    assert (k_pool == 0).all() and (v_pool == 0).all()


@pytest.mark.parametrize("ps,hkv", [(64, 8), (24, 8), (64, 3), (24, 3)])
def test_kv_append_many_rows(ps, hkv):
    """A long append (4 branches x 700 new tokens: several items per warp) lands
    every row where the oracle's append puts it, bit for bit, for power-of-two
    and other page sizes (24 tokens) and KV head counts (3)."""
    ensure_lib()
    rng = np.random.default_rng(ps * 10 + hkv)
    B, d = 4, 128
    s_old = rng.integers(0, 300, size=B).astype(np.int32)
    add = np.full(B, 700, dtype=np.int32)
    P = 2 * ps
    ends = P + s_old + add
    mp = int(((ends + ps - 1) // ps).max())
    n_pages = B * mp + 8
    perm = rng.permutation(n_pages).astype(np.int32)
    table = np.full((B, mp), -1, dtype=np.int32)
    n_pre, nxt = P // ps, P // ps
    for b in range(B):
        need = int((ends[b] + ps - 1) // ps)
        table[b, :n_pre] = perm[:n_pre]                    # the shared prefix pages
        table[b, n_pre:need] = perm[nxt:nxt + need - n_pre]
        nxt += need - n_pre
    kp = rng.integers(0, 2**16, size=(n_pages, hkv, ps, d), dtype=np.uint16)
    vp = rng.integers(0, 2**16, size=(n_pages, hkv, ps, d), dtype=np.uint16)
    R = int(add.sum())
    kn = rng.integers(0, 2**16, size=(R, hkv, d), dtype=np.uint16)
    vn = rng.integers(0, 2**16, size=(R, hkv, d), dtype=np.uint16)
    rk, rv = oracle.kv_append(kn, vn, kp, vp, table, P, s_old, add)
    gk, gv = to_dev_bf16(kp), to_dev_bf16(vp)
    binding.kv_append(to_dev_bf16(kn), to_dev_bf16(vn), gk, gv, torch.from_numpy(table).cuda(),
                      P, s_old, add, ps)
    assert binding.last_error() == binding.OK
    assert np.array_equal(gk.view(torch.int16).cpu().numpy().view(np.uint16), rk)
    assert np.array_equal(gv.view(torch.int16).cpu().numpy().view(np.uint16), rv)


def test_decode_loop_with_page_growth():
    """Six decode steps of a three-branch fan-out, as a caller runs them: grow
    the tables (fanout_extend, new pages as suffixes cross 16-token pages),
    append the new tokens' K/V (fanout_kv_append), attend with those tokens as
    the queries. Every step's tables, pools and attention against the oracle
    doing the same steps."""
    ensure_lib()
    P, ps, hq, hkv = 128, 16, 16, 2
    s0 = np.array([14, 30, 5], dtype=np.int32)
    steps = [np.array(a, dtype=np.int32) for a in ([1, 2, 1], [1, 2, 3], [2, 1, 1],
                                                     [1, 1, 1], [3, 2, 1], [1, 2, 2])]
    s_final = s0 + sum(steps)
    spec = small_spec(h_q=hq, h_kv=hkv, page_size=ps, prefix_len=P, q_rows=[1, 1, 1],
                      suffix_lens=[int(x) for x in s_final], permute_prefix=True,
                      permute_suffix=True, seed=404)
    w = draw(spec)        # a pool with pages for the final lengths
    rng = np.random.default_rng(404)
    mp = w.max_pages_per_branch
    n_used0 = sum(-(-int(s) // ps) for s in s0)
    table = binding.fork(w.prefix_pages, s0, ps, w.free_pages, mp)
    ref_table = oracle.fork(w.prefix_pages, s0, ps, w.free_pages, mp)
    free = w.free_pages[n_used0:]
    k_pool, v_pool = to_dev_bf16(w.k_pool), to_dev_bf16(w.v_pool)
    rk, rv = w.k_pool.copy(), w.v_pool.copy()
    s = s0.copy()
    for i, add in enumerate(steps):
        R = int(add.sum())
        kn = _bf16_bits(torch.from_numpy(rng.standard_normal((R, hkv, 128)).astype(np.float32)))
        vn = _bf16_bits(torch.from_numpy(rng.standard_normal((R, hkv, 128)).astype(np.float32)))
        q = _bf16_bits(torch.from_numpy(rng.standard_normal((R, hq, 128)).astype(np.float32)))
        table, used = binding.extend(table, P, s, add, ps, free)
        ref_table, ref_used = oracle.extend(ref_table, P, s, add, ps, free)
        assert np.array_equal(table, ref_table) and used == ref_used
        free = free[used:]
        t_dev = torch.from_numpy(table).cuda()
        binding.kv_append(to_dev_bf16(kn), to_dev_bf16(vn), k_pool, v_pool, t_dev, P, s, add, ps)
        assert binding.last_error() == binding.OK
        rk, rv = oracle.kv_append(kn, vn, rk, rv, ref_table, P, s, add)
        s = s + add
        out, lse = binding.attn(to_dev_bf16(q), k_pool, v_pool, t_dev, P, s, add, hq, hkv, ps,
                                spec.scale, True)
        assert binding.last_error() == binding.OK
        ro, rl = oracle.attn(q, rk, rv, ref_table, P, s, add, hq, hkv, ps, spec.scale, True)
        compare(out, lse, ro, rl, what=f"decode loop step {i}")
    assert np.array_equal(k_pool.view(torch.int16).cpu().numpy().view(np.uint16), rk)

"""Fan-out then join on the GPU ("AHBM Agentic Runtime Architecture" sections
5.2-5.4): branches fork the shared prefix and decode privately; at the join
the main agent's page table is [shared prefix pages] + [join-input pages] +
[continuation pages] -- the branches' private pages are not attached -- and
the join input plus continuation are prefilled causally through the same
kernel. Checked against the oracle running the same steps."""
import numpy as np
import pytest
import torch

import oracle
from shared_prefix_fan_gb300 import binding
from shared_prefix_fan_gb300.workloads import _bf16_bits
from tests.gpu_helpers import compare, ensure_lib, to_dev_bf16

pytestmark = pytest.mark.gpu


def _bf16(rng, shape):
    return _bf16_bits(torch.from_numpy(rng.standard_normal(shape).astype(np.float32)))


def test_fanout_then_join_continuation_prefill():
    ensure_lib()
    rng = np.random.default_rng(7)
    hq, hkv, ps, P = 32, 4, 64, 1000           # prefix ends inside a page
    S_br = [150, 90, 200]                       # private branch suffixes (already decoded)
    J, C = 120, 40                              # join-input tokens, continuation tokens
    n_pages = 200
    pool_k = _bf16(rng, (n_pages, hkv, ps, 128))
    pool_v = _bf16(rng, (n_pages, hkv, ps, 128))
    free = list(rng.permutation(np.arange(n_pages, dtype=np.int32)))
    n_pre = -(-P // ps)
    pre_ids, free = np.array(free[:n_pre], np.int32), free[n_pre:]
    # fan-out: branches fork the prefix (copy-on-write of its partial last page)
    mp = 40
    t_br, cow_br, used = binding.fork_cow(pre_ids, P, S_br, ps, free, mp)
    free = free[used:]
    dk, dv = to_dev_bf16(pool_k), to_dev_bf16(pool_v)
    binding.copy_pages(dk, dv, torch.from_numpy(cow_br).cuda(), P % ps)
    rk, rv = oracle.copy_pages(pool_k, pool_v, cow_br, P % ps)
    # join: the main agent gets the prefix + its own pages for join input and continuation
    t_main, cow_main, used = binding.fork_cow(pre_ids, P, [0], ps, free, mp)
    free = free[used:]
    assert not np.isin(t_main[t_main >= 0], t_br[:, n_pre - 1:]).any(), "branch pages attached"
    binding.copy_pages(dk, dv, torch.from_numpy(cow_main).cuda(), P % ps)
    rk, rv = oracle.copy_pages(rk, rv, cow_main, P % ps)
    t_main, used = binding.extend(t_main, P, [0], [J + C], ps, free)
    k_new, v_new = _bf16(rng, (J + C, hkv, 128)), _bf16(rng, (J + C, hkv, 128))
    dt = torch.from_numpy(t_main).cuda()
    binding.kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), dk, dv, dt, P, [0], [J + C], ps)
    rk, rv = oracle.kv_append(k_new, v_new, rk, rv, t_main, P, [0], [J + C])
    # continuation prefill of the join input + continuation, causal
    q = _bf16(rng, (J + C, hq, 128))
    out, lse = binding.attn(to_dev_bf16(q), dk, dv, dt, P, [J + C], [J + C], hq, hkv, ps,
                            128 ** -0.5, True)
    assert binding.last_error() == binding.OK
    ro, rl = oracle.attn(q, rk, rv, t_main, P, [J + C], [J + C], hq, hkv, ps, 128 ** -0.5, True)
    compare(out, lse, ro, rl, what="join continuation prefill")
    # the join saw only the prefix and the main agent's own tokens: branch pages untouched
    for b in range(len(S_br)):
        own = t_br[b, n_pre:][t_br[b, n_pre:] >= 0]
        assert np.array_equal(dk[torch.from_numpy(own).long().cuda()].view(torch.int16).cpu()
                              .numpy().view(np.uint16), rk[own])

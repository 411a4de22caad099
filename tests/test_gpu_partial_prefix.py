"""A shared prefix that ends inside a page, on the GPU: copy-on-write fork,
device page copy (bit-exact against the oracle), attention against the oracle,
and an append after the fork that leaves the shared pages untouched."""
import numpy as np
import pytest
import torch

import oracle
from shared_prefix_fan_gb300 import binding
from shared_prefix_fan_gb300.workloads import _bf16_bits
from tests.gpu_helpers import compare, ensure_lib, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", range(3))
def test_partial_prefix_fork_copy_attend(case):
    ensure_lib()
    P, S, T, ps, hq, hkv = [
        (1000, [300, 7, 64], [5, 7, 30], 64, 64, 8),
        (37, [20, 20], [1, 16], 16, 8, 2),
        (4095, [1] * 8, [1] * 8, 128, 16, 2),
    ][case]
    rng = np.random.default_rng(case)
    n_pre = -(-P // ps)
    n_pages = n_pre + sum(-(-(P % ps + s) // ps) + 1 for s in S) + 8
    ids = rng.permutation(n_pages).astype(np.int32)
    mp = max(-(-(P + s) // ps) for s in S) + 1
    table, cow, used = binding.fork_cow(ids[:n_pre], P, S, ps, ids[n_pre:], mp)
    kp = _bf16_bits(torch.from_numpy(rng.standard_normal((n_pages, hkv, ps, 128)).astype(np.float32)))
    vp = _bf16_bits(torch.from_numpy(rng.standard_normal((n_pages, hkv, ps, 128)).astype(np.float32)))
    dk, dv = to_dev_bf16(kp), to_dev_bf16(vp)
    if P % ps:
        binding.copy_pages(dk, dv, torch.from_numpy(cow).cuda(), P % ps)
        assert binding.last_error() == binding.OK
        rk, rv = oracle.copy_pages(kp, vp, cow, P % ps)
    else:
        rk, rv = kp, vp
    assert np.array_equal(dk.view(torch.int16).cpu().numpy().view(np.uint16), rk)
    assert np.array_equal(dv.view(torch.int16).cpu().numpy().view(np.uint16), rv)
    q = _bf16_bits(torch.from_numpy(rng.standard_normal((sum(T), hq, 128)).astype(np.float32)))
    out, lse = binding.attn(to_dev_bf16(q), dk, dv, torch.from_numpy(table).cuda(), P, S, T, hq,
                            hkv, ps, 128 ** -0.5, True)
    assert binding.last_error() == binding.OK
    ro, rl = oracle.attn(q, rk, rv, table, P, S, T, hq, hkv, ps, 128 ** -0.5, True)
    compare(out, lse, ro, rl, what=f"partial prefix case {case}")


def test_append_after_cow_fork_leaves_shared_pages():
    ensure_lib()
    P, S, ps, hkv = 40, [0, 0, 0], 16, 2
    ids = np.arange(20, dtype=np.int32)
    table, cow, _ = binding.fork_cow(ids[:3], P, S, ps, ids[3:], 4)
    kp = torch.randn((20, hkv, ps, 128), device="cuda").to(torch.bfloat16)
    vp = torch.randn((20, hkv, ps, 128), device="cuda").to(torch.bfloat16)
    binding.copy_pages(kp, vp, torch.from_numpy(cow).cuda(), P % ps)
    shared_k = kp[ids[:3]].clone()
    shared_v = vp[ids[:3]].clone()
    k_new = torch.randn((3 * 5, hkv, 128), device="cuda").to(torch.bfloat16)
    v_new = torch.randn((3 * 5, hkv, 128), device="cuda").to(torch.bfloat16)
    binding.kv_append(k_new, v_new, kp, vp, torch.from_numpy(table).cuda(), P, S, [5, 5, 5], ps)
    assert binding.last_error() == binding.OK
    assert torch.equal(kp[ids[:3]], shared_k) and torch.equal(vp[ids[:3]], shared_v)
    for b in range(3):  # new token t of branch b at position 40 + t: the branch's own page 2
        own = int(table[b, 2])
        assert torch.equal(kp[own, :, 8:13], k_new[5 * b:5 * b + 5].transpose(0, 1))

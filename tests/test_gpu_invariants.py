"""GPU invariants the pages fix: determinism, page-placement invariance,
batching invariance, split invariance, one-token causal == non-causal,
identical keys -> mean of V; plus the merge kernel against the oracle's merge
and the edge cases (empty problem, branches without rows)."""
import numpy as np
import pytest
import torch

import oracle
from shared_prefix_fan_gb300 import binding
from shared_prefix_fan_gb300.workloads import WORKLOADS, draw, small_spec
from tests.gpu_helpers import DevWorkload, compare, oracle_ref, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_deterministic_bitwise():
    dw = DevWorkload(draw(WORKLOADS["batching"]))
    o0, l0 = dw.run()
    for _ in range(2):
        o, l = dw.run()
        assert torch.equal(o, o0) and torch.equal(l, l0)


def test_page_placement_bitwise():
    w = draw(small_spec(h_q=16, h_kv=2, page_size=16, prefix_len=512, q_rows=[4, 9],
                        suffix_lens=[70, 300], seed=9))
    dw = DevWorkload(w)
    o0, l0 = dw.run()
    n = dw.k.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(1))
    inv = torch.argsort(perm)
    k2, v2 = dw.k[perm.cuda()].contiguous(), dw.v[perm.cuda()].contiguous()
    t = dw.table.long()
    t2 = torch.where(t >= 0, inv.cuda()[t.clamp(min=0)], t).to(torch.int32).contiguous()
    o1, l1 = dw.run(table=t2, k=k2, v=v2)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_batched_equals_per_branch():
    w = draw(small_spec(h_q=64, h_kv=8, page_size=64, prefix_len=2048, q_rows=[5, 20, 1, 12],
                        suffix_lens=[64, 256, 100, 12], seed=12))
    dw = DevWorkload(w)
    ob, lb = dw.run()
    r0 = 0
    for b in range(w.num_branches):
        T = int(w.q_rows[b])
        s = w.spec
        o, l = binding.attn(dw.q[r0:r0 + T].contiguous(), dw.k, dw.v,
                            dw.table[b:b + 1].contiguous(), s.prefix_len, [w.suffix_lens[b]], [T],
                            s.h_q, s.h_kv, s.page_size, s.scale, s.causal)
        assert binding.last_error() == binding.OK
        d = (o - ob[r0:r0 + T]).abs().max().item()
        assert d <= 2e-3, d
        assert (l - lb[r0:r0 + T]).abs().max().item() <= 1e-4
        r0 += T


def test_split_invariance():
    dw = DevWorkload(draw(WORKLOADS["decode"]))
    try:
        binding.set_option(binding.OPT_SPLITS, 1)
        o1, l1 = dw.run()
        binding.set_option(binding.OPT_SPLITS, 7)
        o7, l7 = dw.run()
    finally:
        binding.set_option(binding.OPT_SPLITS, 0)
    assert (o1 - o7).abs().max().item() <= 1e-4
    assert (l1 - l7).abs().max().item() <= 1e-4


@pytest.mark.parametrize("name", ["decode", "batching", "tiny"])
def test_fused_merge_equals_separate_merge(name):
    """The merge inside the attention kernel (grid flags, cooperative launch) and
    the separate merge kernel run the same per-row fold on the same partials:
    bitwise equal, and both match the oracle."""
    w = draw(WORKLOADS[name])
    dw = DevWorkload(w)
    try:
        binding.set_option(binding.OPT_FUSED_MERGE, 0)
        o_sep, l_sep = dw.run()
        binding.set_option(binding.OPT_FUSED_MERGE, 1)
        o_fused, l_fused = dw.run()
        o_again, l_again = dw.run()   # next epoch on the same flags
    finally:
        binding.set_option(binding.OPT_FUSED_MERGE, 0)
    assert torch.equal(o_sep, o_fused) and torch.equal(l_sep, l_fused)
    assert torch.equal(o_fused, o_again) and torch.equal(l_fused, l_again)
    compare(o_fused, l_fused, *oracle_ref(w), what=name + " fused merge")


def test_grid_larger_than_device_merges_separately():
    """A plan for more CTAs than the device holds at once cannot be launched
    cooperatively: the separate merge kernel runs instead, same results."""
    w = draw(WORKLOADS["decode"])
    dw = DevWorkload(w)
    o0, l0 = dw.run()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    try:
        binding.set_option(binding.OPT_NUM_SMS, 2 * sms)
        o1, l1 = dw.run()
    finally:
        binding.set_option(binding.OPT_NUM_SMS, 0)
    assert binding.last_error() == binding.OK
    assert (o1 - o0).abs().max().item() <= 1e-4
    assert (l1 - l0).abs().max().item() <= 1e-4


def test_single_token_causal_equals_noncausal():
    dw = DevWorkload(draw(WORKLOADS["decode"]))
    oc, lc = dw.run(causal=True)
    on, ln = dw.run(causal=False)
    assert torch.equal(oc, on) and torch.equal(lc, ln)


def test_identical_keys_give_mean_of_v():
    spec = small_spec(h_q=8, h_kv=1, page_size=16, prefix_len=256, q_rows=[3, 5],
                      suffix_lens=[40, 77], seed=4)
    w = draw(spec)
    w.k_pool[:] = w.k_pool[0, 0, 0][None, None, None, :]
    dw = DevWorkload(w)
    out, lse = dw.run()
    table = dw.table_host
    ps, P = spec.page_size, spec.prefix_len
    from shared_prefix_fan_gb300.workloads import bf16_bits_to_f32
    v = bf16_bits_to_f32(w.v_pool).astype(np.float64)
    r = 0
    for b in range(w.num_branches):
        n_all = P + int(w.suffix_lens[b])
        for t in range(int(w.q_rows[b])):
            n_vis = n_all - int(w.q_rows[b]) + t + 1
            keys = np.arange(n_vis)
            vs = v[table[b, keys // ps], 0, keys % ps]
            got = out[r].double().cpu().numpy()
            assert np.abs(got - vs.mean(0)[None]).max() <= 2e-3
            r += 1


def test_merge_kernel_matches_oracle_merge():
    rng = np.random.default_rng(0)
    n_parts, n, d = 5, 300, 128
    m = rng.normal(0, 3, size=(n_parts, n))
    l = rng.uniform(0.5, 40, size=(n_parts, n))
    l[1, ::7] = 0.0          # empty shards
    m[1, ::7] = -np.inf
    o = rng.normal(size=(n_parts, n, d)) * l[..., None]
    ml = np.stack([m / np.log(2), l], -1).astype(np.float32)   # kernel keeps m in log2 units
    po = torch.from_numpy(o.astype(np.float32)).cuda()
    pml = torch.from_numpy(ml).cuda()
    out, lse = binding.lse_merge(po, pml)
    torch.cuda.synchronize()
    # oracle on the fp32-rounded partials, natural-log domain
    m32 = ml[..., 0].astype(np.float64) * np.log(2)
    ro, rl = oracle.merge(m32, ml[..., 1].astype(np.float64), o.astype(np.float32).astype(np.float64))
    assert np.abs(out.double().cpu().numpy() - ro).max() <= 1e-5
    assert np.abs(lse.double().cpu().numpy() - rl).max() <= 1e-5


def test_empty_and_rowless_branches():
    spec = small_spec(h_q=8, h_kv=2, page_size=16, prefix_len=64, q_rows=[0, 0],
                      suffix_lens=[5, 9], seed=2)
    w = draw(spec)
    dw = DevWorkload(w)
    out, lse = dw.run()
    assert out.shape[0] == 0
    spec = small_spec(h_q=8, h_kv=2, page_size=16, prefix_len=64, q_rows=[0, 6, 0],
                      suffix_lens=[5, 9, 30], seed=3)
    w = draw(spec)
    out, lse = DevWorkload(w).run()
    compare(out, lse, *oracle_ref(w), what="row-less branches")


def test_two_threads_on_two_streams():
    """Two host threads call fanout_attn at the same time, each on its own
    stream (so each uses its own workspace and plan cache, under its own lock):
    every result equals the single-threaded result bit for bit."""
    import threading

    dws = [DevWorkload(draw(WORKLOADS["batching"])),
           DevWorkload(draw(small_spec(h_q=16, h_kv=2, page_size=32, prefix_len=512,
                                       q_rows=[5, 9, 3], suffix_lens=[70, 200, 33], seed=31)))]
    refs = [dw.run() for dw in dws]
    streams = [torch.cuda.Stream() for _ in dws]
    results, errors = {}, []

    def worker(k):
        try:
            with torch.cuda.stream(streams[k]):
                for _ in range(6):
                    results[k] = dws[k].run(stream=streams[k])
        except Exception as e:  # noqa: BLE001 -- reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(len(dws))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for k, (o, l) in enumerate(refs):
        assert torch.equal(results[k][0], o) and torch.equal(results[k][1], l)


@pytest.mark.parametrize("fused", [0, 1], ids=["separate_merge", "fused_merge"])
def test_without_lse(fused):
    """lse = NULL (a caller that needs only out): the same out, bit for bit,
    from the merge (separate and fused) and from units written directly."""
    specs = [
        small_spec(h_q=16, h_kv=2, page_size=16, prefix_len=1024, q_rows=[3, 9, 1],
                   suffix_lens=[200, 45, 700], seed=61),             # split: partials + merge
        small_spec(h_q=16, h_kv=2, page_size=64, prefix_len=0, q_rows=[300],
                   suffix_lens=[300], seed=62),                      # one branch: direct units
    ]
    try:
        binding.set_option(binding.OPT_FUSED_MERGE, fused)
        for spec in specs:
            dw = DevWorkload(draw(spec))
            s = dw.w.spec
            ref_out, _ = dw.run()
            out, lse = binding.attn(dw.q, dw.k, dw.v, dw.table, s.prefix_len, dw.w.suffix_lens,
                                    dw.w.q_rows, s.h_q, s.h_kv, s.page_size, s.scale, s.causal,
                                    want_lse=False)
            assert lse is None and binding.last_error() == binding.OK
            assert torch.equal(out, ref_out)
    finally:
        binding.set_option(binding.OPT_FUSED_MERGE, 0)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_lazy_rescale_every_tile(causal):
    """Scores that rise by about 70 every 128 keys (keys along one direction u
    with a magnitude growing with their position, queries along u): each tile's
    row max passes the reference by more than 2^8, so O is rescaled in TMEM on
    every tile and every split starts from its own reference. Against the
    oracle on the same bf16 inputs."""
    import dataclasses
    spec = small_spec(h_q=16, h_kv=2, page_size=64, prefix_len=1024, q_rows=[2, 5],
                      suffix_lens=[300, 520], causal=causal, permute_prefix=True,
                      permute_suffix=True, seed=71)
    w = draw(spec)
    s = w.spec
    d = s.d
    rng = np.random.default_rng(0)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    R = w.total_rows
    q = 8.0 * u[None, None, :] + 0.1 * rng.standard_normal((R, s.h_q, d))
    table = oracle.fork(w.prefix_pages, w.suffix_lens, s.page_size, w.free_pages,
                        w.max_pages_per_branch)
    k = w.k_pool.copy()
    # the shared prefix pages hold one set of keys for every branch
    noise_prefix = 0.1 * rng.standard_normal((s.h_kv, s.prefix_len, d))
    for b in range(w.num_branches):
        n = s.prefix_len + int(w.suffix_lens[b])
        j = np.arange(n)
        base = (70.0 / (128 * 8.0)) * j[:, None] * u[None, :]          # score ~ 0.55 j
        for h in range(s.h_kv):
            vals = base.copy()
            vals[:s.prefix_len] += noise_prefix[h]
            vals[s.prefix_len:] += 0.1 * rng.standard_normal((n - s.prefix_len, d))
            k[table[b, j // s.page_size], h, j % s.page_size, :] = _bf16_bits(vals)
    w2 = dataclasses.replace(w, q=_bf16_bits(q), k_pool=k)
    out, lse = DevWorkload(w2).run()
    compare(out, lse, *oracle_ref(w2), what=f"rescale every tile, causal={causal}")

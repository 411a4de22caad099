"""fanout_fork (product, C++) against the oracle's fork (C): bit-exact (CPU only)."""
import numpy as np
import pytest

import oracle
from shared_prefix_fan_gb300 import binding, build
from shared_prefix_fan_gb300.workloads import WORKLOADS, draw, small_spec


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("name", ["tiny", "decode", "batching", "wide"])
def test_fork_matches_oracle(name):
    spec = WORKLOADS[name]
    w = draw(spec) if name != "wide" else draw(spec)
    mp = w.max_pages_per_branch
    got = binding.fork(w.prefix_pages, w.suffix_lens, spec.page_size, w.free_pages, mp)
    ref = oracle.fork(w.prefix_pages, w.suffix_lens, spec.page_size, w.free_pages, mp)
    assert np.array_equal(got, ref)
    n_pre = spec.prefix_len // spec.page_size
    assert (got[:, :n_pre] == w.prefix_pages[None]).all()


def test_fork_edge_cases():
    # zero branches, zero-length suffixes, exact-fit free list
    assert binding.fork([1, 2], [], 16, [], 4).shape == (0, 4)
    t = binding.fork([5], [0, 16, 17], 16, [9, 8, 7], 3)
    assert t.tolist() == [[5, -1, -1], [5, 9, -1], [5, 8, 7]]
    with pytest.raises(binding.FanoutError):
        binding.fork([5], [40], 16, [1, 2], 4)   # free list too short
    with pytest.raises(binding.FanoutError):
        binding.fork([5], [40], 16, [1, 2, 3], 3)  # row too narrow


def test_fork_small_random():
    rng = np.random.default_rng(3)
    for _ in range(20):
        B = int(rng.integers(0, 6))
        ps = int(rng.choice([16, 32, 64]))
        S = rng.integers(0, 200, size=B)
        n_pre = int(rng.integers(0, 5))
        need = sum((int(s) + ps - 1) // ps for s in S)
        ids = rng.permutation(n_pre + need + 3).astype(np.int32)
        mp = n_pre + max([(int(s) + ps - 1) // ps for s in S] + [0]) + int(rng.integers(0, 3))
        got = binding.fork(ids[:n_pre], S, ps, ids[n_pre:], mp)
        ref = oracle.fork(ids[:n_pre], S, ps, ids[n_pre:], mp) if B else got
        assert np.array_equal(got, ref)

"""fanout_extend (product, C++) against the oracle's page-table growth: bit-exact;
and host-side validation of the append entry points (CPU only)."""
import ctypes

import numpy as np
import pytest

import oracle
from shared_prefix_fan_gb300 import binding, build


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("seed", range(12))
def test_extend_matches_oracle(seed):
    """Odd seeds: a prefix ending inside a page, forked with copy-on-write."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 7))
    ps = int(rng.choice([16, 32, 64]))
    P = int(rng.integers(0, 4)) * ps + (int(rng.integers(1, ps)) if seed % 2 else 0)
    n_pre = -(-P // ps)
    S = rng.integers(0, 150, size=B)
    T = rng.integers(0, 90, size=B)
    ids = rng.permutation(4000).astype(np.int32)
    mp = int(max(-(-(P + s + t) // ps) for s, t in zip(S, T))) + int(rng.integers(0, 3))
    if P % ps:
        table, _, n_old = binding.fork_cow(ids[:n_pre], P, S, ps, ids[n_pre:], mp)
    else:
        n_old = sum((int(s) + ps - 1) // ps for s in S)
        table = binding.fork(ids[:n_pre], S, ps, ids[n_pre:], mp)
    free = ids[n_pre + n_old:]
    got, used = binding.extend(table, P, S, T, ps, free)
    ref, used_ref = oracle.extend(table, P, S, T, ps, free)
    assert np.array_equal(got, ref) and used == used_ref


def test_extend_rejects_without_touching_table():
    table = binding.fork([7], [16, 16], 16, [1, 2], 3)
    with pytest.raises(binding.FanoutError):
        binding.extend(table, 16, [16, 16], [40, 0], 16, [9])   # free list too short
    with pytest.raises(binding.FanoutError):
        binding.extend(table, 16, [16, 16], [60, 0], 16, [9, 10, 11, 12])  # row too narrow


def test_kv_append_rejects_bad_arguments_on_host():
    lib = binding.load()
    p32 = ctypes.POINTER(ctypes.c_int32)
    S = np.array([4, 4], np.int32)
    T = np.array([1, 1], np.int32)
    def rc(**kw):
        a = dict(k=1024, v=1024, kp=1024, vp=1024, pt=1024, P=16, B=2, mp=4, np_=8, hkv=2, d=128,
                 ps=16)
        a.update(kw)
        return lib.fanout_kv_append(a["k"], a["v"], a["kp"], a["vp"], a["pt"], a["P"],
                                    S.ctypes.data_as(p32), T.ctypes.data_as(p32), a["B"], a["mp"],
                                    a["np_"], a["hkv"], a["d"], a["ps"], None)
    assert rc(d=12) == binding.EUNSUPPORTED
    assert rc(B=2000) == binding.EUNSUPPORTED
    assert rc(mp=1) == binding.EINVAL          # rows too narrow for the grown suffix
    assert rc(k=None) == binding.EINVAL
    assert rc(kp=1032 + 2) == binding.EINVAL   # not 16-byte aligned


@pytest.mark.parametrize("seed", range(8))
def test_fork_cow_matches_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 6))
    ps = int(rng.choice([16, 32, 64]))
    P = int(rng.integers(0, 5 * ps))
    S = rng.integers(0, 150, size=B)
    n_pre = -(-P // ps)
    ids = rng.permutation(5000).astype(np.int32)
    mp = max(n_pre, max(-(-(P + int(s)) // ps) for s in S)) + int(rng.integers(0, 3))
    got_t, got_c, got_u = binding.fork_cow(ids[:n_pre], P, S, ps, ids[n_pre:], mp)
    ref_t, ref_c, ref_u = oracle.fork_cow(ids[:n_pre], P, S, ps, ids[n_pre:], mp)
    assert np.array_equal(got_t, ref_t) and got_u == ref_u
    if P % ps:
        assert np.array_equal(got_c, ref_c)
    else:  # page-aligned prefix: the ordinary fork
        assert np.array_equal(got_t, binding.fork(ids[:n_pre], S, ps, ids[n_pre:], mp))

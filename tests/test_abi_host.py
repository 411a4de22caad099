"""The C-ABI library on the host: it loads, exports what include/fanout.h
declares, and rejects bad arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import numpy as np
import pytest

from shared_prefix_fan_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "fanout.h")).read()
    return sorted(set(re.findall(r"FANOUT_API\s+(?:const\s+char\s*\*|int)\s*(fanout_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in binding.ABI, f"binding lacks {n}"
    assert set(binding.ABI) == set(names)


def test_strerror_and_version(lib):
    assert binding.version().count(".") == 2
    for code in range(6):
        assert lib.fanout_strerror(code)
    assert b"unknown" in lib.fanout_strerror(77)


def test_options_validated(lib):
    assert lib.fanout_set_option(binding.OPT_SPLITS, -1) == binding.EINVAL
    assert lib.fanout_set_option(99, 1) == binding.EINVAL
    assert lib.fanout_set_option(binding.OPT_WAIT_LIMIT_NS, 0) == binding.EINVAL
    assert lib.fanout_set_option(binding.OPT_SPLITS, 0) == binding.OK
    assert lib.fanout_set_option(binding.OPT_FUSED_MERGE, 2) == binding.EINVAL
    assert lib.fanout_set_option(binding.OPT_FUSED_MERGE, 0) == binding.OK
    assert lib.fanout_set_option(binding.OPT_FUSED_MERGE, 1) == binding.OK


def _device_visible() -> bool:
    """These tests pass made-up addresses; a call that passes validation would
    launch kernels on them, so such calls run only where no GPU is visible."""
    import torch
    return torch.cuda.is_available()


def _attn_rc(lib, **kw):
    a = dict(q=1024, k=1024, v=1024, pt=1024, P=64, S=[32, 32], T=[2, 2], B=2, maxp=8,
             npages=16, hq=8, hkv=2, d=128, ps=16, scale=0.088, causal=1, out=1024, od=0,
             lse=None)
    a.update(kw)
    S = np.asarray(a["S"], np.int32)
    T = np.asarray(a["T"], np.int32)
    p32 = ctypes.POINTER(ctypes.c_int32)
    return lib.fanout_attn(a["q"], a["k"], a["v"], a["pt"], a["P"], S.ctypes.data_as(p32),
                           T.ctypes.data_as(p32), a["B"], a["maxp"], a["npages"], a["hq"],
                           a["hkv"], a["d"], a["ps"], a["scale"], a["causal"], a["out"], a["od"],
                           a["lse"], None)


def test_attn_rejects_bad_arguments_on_host(lib):
    E, U = binding.EINVAL, binding.EUNSUPPORTED
    assert _attn_rc(lib, d=64) == U
    assert _attn_rc(lib, ps=24) == U
    if not _device_visible():   # accepted calls go on to launch: only with no GPU to launch on
        assert _attn_rc(lib, P=40) not in (E, U)   # a prefix ending inside a page is accepted
    assert _attn_rc(lib, hq=6, hkv=4) == E     # H_q not a multiple of H_kv
    assert _attn_rc(lib, hq=256, hkv=1) == U   # G > 128
    assert _attn_rc(lib, T=[40, 2]) == E       # causal: more new tokens than suffix
    assert _attn_rc(lib, S=[-1, 2]) == E
    assert _attn_rc(lib, q=None) == E
    assert _attn_rc(lib, q=1026) == E          # not 16-byte aligned
    assert _attn_rc(lib, maxp=2) == E          # table rows too narrow
    assert _attn_rc(lib, od=7) == E
    assert _attn_rc(lib, scale=0.0) == E
    assert _attn_rc(lib, scale=-0.1) == E
    assert _attn_rc(lib, P=0, S=[0, 4], T=[1, 1], causal=0) == E  # a row with no key
    assert _attn_rc(lib, S=[1 << 29, 2]) == U      # more than 2^29 keys in a branch
    assert _attn_rc(lib, T=[1 << 21, 2], S=[1 << 21, 2], causal=0) == U   # R * H_q > 2^24
    # nothing to do is not an error, and needs no device
    assert _attn_rc(lib, T=[0, 0], q=None, out=None) == binding.OK


def test_merge_rejects_bad_arguments_on_host(lib):
    assert lib.fanout_lse_merge(1024, 1024, 2, 10, 64, 1024, 0, None, None) == binding.EUNSUPPORTED
    assert lib.fanout_lse_merge(1024, 1024, -1, 10, 128, 1024, 0, None, None) == binding.EINVAL
    assert lib.fanout_lse_merge(None, 1024, 2, 10, 128, 1024, 0, None, None) == binding.EINVAL
    assert lib.fanout_lse_merge(None, None, 2, 0, 128, None, 0, None, None) == binding.OK


def test_selftest_rejects_bad_limit(lib):
    assert lib.fanout_selftest_wait_timeout(0, None) == binding.EINVAL


def test_read_floor_rejects_bad_arguments_on_host(lib):
    E = binding.EINVAL
    assert lib.fanout_read_floor(1032, 512, 2048, None) == E   # buffer not 16-byte aligned
    assert lib.fanout_read_floor(1024, 520, 2048, None) == E   # size not a multiple of 16
    assert lib.fanout_read_floor(1024, 0, 2048, None) == E
    assert lib.fanout_read_floor(1024, -16, 2048, None) == E
    assert lib.fanout_read_floor(None, 512, 2048, None) == E
    assert lib.fanout_read_floor(1024, 512, None, None) == E
    assert lib.fanout_read_floor(1024, 512, 2050, None) == E   # xor word not 4-byte aligned

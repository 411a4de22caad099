"""fp64 CPU oracle for shared-prefix fan-out attention (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the benchmark's CPU-baseline leg. The product path never imports this package.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over rows x heads);
this file only compiles it and marshals numpy arrays. See the header of
``oracle.c`` for the definitions it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags: Sequence[str] = ()) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", src, "-o", out, "-lm"]
    base[1:1] = list(extra_flags)
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    return out


def _stale(lib: str, src: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle library; a path loads a variant build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if _stale(_LIB, _SRC):
            build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _bind(lib):
    i32p = ctypes.POINTER(ctypes.c_int32)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i32, f64 = ctypes.c_int32, ctypes.c_double
    lib.oracle_fork.argtypes = [i32p, i32, i32, i32p, i32, i32p, i32, i32p, i32]
    lib.oracle_fork.restype = ctypes.c_int
    lib.oracle_attn.argtypes = [u16p, u16p, u16p, i32p, i32, i32, i32p, i32p, i32, i32, i32, i32,
                                i32, f64, ctypes.c_int, i32p, i32, f64p, f64p]
    lib.oracle_attn.restype = ctypes.c_int
    lib.oracle_attn_partial.argtypes = [u16p, u16p, u16p, i32p, i32, i32, i32p, i32p, i32, i32,
                                        i32, i32, i32, f64, ctypes.c_int, i32p, i32, i32, i32,
                                        f64p, f64p, f64p]
    lib.oracle_attn_partial.restype = ctypes.c_int
    lib.oracle_merge.argtypes = [f64p, f64p, f64p, i32, ctypes.c_int64, i32, f64p, f64p]
    lib.oracle_merge.restype = None
    lib.oracle_count_pairs.argtypes = [i32, i32p, i32p, i32, i32, ctypes.c_int]
    lib.oracle_count_pairs.restype = ctypes.c_int64
    lib.oracle_fork_cow.argtypes = [i32p, i32, i32, i32p, i32, i32p, i32, i32p, i32, i32p]
    lib.oracle_fork_cow.restype = ctypes.c_int
    lib.oracle_copy_pages.argtypes = [u16p, u16p, i32p, i32, i32, i32, i32, i32]
    lib.oracle_copy_pages.restype = None
    lib.oracle_extend.argtypes = [i32p, i32, i32, i32, i32p, i32p, i32, i32p, i32]
    lib.oracle_extend.restype = ctypes.c_int
    lib.oracle_kv_append.argtypes = [u16p, u16p, u16p, u16p, i32p, i32, i32, i32p, i32p, i32, i32,
                                     i32, i32]
    lib.oracle_kv_append.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def num_threads(lib=None) -> int:
    return int((lib or load()).oracle_num_threads())


def fork(prefix_pages, suffix_lens, page_size: int, free_pages, max_pages: int,
         lib=None) -> np.ndarray:
    """Branch page tables [B][max_pages] (-1 = unused)."""
    lib = lib or load()
    pre, sl, fr = _i32(prefix_pages), _i32(suffix_lens), _i32(free_pages)
    nb = int(sl.shape[0])
    table = np.full((max(nb, 1), max_pages), -1, dtype=np.int32)
    rc = lib.oracle_fork(_p(pre, ctypes.c_int32), int(pre.shape[0]), nb, _p(sl, ctypes.c_int32),
                         int(page_size), _p(fr, ctypes.c_int32), int(fr.shape[0]),
                         _p(table, ctypes.c_int32), int(max_pages))
    if rc != 0:
        raise ValueError("oracle_fork: free list or table width too small")
    return table[:nb]


def attn(q, k_pool, v_pool, table, prefix_len: int, suffix_lens, q_rows, h_q: int, h_kv: int,
         page_size: int, scale: float, causal: bool, rows=None, lib=None):
    """fp64 attention for the listed tokens (all when rows is None): (out, lse)."""
    lib = lib or load()
    q, k_pool, v_pool = (np.ascontiguousarray(a, dtype=np.uint16) for a in (q, k_pool, v_pool))
    table, sl, tq = _i32(table), _i32(suffix_lens), _i32(q_rows)
    d = int(q.shape[-1])
    n_total = int(tq.sum())
    rws = None if rows is None else _i32(rows)
    n = n_total if rws is None else int(rws.shape[0])
    out = np.empty((n, h_q, d), dtype=np.float64)
    lse = np.empty((n, h_q), dtype=np.float64)
    if n == 0:
        return out, lse
    rc = lib.oracle_attn(_p(q, ctypes.c_uint16), _p(k_pool, ctypes.c_uint16),
                         _p(v_pool, ctypes.c_uint16), _p(table, ctypes.c_int32),
                         int(table.shape[1]), int(prefix_len), _p(sl, ctypes.c_int32),
                         _p(tq, ctypes.c_int32), int(tq.shape[0]), int(h_q), int(h_kv), d,
                         int(page_size), float(scale), int(bool(causal)),
                         None if rws is None else _p(rws, ctypes.c_int32), n,
                         _p(out, ctypes.c_double), _p(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_attn failed ({rc})")
    return out, lse


def attn_partial(q, k_pool, v_pool, table, prefix_len: int, suffix_lens, q_rows, h_q: int,
                 h_kv: int, page_size: int, scale: float, causal: bool, lo: int, hi: int,
                 rows=None, lib=None):
    """Partial state (m, l, o) over keys [lo, hi) of each token's branch."""
    lib = lib or load()
    q, k_pool, v_pool = (np.ascontiguousarray(a, dtype=np.uint16) for a in (q, k_pool, v_pool))
    table, sl, tq = _i32(table), _i32(suffix_lens), _i32(q_rows)
    d = int(q.shape[-1])
    rws = None if rows is None else _i32(rows)
    n = int(tq.sum()) if rws is None else int(rws.shape[0])
    m = np.empty((n, h_q), dtype=np.float64)
    l = np.empty((n, h_q), dtype=np.float64)
    o = np.empty((n, h_q, d), dtype=np.float64)
    lib.oracle_attn_partial(_p(q, ctypes.c_uint16), _p(k_pool, ctypes.c_uint16),
                            _p(v_pool, ctypes.c_uint16), _p(table, ctypes.c_int32),
                            int(table.shape[1]), int(prefix_len), _p(sl, ctypes.c_int32),
                            _p(tq, ctypes.c_int32), int(tq.shape[0]), int(h_q), int(h_kv), d,
                            int(page_size), float(scale), int(bool(causal)),
                            None if rws is None else _p(rws, ctypes.c_int32), n, int(lo),
                            int(hi), _p(m, ctypes.c_double), _p(l, ctypes.c_double),
                            _p(o, ctypes.c_double))
    return m, l, o


def merge(parts_m, parts_l, parts_o, lib=None):
    """Fold partials in order with the pairwise merge: (out, lse).

    parts_m, parts_l: [n_parts, ...]; parts_o: [n_parts, ..., d].
    """
    lib = lib or load()
    pm = np.ascontiguousarray(parts_m, dtype=np.float64)
    pl = np.ascontiguousarray(parts_l, dtype=np.float64)
    po = np.ascontiguousarray(parts_o, dtype=np.float64)
    n_parts = int(pm.shape[0])
    lead = pm.shape[1:]
    n = int(np.prod(lead)) if lead else 1
    d = int(po.shape[-1])
    out = np.empty(lead + (d,), dtype=np.float64)
    lse = np.empty(lead, dtype=np.float64)
    lib.oracle_merge(_p(pm, ctypes.c_double), _p(pl, ctypes.c_double), _p(po, ctypes.c_double),
                     n_parts, n, d, _p(out, ctypes.c_double), _p(lse, ctypes.c_double))
    return out, lse


def count_pairs(prefix_len: int, suffix_lens, q_rows, h_q: int, causal: bool, lib=None) -> int:
    """Visible (token, query head, key) triples; attention flops = 4 d x this."""
    lib = lib or load()
    sl, tq = _i32(suffix_lens), _i32(q_rows)
    return int(lib.oracle_count_pairs(int(prefix_len), _p(sl, ctypes.c_int32),
                                      _p(tq, ctypes.c_int32), int(tq.shape[0]), int(h_q),
                                      int(bool(causal))))


def fork_cow(prefix_pages, prefix_len: int, suffix_lens, page_size: int, free_pages,
             max_pages: int, lib=None):
    """(tables [B][max_pages], cow pairs [B][2], free pages used)."""
    lib = lib or load()
    pre, sl, fr = _i32(prefix_pages), _i32(suffix_lens), _i32(free_pages)
    nb = int(sl.shape[0])
    table = np.full((max(nb, 1), max_pages), -1, dtype=np.int32)
    cow = np.full((max(nb, 1), 2), -1, dtype=np.int32)
    used = lib.oracle_fork_cow(_p(pre, ctypes.c_int32), int(prefix_len), nb,
                               _p(sl, ctypes.c_int32), int(page_size), _p(fr, ctypes.c_int32),
                               int(fr.shape[0]), _p(table, ctypes.c_int32), int(max_pages),
                               _p(cow, ctypes.c_int32))
    if used < 0:
        raise ValueError("oracle_fork_cow: free list or table width too small")
    return table[:nb], cow[:nb], int(used)


def copy_pages(k_pool, v_pool, pairs, rows: int, lib=None):
    """Copies of the pools with token slots [0, rows) of each pair's page copied."""
    lib = lib or load()
    kp, vp = (np.array(a, dtype=np.uint16, copy=True, order="C") for a in (k_pool, v_pool))
    pr = _i32(pairs).reshape(-1, 2)
    _, h_kv, page, d = kp.shape
    lib.oracle_copy_pages(_p(kp, ctypes.c_uint16), _p(vp, ctypes.c_uint16),
                          _p(pr, ctypes.c_int32), int(pr.shape[0]), int(rows), int(h_kv),
                          int(page), int(d))
    return kp, vp


def extend(table, prefix_len: int, suffix_lens, add_lens, page_size: int, free_pages,
           lib=None):
    """Grown copy of the page tables and the number of free pages used."""
    lib = lib or load()
    t = np.array(table, dtype=np.int32, copy=True, order="C")
    sl, al, fr = _i32(suffix_lens), _i32(add_lens), _i32(free_pages)
    used = lib.oracle_extend(_p(t, ctypes.c_int32), int(t.shape[0]), int(t.shape[1]),
                             int(prefix_len), _p(sl, ctypes.c_int32), _p(al, ctypes.c_int32),
                             int(page_size), _p(fr, ctypes.c_int32), int(fr.shape[0]))
    if used < 0:
        raise ValueError("oracle_extend: free list or table width too small")
    return t, int(used)


def kv_append(k_new, v_new, k_pool, v_pool, table, prefix_len: int, suffix_lens, add_lens,
              lib=None):
    """Pools with the new rows written (copies; inputs untouched)."""
    lib = lib or load()
    kn, vn = (np.ascontiguousarray(a, dtype=np.uint16) for a in (k_new, v_new))
    kp, vp = (np.array(a, dtype=np.uint16, copy=True, order="C") for a in (k_pool, v_pool))
    t, sl, al = _i32(table), _i32(suffix_lens), _i32(add_lens)
    _, h_kv, page, d = kp.shape
    lib.oracle_kv_append(_p(kn, ctypes.c_uint16), _p(vn, ctypes.c_uint16), _p(kp, ctypes.c_uint16),
                         _p(vp, ctypes.c_uint16), _p(t, ctypes.c_int32), int(t.shape[1]),
                         int(prefix_len), _p(sl, ctypes.c_int32), _p(al, ctypes.c_int32),
                         int(t.shape[0]), int(h_kv), int(d), int(page))
    return kp, vp


def run_workload(w, rows=None, lib=None):
    """Oracle result for a drawn workload (see the shared input generator)."""
    s = w.spec
    table = fork(w.prefix_pages, w.suffix_lens, s.page_size, w.free_pages,
                 w.max_pages_per_branch, lib=lib)
    return attn(w.q, w.k_pool, w.v_pool, table, s.prefix_len, w.suffix_lens, w.q_rows, s.h_q,
                s.h_kv, s.page_size, s.scale, s.causal, rows=rows, lib=lib)


if __name__ == "__main__":  # pragma: no cover
    print(build(), file=sys.stderr)

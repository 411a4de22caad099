"""Python binding of libfanout.so (ctypes): argument marshalling only.

Every step of the attention path runs in the library's CUDA kernels; this
module turns torch tensors into pointers, checks dtypes/devices/shapes, calls
the C ABI and raises on a non-zero status. There is no fallback: if the
library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libfanout.so")

OK, EINVAL, EUNSUPPORTED, ECUDA, ENOMEM, ETIMEOUT = range(6)
OUT_F32, OUT_BF16 = 0, 1
OPT_SPLITS, OPT_VALIDATE_TABLE, OPT_WAIT_LIMIT_NS, OPT_NUM_SMS, OPT_FUSED_MERGE = 1, 2, 3, 4, 5

# The C ABI (include/fanout.h): name -> (restype, argtypes)
_i32, _i64, _f32, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
ABI = {
    "fanout_fork": (ctypes.c_int, [_i32p, _i32, _i32, _i32p, _i32, _i32p, _i32, _i32p, _i32]),
    "fanout_fork_cow": (ctypes.c_int, [_i32p, _i32, _i32, _i32p, _i32, _i32p, _i32, _i32p, _i32,
                                       _i32p, _i32p]),
    "fanout_copy_pages": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp]),
    "fanout_extend": (ctypes.c_int, [_i32p, _i32, _i32, _i32, _i32p, _i32p, _i32, _i32p, _i32,
                                     _i32p]),
    "fanout_kv_append": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, _i32p, _i32p, _i32, _i32,
                                        _i32, _i32, _i32, _i32, _vp]),
    "fanout_attn": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32p, _i32p, _i32, _i32, _i32, _i32,
                                   _i32, _i32, _i32, _f32, _i32, _vp, _i32, _vp, _vp]),
    "fanout_attn_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32p, _i32p, _i32, _i32,
                                           _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp, _i32,
                                           _vp, _vp]),
    "fanout_lse_merge": (ctypes.c_int, [_vp, _vp, _i32, _i64, _i32, _vp, _i32, _vp, _vp]),
    "fanout_last_error": (ctypes.c_int, [_vp]),
    "fanout_last_error_detail": (ctypes.c_int, [_vp, _i32p, _i32p]),
    "fanout_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "fanout_set_option": (ctypes.c_int, [_i32, _i64]),
    "fanout_set_profile_events": (ctypes.c_int, [_vp, _vp]),
    "fanout_plan": (ctypes.c_int, [_i32p, _i32p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32p,
                                   _i32, _i32p, _i32p, _i32, _i32p, _i32p]),
    "fanout_plan_step": (ctypes.c_int, [_i32p, _i32p, _i32p, _i32, _i32, _i32, _i32, _i32, _i32,
                                        _i32, _i32p, _i32, _i32p, _i32p, _i32, _i32p, _i32p,
                                        _i32p]),
    "fanout_selftest_wait_timeout": (ctypes.c_int, [_i64, _vp]),
    "fanout_read_floor": (ctypes.c_int, [_vp, _i64, _vp, _vp]),
    "fanout_release": (ctypes.c_int, []),
    "fanout_version": (ctypes.c_char_p, []),
}

_lib = None


class FanoutError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


def load(path: Optional[str] = None):
    """Load libfanout.so (built by shared_prefix_fan_gb300.build). Raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libfanout.so not built ({p}); run shared_prefix_fan_gb300.build.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in ABI.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    if path is None:
        _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().fanout_strerror(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise FanoutError(rc, what)


def _i32arr(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_i32p)


def version() -> str:
    return load().fanout_version().decode()


def fork(prefix_pages, suffix_lens, page_size: int, free_pages, max_pages: int) -> np.ndarray:
    """Branch page tables (host): row b = prefix ids + branch b's private ids, then -1."""
    pre, sl, fr = _i32arr(prefix_pages), _i32arr(suffix_lens), _i32arr(free_pages)
    nb = int(sl.shape[0])
    table = np.full((max(nb, 1), int(max_pages)), -1, dtype=np.int32)
    _check(load().fanout_fork(_ptr(pre), int(pre.shape[0]), nb, _ptr(sl), int(page_size),
                              _ptr(fr), int(fr.shape[0]), _ptr(table), int(max_pages)),
           "fanout_fork")
    return table[:nb]


def fork_cow(prefix_pages, prefix_len: int, suffix_lens, page_size: int, free_pages,
             max_pages: int):
    """Fork with a prefix that may end inside a page: (tables, cow_pairs [B, 2], used)."""
    pre, sl, fr = _i32arr(prefix_pages), _i32arr(suffix_lens), _i32arr(free_pages)
    nb = int(sl.shape[0])
    table = np.full((max(nb, 1), int(max_pages)), -1, dtype=np.int32)
    pairs = np.full((max(nb, 1), 2), -1, dtype=np.int32)
    used = ctypes.c_int32(0)
    _check(load().fanout_fork_cow(_ptr(pre), int(prefix_len), nb, _ptr(sl), int(page_size),
                                  _ptr(fr), int(fr.shape[0]), _ptr(table), int(max_pages),
                                  _ptr(pairs), ctypes.byref(used)), "fanout_fork_cow")
    return table[:nb], pairs[:nb], int(used.value)


def copy_pages(k_pages, v_pages, pairs, rows: int, stream=None) -> None:
    """Device copy of token slots [0, rows) for page pairs (int32 [n, 2] on the device)."""
    n, h_kv, page, d = (int(x) for x in k_pages.shape)
    _check(load().fanout_copy_pages(k_pages.data_ptr(), v_pages.data_ptr(), pairs.data_ptr(),
                                    int(pairs.shape[0]), int(rows), n, h_kv, d, page,
                                    _stream_handle(stream)), "fanout_copy_pages")


def extend(page_table, prefix_len: int, suffix_lens, add_lens, page_size: int, free_pages):
    """Grown copy of host page tables [B][max_pages] and the free pages used."""
    t = np.array(page_table, dtype=np.int32, copy=True, order="C")
    sl, al, fr = _i32arr(suffix_lens), _i32arr(add_lens), _i32arr(free_pages)
    used = ctypes.c_int32(0)
    _check(load().fanout_extend(_ptr(t), int(t.shape[0]), int(t.shape[1]), int(prefix_len),
                                _ptr(sl), _ptr(al), int(page_size), _ptr(fr), int(fr.shape[0]),
                                ctypes.byref(used)), "fanout_extend")
    return t, int(used.value)


def kv_append(k_new, v_new, k_pages, v_pages, page_table, prefix_len: int, suffix_lens,
              add_lens, page_size: int, stream=None) -> None:
    """Write new K/V rows [R, H_kv, d] (bf16, device) into the page pools in place."""
    import torch
    for name, t in (("k_new", k_new), ("v_new", v_new), ("k_pages", k_pages),
                    ("v_pages", v_pages)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    sl, al = _i32arr(suffix_lens), _i32arr(add_lens)
    _check(load().fanout_kv_append(
        k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
        page_table.data_ptr(), int(prefix_len), _ptr(sl), _ptr(al), int(sl.shape[0]),
        int(page_table.shape[1]), int(k_pages.shape[0]), int(k_pages.shape[1]),
        int(k_pages.shape[3]), int(page_size), _stream_handle(stream)), "fanout_kv_append")


def plan(suffix_lens, q_rows, prefix_len: int, h_q: int, h_kv: int, page_size: int,
         causal: bool, num_sms: int = 152) -> Tuple[np.ndarray, np.ndarray, int]:
    """The work plan fanout_attn would run: (units [n, 8], cta_first [n_cta+1], n_parts)."""
    sl, tq = _i32arr(suffix_lens), _i32arr(q_rows)
    lib = load()
    n_units, n_ctas, n_parts = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    args = (_ptr(sl), _ptr(tq), int(sl.shape[0]), int(prefix_len), int(h_q), int(h_kv),
            int(page_size), int(bool(causal)), int(num_sms))
    _check(lib.fanout_plan(*args, None, 0, ctypes.byref(n_units), None, 0, ctypes.byref(n_ctas),
                           ctypes.byref(n_parts)), "fanout_plan")
    units = np.zeros((max(n_units.value, 1), 8), dtype=np.int32)
    cta = np.zeros(n_ctas.value + 1, dtype=np.int32)
    _check(lib.fanout_plan(*args, _ptr(units), int(units.shape[0]), ctypes.byref(n_units),
                           _ptr(cta), int(cta.shape[0]), ctypes.byref(n_ctas),
                           ctypes.byref(n_parts)), "fanout_plan")
    return units[:n_units.value], cta, int(n_parts.value)


def plan_step(prev_suffix_lens, suffix_lens, q_rows, prefix_len: int, h_q: int, h_kv: int,
              page_size: int, causal: bool, num_sms: int = 152):
    """The plan fanout_attn runs after a call that differed only in suffix
    lengths: (units [n, 8], cta_first [n_cta+1], n_parts, reused)."""
    ps_, sl, tq = _i32arr(prev_suffix_lens), _i32arr(suffix_lens), _i32arr(q_rows)
    lib = load()
    n_units, n_ctas, n_parts, reused = (ctypes.c_int32(0) for _ in range(4))
    args = (_ptr(ps_), _ptr(sl), _ptr(tq), int(sl.shape[0]), int(prefix_len), int(h_q),
            int(h_kv), int(page_size), int(bool(causal)), int(num_sms))
    _check(lib.fanout_plan_step(*args, None, 0, ctypes.byref(n_units), None, 0,
                                ctypes.byref(n_ctas), ctypes.byref(n_parts), None),
           "fanout_plan_step")
    units = np.zeros((max(n_units.value, 1), 8), dtype=np.int32)
    cta = np.zeros(n_ctas.value + 1, dtype=np.int32)
    _check(lib.fanout_plan_step(*args, _ptr(units), int(units.shape[0]), ctypes.byref(n_units),
                                _ptr(cta), int(cta.shape[0]), ctypes.byref(n_ctas),
                                ctypes.byref(n_parts), ctypes.byref(reused)), "fanout_plan_step")
    return units[:n_units.value], cta, int(n_parts.value), bool(reused.value)


def set_option(option: int, value: int) -> None:
    _check(load().fanout_set_option(int(option), int(value)), "fanout_set_option")


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def attn(q, k_pages, v_pages, page_table, prefix_len: int, suffix_lens: Sequence[int],
         q_rows: Sequence[int], h_q: int, h_kv: int, page_size: int, scale: float,
         causal: bool, out=None, lse=None, out_dtype: str = "f32", want_lse: bool = True,
         stream=None):
    """Fan-out attention through fanout_attn. Device tensors in, (out, lse) back.

    q: bf16 [R, H_q, d]; k_pages / v_pages: bf16 [num_pages, H_kv, page, d];
    page_table: int32 [B, max_pages] on the same device; suffix_lens / q_rows:
    host sequences of length B. `out` / `lse` are allocated when not given.
    """
    import torch
    lib = load()
    sl, tq = _i32arr(suffix_lens), _i32arr(q_rows)
    R = int(tq.sum())
    d = int(q.shape[-1])
    dev = q.device
    for name, t, dt in (("q", q, torch.bfloat16), ("k_pages", k_pages, torch.bfloat16),
                        ("v_pages", v_pages, torch.bfloat16), ("page_table", page_table, torch.int32)):
        if t.dtype != dt or t.device != dev or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor on {dev}")
    if tuple(q.shape) != (R, h_q, d):
        raise ValueError(f"q shape {tuple(q.shape)} != {(R, h_q, d)}")
    if k_pages.shape != v_pages.shape or k_pages.dim() != 4:
        raise ValueError("k_pages / v_pages must be [num_pages, H_kv, page, d]")
    odt = {"f32": (torch.float32, OUT_F32), "bf16": (torch.bfloat16, OUT_BF16)}[out_dtype]
    if out is None:
        out = torch.empty((R, h_q, d), dtype=odt[0], device=dev)
    if lse is None and want_lse:
        lse = torch.empty((R, h_q), dtype=torch.float32, device=dev)
    if out.dtype != odt[0] or not out.is_contiguous():
        raise ValueError("out dtype/layout mismatch")
    rc = lib.fanout_attn(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                         page_table.data_ptr(), int(prefix_len), _ptr(sl), _ptr(tq),
                         int(sl.shape[0]), int(page_table.shape[1]) if page_table.dim() == 2 else 0,
                         int(k_pages.shape[0]), int(h_q), int(h_kv), d, int(page_size),
                         float(scale), int(bool(causal)), out.data_ptr(), odt[1],
                         lse.data_ptr() if lse is not None else None, _stream_handle(stream))
    _check(rc, "fanout_attn")
    return out, lse


# Fixed scratch of fanout_attn_noalloc (FANOUT_NOALLOC_SCRATCH_BYTES in include/fanout.h).
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def attn_noalloc(q, k_pages, v_pages, page_table, prefix_len: int, suffix_lens, q_rows,
                 h_q: int, h_kv: int, page_size: int, scale: float, causal: bool, out, lse,
                 out_dtype: str = "f32", stream=None) -> int:
    """fanout_attn_noalloc: same call as attn() into caller-allocated out/lse,
    for callers that must not allocate device memory during a call (the library
    uses its fixed scratch array instead of a cudaMalloc'd workspace). Returns
    the status code (FANOUT_ENOMEM when the problem needs more scratch than the
    fixed array holds) instead of raising, and allocates nothing itself."""
    sl, tq = _i32arr(suffix_lens), _i32arr(q_rows)
    odt = {"f32": OUT_F32, "bf16": OUT_BF16}[out_dtype]
    return int(load().fanout_attn_noalloc(
        q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), page_table.data_ptr(),
        int(prefix_len), _ptr(sl), _ptr(tq), int(sl.shape[0]), int(page_table.shape[1]),
        int(k_pages.shape[0]), int(h_q), int(h_kv), int(q.shape[-1]), int(page_size),
        float(scale), int(bool(causal)), out.data_ptr(), odt,
        lse.data_ptr() if lse is not None else None, _stream_handle(stream)))


def lse_merge(part_o, part_ml, out=None, lse=None, out_dtype: str = "f32", stream=None):
    """Merge partials: part_o fp32 [P, N, d], part_ml fp32 [P, N, 2] -> (out [N, d], lse [N])."""
    import torch
    n_parts, n_out, d = (int(x) for x in part_o.shape)
    odt = {"f32": (torch.float32, OUT_F32), "bf16": (torch.bfloat16, OUT_BF16)}[out_dtype]
    if out is None:
        out = torch.empty((n_out, d), dtype=odt[0], device=part_o.device)
    if lse is None:
        lse = torch.empty((n_out,), dtype=torch.float32, device=part_o.device)
    _check(load().fanout_lse_merge(part_o.data_ptr(), part_ml.data_ptr(), n_parts, n_out, d,
                                   out.data_ptr(), odt[1], lse.data_ptr(), _stream_handle(stream)),
           "fanout_lse_merge")
    return out, lse


def last_error(stream=None) -> int:
    return int(load().fanout_last_error(_stream_handle(stream)))


def last_error_detail(stream=None) -> Tuple[int, int, int]:
    """(status, wait site, CTA) of the device error word, then cleared."""
    site, block = ctypes.c_int32(0), ctypes.c_int32(0)
    rc = load().fanout_last_error_detail(_stream_handle(stream), ctypes.byref(site),
                                         ctypes.byref(block))
    return int(rc), int(site.value), int(block.value)


def set_profile_events(before=None, after=None) -> None:
    """Record torch.cuda.Event objects around the split-KV kernel (None, None: off)."""
    b = before.cuda_event if before is not None else None
    a = after.cuda_event if after is not None else None
    _check(load().fanout_set_profile_events(b, a), "fanout_set_profile_events")


def selftest_wait_timeout(limit_ns: int = 20_000_000, stream=None) -> int:
    return int(load().fanout_selftest_wait_timeout(int(limit_ns), _stream_handle(stream)))


def read_floor(buf, xor_out, stream=None) -> None:
    """One plain streaming read of the device tensor `buf` (all its bytes);
    *xor_out (a 1-element int32/uint32 CUDA tensor) ^= the xor of its words."""
    import torch
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    if not xor_out.is_cuda or xor_out.dtype not in (torch.int32, torch.uint32):
        raise ValueError("xor_out must be an int32 CUDA tensor")
    _check(load().fanout_read_floor(buf.data_ptr(), int(buf.numel() * buf.element_size()),
                                    xor_out.data_ptr(), _stream_handle(stream)),
           "fanout_read_floor")


def release() -> None:
    _check(load().fanout_release(), "fanout_release")

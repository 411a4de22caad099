"""Shared helpers of the GPU tests: run a drawn workload through the C ABI and
compare it with the fp64 oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from shared_prefix_fan_gb300 import binding, build

# Acceptance bar (bf16 inputs, fp32 accumulation): max |dO| <= 1e-2,
# mean |dO| <= 1e-3, max |d lse| <= 1e-3.
TOL_MAX_O, TOL_MEAN_O, TOL_LSE = 1e-2, 1e-3, 1e-3

_ready = False


def ensure_lib():
    global _ready
    if not _ready:
        build.build()
        binding.load()
        assert torch.cuda.is_available(), "GPU tests need CUDA"
        _ready = True


def to_dev_bf16(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


class DevWorkload:
    """A drawn workload resident on the GPU, page table from fanout_fork."""

    def __init__(self, w, dev="cuda"):
        ensure_lib()
        s = w.spec
        self.w = w
        self.table_host = binding.fork(w.prefix_pages, w.suffix_lens, s.page_size, w.free_pages,
                                       w.max_pages_per_branch)
        self.q = to_dev_bf16(w.q, dev)
        self.k = to_dev_bf16(w.k_pool, dev)
        self.v = to_dev_bf16(w.v_pool, dev)
        self.table = torch.from_numpy(self.table_host).to(dev)

    def run(self, out_dtype="f32", table=None, k=None, v=None, causal=None, stream=None):
        s = self.w.spec
        out, lse = binding.attn(self.q, self.k if k is None else k, self.v if v is None else v,
                                self.table if table is None else table, s.prefix_len,
                                self.w.suffix_lens, self.w.q_rows, s.h_q, s.h_kv, s.page_size,
                                s.scale, s.causal if causal is None else causal,
                                out_dtype=out_dtype, stream=stream)
        rc, site, block = binding.last_error_detail(stream)
        assert rc == binding.OK, f"device error {rc}: {binding.strerror(rc)} (site {site}, block {block})"
        return out, lse


def oracle_ref(w, rows=None, causal=None):
    s = w.spec
    table = oracle.fork(w.prefix_pages, w.suffix_lens, s.page_size, w.free_pages,
                        w.max_pages_per_branch)
    return oracle.attn(w.q, w.k_pool, w.v_pool, table, s.prefix_len, w.suffix_lens, w.q_rows,
                       s.h_q, s.h_kv, s.page_size, s.scale, s.causal if causal is None else causal,
                       rows=rows)


def compare(out, lse, ref_out, ref_lse, rows=None, what=""):
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.isfinite(o).all() and np.isfinite(l).all(), f"{what}: non-finite output"
    d = np.abs(o - ref_out)
    dl = np.abs(l - ref_lse)
    stats = dict(max_o=float(d.max()), mean_o=float(d.mean()), max_lse=float(dl.max()))
    assert stats["max_o"] <= TOL_MAX_O, (what, stats)
    assert stats["mean_o"] <= TOL_MEAN_O, (what, stats)
    assert stats["max_lse"] <= TOL_LSE, (what, stats)
    return stats


def sample_rows(w, every=64):
    """First and last token of every branch plus every `every`-th token."""
    T = w.q_rows
    tok0 = np.concatenate([[0], np.cumsum(T)])
    rows = set(range(0, int(tok0[-1]), every))
    for b in range(len(T)):
        if T[b]:
            rows.add(int(tok0[b]))
            rows.add(int(tok0[b + 1] - 1))
    return np.array(sorted(rows), dtype=np.int32)

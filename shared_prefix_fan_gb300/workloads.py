"""Seeded synthetic workloads for shared-prefix fan-out attention.

This module only draws inputs. It holds none of the method's arithmetic: no
page-table fork, no attention, no merge. Both the CUDA path and the CPU oracle
take their inputs from here, and each side then builds its own page tables
and computes its own results.

The shapes follow the Llama3-70B attention head layout the ADR works with
(ADR-0060, section 0 "reference dimensions": H_q = 64, H_kv = 8, G = 8,
d = 128) and the fan-out structure of "AHBM Agentic Runtime Architecture"
(section 3.1 "Fan-out context structure": every branch = shared prefix pages +
private suffix pages; section 3.2 "Sub-agent query batching": 8 sub-agents x
20 new tokens).

Draw order for a workload (fixed, so a seed pins every value):
  1. branch sizes (only where the workload draws them: the ragged one),
  2. the physical page permutation of the KV pool,
  3. Q, then the K pool, then the V pool, as fp32 N(0, 1) rounded to bf16.

Tokens past the end of a branch's last (partial) page are filled with random
values too: they are not part of any sequence and must never be read.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    """Sizes of one fan-out attention problem (before any value is drawn)."""

    name: str
    h_q: int
    h_kv: int
    d: int
    page_size: int
    prefix_len: int
    causal: bool
    # Either fixed per-branch sizes, or a ragged recipe drawn from the seed.
    q_rows: Optional[List[int]] = None  # new query tokens per branch (T_q,b)
    suffix_lens: Optional[List[int]] = None  # private suffix tokens per branch (S_b)
    ragged_branches: int = 0  # >0: draw T_q ~ U{tq_lo..tq_hi}, S ~ U{s_lo..s_hi}
    tq_lo: int = 1
    tq_hi: int = 1
    s_lo: int = 0
    s_hi: int = 0
    k_scale: float = 1.0  # K drawn as k_scale * N(0, 1)
    permute_prefix: bool = False  # physical placement of shared prefix pages
    permute_suffix: bool = False  # physical placement of private suffix pages
    seed: int = 0

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))


# The five workloads. Sizes come from the fan-out description (shared prefix,
# private suffix, new tokens as the suffix tail) and the Llama3-70B head shape.
WORKLOADS = {
    # Tiny case: one KV head, 3 branches x 4 new tokens, 256-token prefix.
    "tiny": WorkloadSpec(
        name="tiny", h_q=8, h_kv=1, d=128, page_size=16, prefix_len=256, causal=True,
        q_rows=[4, 4, 4], suffix_lens=[16, 16, 16], permute_suffix=True, seed=1001),
    # Fan-out decode: 8 branches x 1 new token, 32k shared prefix, 512 private.
    "decode": WorkloadSpec(
        name="decode", h_q=64, h_kv=8, d=128, page_size=64, prefix_len=32768,
        causal=True, q_rows=[1] * 8, suffix_lens=[512] * 8, seed=1002),
    # The pages' batching example: 8 sub-agents x 20 new tokens.
    "batching": WorkloadSpec(
        name="batching", h_q=64, h_kv=8, d=128, page_size=64, prefix_len=16384,
        causal=True, q_rows=[20] * 8, suffix_lens=[256] * 8, seed=1003),
    # Wide ragged fan-out: 32 branches, T_q ~ U{1..32}, S ~ U{64..4096},
    # every physical page permuted, K scaled x4 to widen the score range.
    "wide": WorkloadSpec(
        name="wide", h_q=64, h_kv=8, d=128, page_size=16, prefix_len=65536,
        causal=True, ragged_branches=32, tq_lo=1, tq_hi=32, s_lo=64, s_hi=4096,
        k_scale=4.0, permute_prefix=True, permute_suffix=True, seed=1004),
    # Single-sequence long-context causal prefill: 8192 new tokens over a
    # 131072-token context whose first 122880 tokens are cached.
    "prefill": WorkloadSpec(
        name="prefill", h_q=64, h_kv=8, d=128, page_size=64, prefix_len=122880,
        causal=True, q_rows=[8192], suffix_lens=[8192], seed=1005),
}


@dataclasses.dataclass
class Workload:
    """Drawn inputs of one problem. bf16 tensors are stored as uint16 bit patterns."""

    spec: WorkloadSpec
    q_rows: np.ndarray  # int32 [B]
    suffix_lens: np.ndarray  # int32 [B]
    prefix_pages: np.ndarray  # int32 [P / page_size]  physical ids of the shared prefix
    free_pages: np.ndarray  # int32 [n_free]  physical ids handed out to suffixes, in order
    num_pages: int
    q: np.ndarray  # uint16 [R, H_q, d]
    k_pool: np.ndarray  # uint16 [num_pages, H_kv, page_size, d]
    v_pool: np.ndarray  # uint16 [num_pages, H_kv, page_size, d]

    @property
    def num_branches(self) -> int:
        return int(self.q_rows.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.q_rows.sum())

    @property
    def max_pages_per_branch(self) -> int:
        ps = self.spec.page_size
        n_pre = self.spec.prefix_len // ps
        return n_pre + int(max([(int(s) + ps - 1) // ps for s in self.suffix_lens] + [0]))


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    """fp32 tensor -> bf16 (round to nearest even) -> uint16 bit pattern."""
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def draw(spec: WorkloadSpec, seed: Optional[int] = None,
         q_rows: Optional[List[int]] = None,
         suffix_lens: Optional[List[int]] = None) -> Workload:
    """Draw one workload. `q_rows` / `suffix_lens` override the spec's sizes."""
    g = torch.Generator().manual_seed(spec.seed if seed is None else seed)
    ps = spec.page_size
    if spec.prefix_len % ps:
        raise ValueError("prefix_len must be a multiple of page_size")
    # 1. sizes
    if q_rows is not None:
        tq = list(q_rows)
        sl = list(suffix_lens) if suffix_lens is not None else list(spec.suffix_lens)
    elif spec.ragged_branches:
        nb = spec.ragged_branches
        tq = torch.randint(spec.tq_lo, spec.tq_hi + 1, (nb,), generator=g).tolist()
        sl = torch.randint(spec.s_lo, spec.s_hi + 1, (nb,), generator=g).tolist()
    else:
        tq = list(spec.q_rows)
        sl = list(spec.suffix_lens) if suffix_lens is None else list(suffix_lens)
    if len(tq) != len(sl):
        raise ValueError("q_rows and suffix_lens differ in length")
    n_pre = spec.prefix_len // ps
    n_suf = sum((s + ps - 1) // ps for s in sl)
    num_pages = n_pre + n_suf
    # 2. physical placement
    ids = np.arange(num_pages, dtype=np.int32)
    if spec.permute_prefix and spec.permute_suffix:
        ids = torch.randperm(num_pages, generator=g).numpy().astype(np.int32)
    elif spec.permute_suffix and n_suf:
        tail = torch.randperm(n_suf, generator=g).numpy().astype(np.int32) + n_pre
        ids = np.concatenate([ids[:n_pre], tail])
    elif spec.permute_prefix and n_pre:
        head = torch.randperm(n_pre, generator=g).numpy().astype(np.int32)
        ids = np.concatenate([head, ids[n_pre:]])
    prefix_pages = np.ascontiguousarray(ids[:n_pre])
    free_pages = np.ascontiguousarray(ids[n_pre:])
    # 3. values
    r_total = int(sum(tq))
    q = _bf16_bits(torch.randn((r_total, spec.h_q, spec.d), generator=g))
    kshape = (num_pages, spec.h_kv, ps, spec.d)
    k = torch.randn(kshape, generator=g)
    if spec.k_scale != 1.0:
        k = k * spec.k_scale
    k_pool = _bf16_bits(k)
    del k
    v_pool = _bf16_bits(torch.randn(kshape, generator=g))
    return Workload(spec=spec, q_rows=np.asarray(tq, dtype=np.int32),
                    suffix_lens=np.asarray(sl, dtype=np.int32),
                    prefix_pages=prefix_pages, free_pages=free_pages,
                    num_pages=num_pages, q=q, k_pool=k_pool, v_pool=v_pool)


def small_spec(**kw) -> WorkloadSpec:
    """A small custom problem (tests): defaults are a 2-branch, G=4 layout."""
    base = dict(name="small", h_q=8, h_kv=2, d=128, page_size=16, prefix_len=64,
                causal=True, q_rows=[3, 5], suffix_lens=[20, 33], seed=7)
    base.update(kw)
    return WorkloadSpec(**base)

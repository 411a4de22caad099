#!/usr/bin/env python3
"""Benchmark of shared-prefix fan-out attention on GB300.

One step = one fanout_attn call (split-KV attention kernel + log-sum-exp
merge) over one synthetic workload already resident in HBM. The default
workload is the fan-out decode configuration (H_q=64, H_kv=8, d=128;
8 branches x 1 new token; 32768-token shared prefix + 512 private tokens per
branch; page 64; split-KV 32 ways). Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--per-config all|none|a,b] [--impl gpu|reference]

The line's top-level value, roofline, cpu_baseline, e2e and clocks are those
of --config (decode by default); "per_config" holds the same measurements for
each of the five workloads (tiny, decode, batching, wide, prefill).

Under torchrun (N > 1) every rank runs an independent replica of the same
problem on its own GPU (the path has no exchange step); timing is the max
over ranks, value = per-call latency of the slowest rank.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import tempfile
import time
import types

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from shared_prefix_fan_gb300.workloads import WORKLOADS, draw  # noqa: E402

METRIC = "us/call and achieved roofline % (KV HBM GB/s or tensor TFLOP/s) per config"
KERNEL_SOURCES = ["attn_fwd.cu", "ptx_sm100.cuh", "fanout_internal.h", "merge_row.cuh"]


# ------------------------------------------------------------------ accounting
def visible_pairs(w) -> int:
    """(token, query head, key) triples the method must compute (causal-visible only)."""
    s = w.spec
    total = 0
    for T, S in zip(w.q_rows.tolist(), w.suffix_lens.tolist()):
        n = s.prefix_len + S
        if s.causal:
            # token t (0..T-1) sees keys 0 .. P + S - T + t
            first = s.prefix_len + S - T + 1
            total += T * first + T * (T - 1) // 2 if T else 0
        else:
            total += T * n
    return total * s.h_q


def algorithmic_work(w, out_bytes_per_elem: int = 4):
    """Bytes and flops the method must move / compute (each unique KV token once)."""
    s = w.spec
    uniq_tokens = s.prefix_len + int(w.suffix_lens.sum())
    kv = uniq_tokens * s.h_kv * s.d * 2 * 2
    R = w.total_rows
    q = R * s.h_q * s.d * 2
    o = R * s.h_q * s.d * out_bytes_per_elem
    lse = R * s.h_q * 4
    flops = 4 * s.d * visible_pairs(w)
    return dict(kv_bytes=kv, q_bytes=q, out_bytes=o, lse_bytes=lse,
                call_bytes=kv + q + o + lse, split_bytes=kv + q, flops=flops)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), tc=float(d["bf16_tflops"]),
                    tc_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sustained=1700.0, source="fallback")


def source_code_text(text: str) -> str:
    """C++ source with comments removed and whitespace collapsed: what the
    compiler sees, so an edit to a comment does not retire a measurement."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "shared_prefix_fan_gb300", "csrc", f)) as fh:
            h.update(source_code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """dram read+write bytes per launch of the split kernel from the committed
    ncu summary, or None when absent or taken on a different kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("source_sha") != kernel_source_sha():
        return None
    return float(d["dram_bytes_per_launch"])


L2_NOTE = ("GPU arm: L2 flushed between timed calls (write 2x L2, then read 2x L2); "
           "CPU oracle arm: no device cache involved")


def workload_config(w, world: int) -> dict:
    """The `config` object of a line: the workload and its sizes only, the same
    in the GPU and the reference arm."""
    s = w.spec
    return {"workload": s.name, "h_q": s.h_q, "h_kv": s.h_kv, "d": s.d,
            "branches": w.num_branches, "q_rows": int(w.total_rows),
            "prefix_len": s.prefix_len, "suffix_tokens": int(w.suffix_lens.sum()),
            "page_size": s.page_size, "causal": s.causal, "l2": L2_NOTE,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def host_bf16(torch, bits):
    """A host bf16 tensor over uint16 bf16 bits (no copy)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def new_token_rows(w, table):
    """(page ids, slots) of every query token's own K/V row, token-major: token
    t of branch b sits at position prefix_len + S_b - T_b + t of the branch's
    sequence, the row a decode step appends just before it attends."""
    s = w.spec
    T = np.asarray(w.q_rows, dtype=np.int64)
    S = np.asarray(w.suffix_lens, dtype=np.int64)
    br = np.repeat(np.arange(len(T)), T)
    tok = np.arange(int(T.sum())) - np.repeat(np.cumsum(T) - T, T)
    pos = s.prefix_len + S[br] - T[br] + tok
    return table[br, pos // s.page_size], pos % s.page_size


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-i", gpu_id,
                                       "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]),
                                 power=float(parts[3]) if parts[3] not in ("[N/A]", "") else 0.0,
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in load:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in load])),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(load)}


def gpu_id_for_smi(torch, local_rank: int) -> str:
    try:
        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", None)
        dev = getattr(props, "pci_device_id", None)
        if bus is not None and dom is not None and dev is not None:
            return f"{dom:08x}:{bus:02x}:{dev:02x}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x for x in vis.split(",") if x]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ------------------------------------------------------------------ oracle leg
def cpu_model() -> str:
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, else the ISA)."""
    import platform
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def oracle_sample(w, budget_s: float = 15.0):
    """Time the fp64 oracle (as it stands) on a bounded sample of rows of `w`;
    returns (us per full call extrapolated, seconds, rows, threads, repetitions)."""
    import oracle
    R = w.total_rows
    lib = oracle.load()
    s = w.spec
    table = oracle.fork(w.prefix_pages, w.suffix_lens, s.page_size, w.free_pages,
                        w.max_pages_per_branch, lib=lib)
    # one probe row sizes the sample
    t0 = time.perf_counter()
    oracle.attn(w.q, w.k_pool, w.v_pool, table, s.prefix_len, w.suffix_lens, w.q_rows, s.h_q,
                s.h_kv, s.page_size, s.scale, s.causal, rows=[R - 1], lib=lib)
    per_row = max(time.perf_counter() - t0, 1e-6)
    n = int(max(1, min(R, budget_s / per_row)))
    rows = np.unique(np.linspace(0, R - 1, n).astype(np.int32))
    # the sample (every row when they all fit), repeated until about 2/3 of the
    # budget is spent so that short calls are timed over many repetitions
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.attn(w.q, w.k_pool, w.v_pool, table, s.prefix_len, w.suffix_lens, w.q_rows,
                    s.h_q, s.h_kv, s.page_size, s.scale, s.causal, rows=rows, lib=lib)
        reps += 1
        if time.perf_counter() - t0 >= budget_s * 2 / 3 or reps >= 100:
            break
    dt = (time.perf_counter() - t0) / reps
    # rows differ in cost (causal): scale by visible keys, not by row count
    vis_all = _row_keys(w)
    frac = vis_all[rows].sum() / vis_all.sum()
    return dt / frac * 1e6, dt * reps, len(rows), oracle.num_threads(lib), reps


def _row_keys(w):
    s = w.spec
    out = []
    for T, S in zip(w.q_rows.tolist(), w.suffix_lens.tolist()):
        for t in range(T):
            n = s.prefix_len + S
            out.append(min(n, s.prefix_len + S - T + t + 1) if s.causal else n)
    return np.asarray(out, dtype=np.float64)


def run_reference(args):
    """Reference arm: the fp64 CPU oracle as it stands, timed on this host's
    cores on bounded samples of the same workloads (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    w = draw(WORKLOADS[args.config])
    per_step = []
    budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    info = None
    for i in range(args.warmup + args.steps):
        info = oracle_sample(w, budget_s=budget)
        if i >= args.warmup:
            per_step.append(info[0])
    v = float(np.mean(per_step))

    def cpu_of(value, info_, what):
        return {"value": value, "unit": "us/call", "cores": info_[3], "kind": "oracle",
                "cpu_model": cpu_model(), "sample": f"{info_[2]} of {what.total_rows} query tokens (all heads) "
                          f"x {info_[4]} repetitions, {info_[1]:.1f} s per step, "
                          f"extrapolated by visible keys"}

    per = {}
    for name in parse_per_config(args.per_config):
        if name == args.config:
            per[name] = {"value": v, "unit": "us/call", "config": workload_config(w, world),
                         "cpu_baseline": cpu_of(v, info, w)}
            continue
        wn = draw(WORKLOADS[name])
        inf = oracle_sample(wn, budget_s=5.0)
        per[name] = {"value": inf[0], "unit": "us/call", "config": workload_config(wn, world),
                     "cpu_baseline": cpu_of(inf[0], inf, wn)}
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/call",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, world),
            "cpu_baseline": cpu_of(v, info, w),
            "e2e": {"value": v, "unit": "us/call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "per_config": {n: per[n] for n in PER_CONFIG_ORDER if n in per}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ranks
def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings (all ranks get the result).

    Replicas: every rank runs the whole problem on its own GPU; the slowest
    rank defines the job's time."""
    if dist is None or not dist.is_available() or not dist.is_initialized() \
            or dist.get_world_size() == 1:
        return [float(v) for v in values]
    import torch
    x = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return x.tolist()


# ------------------------------------------------------------------ GPU arm
def roofline_of(work, peaks, t_kernel_s, workload):
    """Roofline object of the attention kernel: the slower of its algorithmic
    bytes (unique KV + Q) at the measured HBM peak and its flops at the
    measured bf16 peak decides the bound."""
    t_hbm = work["split_bytes"] / (peaks["hbm"] * 1e9)
    t_tc = work["flops"] / (peaks["tc"] * 1e12)
    if t_hbm >= t_tc:
        achieved = work["split_bytes"] / t_kernel_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s"}
    else:
        achieved = work["flops"] / t_kernel_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["tc"], "unit": "TFLOP/s",
                # for a kernel that runs under the power cap (long prefill)
                "peak_sustained": peaks["tc_sustained"],
                "frac_sustained": achieved / peaks["tc_sustained"]}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = ncu_traffic(workload)
    roof["algorithmic_bytes"] = work["split_bytes"]
    roof["algorithmic_flops"] = work["flops"]
    roof["kernel"] = "attn_fwd_kernel"
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json burst figure)" \
        if peaks["source"] == "measured" else "fallback"
    return roof


class Bench:
    """One GPU (one rank): inputs resident in HBM, the L2 flushed between timed
    calls (write a buffer twice the L2 size, then read another one, so no dirty
    line is left to be written back inside the next timed call)."""

    def __init__(self, torch, binding, local, world, dist):
        self.torch, self.binding, self.local, self.world, self.dist = \
            torch, binding, local, world, dist
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        n = max(2 * l2, 256 << 20)
        self.flush_w = torch.empty(n, dtype=torch.uint8, device="cuda")
        self.flush_r = torch.ones(n // 4, dtype=torch.float32, device="cuda")
        self.sms = torch.cuda.get_device_properties(local).multi_processor_count

    def flush_l2(self):
        self.flush_w.zero_()
        self.flush_r.sum()

    def read_floor_us(self, nbytes, steps):
        """Mean time of one fanout_read_floor launch over `nbytes` of device
        memory, L2 flushed before each and CUDA events around it: the shortest
        time one kernel that reads those bytes takes here."""
        torch, binding = self.torch, self.binding
        stream = torch.cuda.current_stream()
        buf = torch.zeros(nbytes // 16 * 16, dtype=torch.uint8, device="cuda")
        xo = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(3):
            self.flush_l2()
            binding.read_floor(buf, xo)
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(steps)]
        for a, b in ev:
            self.flush_l2()
            a.record(stream)
            binding.read_floor(buf, xo)
            b.record(stream)
        torch.cuda.synchronize()
        t = float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3
        del buf
        return self.max_ranks([t])[0]

    def max_ranks(self, vals):
        return max_over_ranks(vals, self.dist if self.world > 1 else None, "cuda")

    def _check(self, name):
        rc = self.binding.last_error()
        if rc != self.binding.OK:
            raise RuntimeError(f"{name}: device error {self.binding.strerror(rc)}")

    def _prepare(self, name):
        """The workload `name` drawn, its page table forked, host copies of its
        inputs and resident device copies, out / lse, and the timed call."""
        torch, binding = self.torch, self.binding
        c = types.SimpleNamespace(name=name)
        c.w = w = draw(WORKLOADS[name])
        c.s = s = w.spec
        c.table = binding.fork(w.prefix_pages, w.suffix_lens, s.page_size, w.free_pages,
                               w.max_pages_per_branch)
        c.h_q, c.h_k, c.h_v = (host_bf16(torch, x) for x in (w.q, w.k_pool, w.v_pool))
        c.h_t = torch.from_numpy(c.table)
        c.q, c.k, c.v, c.t = (x.cuda() for x in (c.h_q, c.h_k, c.h_v, c.h_t))
        c.out = torch.empty((w.total_rows, s.h_q, s.d), dtype=torch.float32, device="cuda")
        c.lse = torch.empty((w.total_rows, s.h_q), dtype=torch.float32, device="cuda")

        def call():
            binding.attn(c.q, c.k, c.v, c.t, s.prefix_len, w.suffix_lens, w.q_rows, s.h_q,
                         s.h_kv, s.page_size, s.scale, s.causal, out=c.out, lse=c.lse)

        c.call = call
        return c

    def _time_calls(self, c, steps, warmup, soak_s):
        """Warm-up, an untimed soak (clocks settle and are sampled), then the
        timed steps: (call ms per step, attention-kernel ms per step, clocks)."""
        torch, binding = self.torch, self.binding
        for _ in range(max(3, warmup)):
            self.flush_l2()
            c.call()
        torch.cuda.synchronize()
        self._check(c.name)
        sampler = ClockSampler(gpu_id_for_smi(torch, self.local))
        t_end = time.perf_counter() + soak_s
        while time.perf_counter() < t_end:
            self.flush_l2()
            c.call()
            torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(steps)]
        for quad in ev:              # the raw CUDA events are created at first record
            for e in quad:
                e.record(stream)
        torch.cuda.synchronize()
        if self.world > 1:
            self.dist.barrier()
        torch.cuda.synchronize()
        # Each step times one call (e0..e1); after it, an untimed call with
        # events around the attention kernel alone (k0..k1), so that both
        # figures come from the same clock and power state (under a power cap
        # the clocks drift within seconds). Events between the attention kernel
        # and the merge launch would stop the merge from overlapping it, so they
        # stay out of the timed calls.
        for e0, e1, k0, k1 in ev:
            self.flush_l2()                    # L2 flushed between timed calls
            e0.record(stream)
            c.call()
            e1.record(stream)
            self.flush_l2()
            binding.set_profile_events(k0, k1)  # brackets the split-KV kernel alone
            c.call()
            binding.set_profile_events(None, None)
        torch.cuda.synchronize()
        if self.world > 1:
            self.dist.barrier()
        clocks = sampler.stop()
        self._check(c.name)
        call_ms = np.array([a.elapsed_time(b) for a, b, _, _ in ev])
        split_ms = np.array([a.elapsed_time(b) for _, _, a, b in ev])
        return call_ms, split_ms, clocks

    def _timed_steps(self, steps, body):
        """Mean µs (max over ranks) of `body` per step, events around it, the L2
        flushed before each step, two untimed steps first."""
        torch = self.torch
        stream = torch.cuda.current_stream()
        ms = []
        for i in range(steps + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            self.flush_l2()
            a.record(stream)
            body()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                ms.append(a.elapsed_time(b))
        return self.max_ranks([float(np.mean(ms)) * 1e3])[0]

    def _e2e_full(self, c, steps):
        """End to end: q, the K/V pools and the page table from pinned host
        memory, the call, out and lse read back, every step."""
        torch = self.torch
        p_q, p_k, p_v, p_t = (x.pin_memory() for x in (c.h_q, c.h_k, c.h_v, c.h_t))
        p_out = torch.empty(c.out.shape, dtype=c.out.dtype).pin_memory()
        p_lse = torch.empty(c.lse.shape, dtype=c.lse.dtype).pin_memory()

        def step():
            c.q.copy_(p_q, non_blocking=True)
            c.k.copy_(p_k, non_blocking=True)
            c.v.copy_(p_v, non_blocking=True)
            c.t.copy_(p_t, non_blocking=True)
            c.call()
            p_out.copy_(c.out, non_blocking=True)
            p_lse.copy_(c.lse, non_blocking=True)

        value = self._timed_steps(steps, step)
        self._check(c.name)
        h2d = sum(x.numel() * x.element_size() for x in (p_q, p_k, p_v, p_t))
        d2h = sum(x.numel() * x.element_size() for x in (p_out, p_lse))
        return {"value": value, "unit": "us/call", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": steps,
                "note": "q, K/V page pool and page table copied from pinned host memory, "
                        "out and lse copied back, every step"}

    def _e2e_resident(self, c, steps):
        """A decode loop keeps the cache in HBM: each step brings only the
        queries and the new tokens' K/V rows, appends the rows to the pools,
        attends, and reads the result back. The appended rows are the ones
        already at those positions, so the pools and the result stay as in
        the timed calls (checked bit for bit)."""
        torch, binding = self.torch, self.binding
        w, s = c.w, c.s
        T = np.asarray(w.q_rows, dtype=np.int64)
        S = np.asarray(w.suffix_lens, dtype=np.int64)
        pages, slot = new_token_rows(w, c.table)
        k_rows = host_bf16(torch, w.k_pool[pages, :, slot, :])   # [R, H_kv, d]
        v_rows = host_bf16(torch, w.v_pool[pages, :, slot, :])
        # One staging buffer each way (one copy per direction per step):
        # q, the new K and V rows and the page table up; out and lse down.
        ups = [c.h_q, k_rows, v_rows, c.h_t]
        offs, n = [], 0
        for x in ups:
            offs.append(n)
            n += (x.numel() * x.element_size() + 255) // 256 * 256
        p_up = torch.empty(n, dtype=torch.uint8).pin_memory()
        d_up = torch.empty(n, dtype=torch.uint8, device="cuda")

        def section(buf, i):
            x = ups[i]
            nb = x.numel() * x.element_size()
            return buf[offs[i]:offs[i] + nb].view(x.dtype).view(x.shape)

        for i, x in enumerate(ups):
            section(p_up, i).copy_(x)
        dq, dkn, dvn, dt = (section(d_up, i) for i in range(4))
        n_out = c.out.numel()
        d_down = torch.empty(n_out + c.lse.numel(), dtype=torch.float32, device="cuda")
        p_down = torch.empty(d_down.shape, dtype=torch.float32).pin_memory()
        out2, lse2 = d_down[:n_out].view(c.out.shape), d_down[n_out:].view(c.lse.shape)
        before = (S - T).astype(np.int32)

        def step():
            d_up.copy_(p_up, non_blocking=True)
            binding.kv_append(dkn, dvn, c.k, c.v, dt, s.prefix_len, before, w.q_rows,
                              s.page_size)
            binding.attn(dq, c.k, c.v, dt, s.prefix_len, w.suffix_lens, w.q_rows, s.h_q,
                         s.h_kv, s.page_size, s.scale, s.causal, out=out2, lse=lse2)
            p_down.copy_(d_down, non_blocking=True)

        value = self._timed_steps(steps, step)
        self._check(c.name)
        # the rows went back where they came from: the result must be the timed
        # calls' result bit for bit (reported; the parity tests are the gate)
        same = bool(torch.equal(out2, c.out) and torch.equal(lse2, c.lse))
        return {"value": value, "unit": "us/call", "h2d_bytes_per_step": int(p_up.numel()),
                "d2h_bytes_per_step": int(p_down.numel() * 4), "steps": steps,
                "result_equals_timed_calls": same,
                "note": "K/V pools resident; q, the step's new K/V rows and the page table "
                        "copied up from one pinned staging buffer, fanout_kv_append, the "
                        "call, out and lse copied down in one copy, every step"}

    def _kv_append(self, c, steps):
        """The cache append of the workload's new tokens (fanout_kv_append, the
        step before attention in a decode loop): every query token's own K and
        V rows written into its page and slot, timed alone like the call. The
        rows written are the bytes already there, so the pools do not change.
        Algorithmic bytes: the new rows read once and written once."""
        torch, binding = self.torch, self.binding
        w, s = c.w, c.s
        T = np.asarray(w.q_rows, dtype=np.int64)
        S = np.asarray(w.suffix_lens, dtype=np.int64)
        pages, slot = new_token_rows(w, c.table)
        kn = host_bf16(torch, w.k_pool[pages, :, slot, :]).cuda()
        vn = host_bf16(torch, w.v_pool[pages, :, slot, :]).cuda()
        before = (S - T).astype(np.int32)

        def step():
            binding.kv_append(kn, vn, c.k, c.v, c.t, s.prefix_len, before, w.q_rows,
                              s.page_size)

        value = self._timed_steps(steps, step)
        self._check(c.name)
        nbytes = 2 * (kn.numel() + vn.numel()) * kn.element_size()
        peak = load_peaks()["hbm"]
        achieved = nbytes / (value * 1e-6) / 1e9
        return {"value": value, "unit": "us/call", "rows": int(w.total_rows),
                "algorithmic_bytes": int(nbytes), "achieved_gbs": achieved,
                "peak_gbs": peak, "frac": achieved / peak, "steps": steps}

    def run(self, name, steps, warmup, soak_s, e2e_steps, cpu_budget_s):
        """One workload's entry of the JSON line."""
        c = self._prepare(name)
        w, s = c.w, c.s
        units, cta_first, n_parts = self.binding.plan(
            w.suffix_lens, w.q_rows, s.prefix_len, s.h_q, s.h_kv, s.page_size, s.causal,
            self.sms)
        launches_per_call = 1 + (1 if n_parts > 0 else 0)
        call_ms, split_ms, clocks = self._time_calls(c, steps, warmup, soak_s)
        mean_call, mean_split = self.max_ranks([float(call_ms.mean()), float(split_ms.mean())])
        e2e = None
        if e2e_steps > 0:
            e2e = self._e2e_full(c, e2e_steps)
            e2e["resident_cache"] = self._e2e_resident(c, e2e_steps)
        append = self._kv_append(c, min(steps, 20))

        work = algorithmic_work(w)
        peaks = load_peaks()
        roof = roofline_of(work, peaks, mean_split * 1e-3, name)
        if roof["bound"] == "hbm":
            # context for an HBM-bound kernel: a plain one-launch read of its
            # algorithmic bytes, timed the same way (launch and ramp included)
            floor = self.read_floor_us(work["split_bytes"], steps)
            roof["read_floor_us"] = floor
            roof["frac_of_read_floor"] = floor / (mean_split * 1e3)
        t_call_roof = max(work["call_bytes"] / (peaks["hbm"] * 1e9),
                          work["flops"] / (peaks["tc"] * 1e12))
        value_us = mean_call * 1e3
        cpu = None
        if cpu_budget_s > 0 and int(os.environ.get("RANK", "0")) == 0:
            us, dt, nrows, threads, reps = oracle_sample(w, budget_s=cpu_budget_s)
            cpu = {"value": us, "unit": "us/call", "cores": threads, "kind": "oracle",
                   "cpu_model": cpu_model(),
                   "sample": f"{nrows} of {w.total_rows} query tokens (all {s.h_q} heads) x "
                             f"{reps} repetitions, {dt:.1f} s, extrapolated to the full call "
                             f"by visible keys"}
        entry = {
            "value": value_us, "unit": "us/call", "steps": steps,
            "kernel_us": mean_split * 1e3,
            # medians over the steps (this rank), beside the means above
            "median_us": float(np.median(call_ms)) * 1e3,
            "kernel_median_us": float(np.median(split_ms)) * 1e3,
            "config": workload_config(w, self.world),
            "plan": {"work_units": int(len(units)), "persistent_ctas": int(len(cta_first) - 1),
                     "partial_blocks": n_parts},
            "call_roofline": {"t_roof_us": t_call_roof * 1e6,
                              "frac": t_call_roof / (value_us * 1e-6),
                              "bytes": work["call_bytes"], "flops": work["flops"]},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "kv_append": append,
            # the timed region holds each step's timed call and its kernel-only twin
            "gpu_launches": 2 * launches_per_call * steps, "clocks": clocks,
        }
        c.__dict__.clear()   # the call closure refers to c: drop the tensors now
        self.torch.cuda.empty_cache()
        return entry


PER_CONFIG_ORDER = ["decode", "tiny", "batching", "wide", "prefill"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="decode", choices=sorted(WORKLOADS),
                    help="the workload of the line's top-level value")
    ap.add_argument("--per-config", default="all",
                    help="comma-separated workloads measured into per_config ('all', 'none')")
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.5,
                    help="seconds of untimed calls before the timed steps (clock sampling)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    from shared_prefix_fan_gb300 import binding, build
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    binding.load()
    bench = Bench(torch, binding, local, world, dist)

    names = parse_per_config(args.per_config)
    e2e_steps = 0 if args.no_e2e else max(3, min(args.steps, 20))
    head = bench.run(args.config, args.steps, args.warmup, args.soak_s, e2e_steps,
                     0.0 if args.no_cpu_baseline else 15.0)
    per = {args.config: head} if args.config in names else {}
    for name in names:
        if name == args.config:
            continue
        try:
            per[name] = bench.run(name, args.steps, args.warmup, min(args.soak_s, 0.5),
                                  0 if args.no_e2e else max(3, min(args.steps, 10)),
                                  0.0 if args.no_cpu_baseline else 6.0)
        except (RuntimeError, MemoryError) as e:
            # one process: the line still carries the other workloads and the
            # error; with several ranks a rank that stopped early would leave
            # the others waiting in a barrier, so every rank stops
            if world > 1:
                raise
            per[name] = {"error": f"{type(e).__name__}: {e}"}

    line = {
        "metric": METRIC, "value": head["value"], "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["value"] / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": head["config"], "plan": head["plan"],
        "call_roofline": head["call_roofline"],
        "split_kernel_us": head["kernel_us"],
        "roofline": head["roofline"], "cpu_baseline": head["cpu_baseline"], "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
        "per_config": {n: per[n] for n in PER_CONFIG_ORDER if n in per},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def parse_per_config(spec: str):
    if spec == "all":
        return list(PER_CONFIG_ORDER)
    if spec in ("", "none"):
        return []
    names = [x.strip() for x in spec.split(",") if x.strip()]
    for n in names:
        if n not in WORKLOADS:
            raise SystemExit(f"unknown workload {n!r}")
    return names


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of shared-prefix fan-out attention on GB300.

One step = one fanout_attn call (split-KV attention kernel + log-sum-exp
merge) over one synthetic workload already resident in HBM. The default
workload is the fan-out decode configuration (H_q=64, H_kv=8, d=128;
8 branches x 1 new token; 32768-token shared prefix + 512 private tokens per
branch; page 64; split-KV 32 ways). Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--impl gpu|reference]

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
    """Reference arm: the fp64 CPU oracle, timed on this host's cores."""
    rank = int(os.environ.get("RANK", "0"))
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
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/call",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.config},
            "cpu_baseline": {"value": v, "unit": "us/call", "cores": info[3], "kind": "oracle",
                             "sample": f"{info[2]} of {w.total_rows} query tokens (all heads) "
                                       f"x {info[4]} repetitions, {info[1]:.1f} s per step, "
                                       f"extrapolated by visible keys"},
            "e2e": {"value": v, "unit": "us/call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
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
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="decode", choices=sorted(WORKLOADS))
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

    w = draw(WORKLOADS[args.config])
    s = w.spec
    table = binding.fork(w.prefix_pages, w.suffix_lens, s.page_size, w.free_pages,
                         w.max_pages_per_branch)

    def host_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    h_q, h_k, h_v = host_bf16(w.q), host_bf16(w.k_pool), host_bf16(w.v_pool)
    h_t = torch.from_numpy(table)
    q, k, v, t = (x.cuda() for x in (h_q, h_k, h_v, h_t))
    R = w.total_rows
    out = torch.empty((R, s.h_q, s.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((R, s.h_q), dtype=torch.float32, device="cuda")
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device="cuda")

    def flush_l2():
        # Write a buffer twice the L2 size, then read another one: the timed call
        # starts with none of its inputs in L2 and no dirty lines left to write back.
        flush.zero_()
        flush_rd.sum()

    def call():
        binding.attn(q, k, v, t, s.prefix_len, w.suffix_lens, w.q_rows, s.h_q, s.h_kv,
                     s.page_size, s.scale, s.causal, out=out, lse=lse)

    for _ in range(max(3, args.warmup)):
        flush_l2()
        call()
    torch.cuda.synchronize()
    rc = binding.last_error()
    if rc != binding.OK:
        raise RuntimeError(f"device error {binding.strerror(rc)}")
    units, cta_first, n_parts = binding.plan(
        w.suffix_lens, w.q_rows, s.prefix_len, s.h_q, s.h_kv, s.page_size, s.causal,
        torch.cuda.get_device_properties(local).multi_processor_count)
    launches_per_call = 1 + (1 if n_parts > 0 else 0)

    sampler = ClockSampler(gpu_id_for_smi(torch, local))
    t_end = time.perf_counter() + args.soak_s
    while time.perf_counter() < t_end:   # untimed soak: clocks settle and get sampled
        flush_l2()
        call()
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for quad in ev:              # the raw CUDA events are created at first record
        for e in quad:
            e.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for e0, e1, _, _ in ev:
        flush_l2()                         # L2 flushed between timed calls
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    # The attention kernel alone, in a second pass: events recorded between it
    # and a separate merge launch would stop the merge from overlapping it, so
    # they stay out of the pass the call time comes from.
    for _, _, k0, k1 in ev:
        flush_l2()
        binding.set_profile_events(k0, k1)  # brackets the split-KV kernel alone
        call()
    torch.cuda.synchronize()
    binding.set_profile_events(None, None)
    call_ms = np.array([a.elapsed_time(b) for a, b, _, _ in ev])
    split_ms = np.array([a.elapsed_time(b) for _, _, a, b in ev])
    rc = binding.last_error()
    if rc != binding.OK:
        raise RuntimeError(f"device error {binding.strerror(rc)}")
    mean_call = float(call_ms.mean())
    mean_split = float(split_ms.mean())
    mean_call, mean_split = max_over_ranks([mean_call, mean_split], dist if world > 1 else None,
                                           "cuda")

    # end to end: inputs from pinned host memory, result read back, every step
    e2e = None
    if not args.no_e2e:
        p_q, p_k, p_v, p_t = (x.pin_memory() for x in (h_q, h_k, h_v, h_t))
        p_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        p_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        n_e2e = max(3, min(args.steps, 20))
        e2e_ms = []
        for i in range(n_e2e + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush_l2()
            a.record(stream)
            q.copy_(p_q, non_blocking=True)
            k.copy_(p_k, non_blocking=True)
            v.copy_(p_v, non_blocking=True)
            t.copy_(p_t, non_blocking=True)
            call()
            p_out.copy_(out, non_blocking=True)
            p_lse.copy_(lse, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                e2e_ms.append(a.elapsed_time(b))
        e2e_val = float(np.mean(e2e_ms)) * 1e3
        e2e_val = max_over_ranks([e2e_val], dist if world > 1 else None, "cuda")[0]
        h2d = sum(x.numel() * x.element_size() for x in (p_q, p_k, p_v, p_t))
        d2h = sum(x.numel() * x.element_size() for x in (p_out, p_lse))
        e2e = {"value": e2e_val, "unit": "us/call", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "note": "q, K/V page pool and page table copied from pinned host memory, "
                       "out and lse copied back, every step"}

    work = algorithmic_work(w)
    peaks = load_peaks()
    t_split = mean_split * 1e-3
    t_hbm = work["split_bytes"] / (peaks["hbm"] * 1e9)
    t_tc = work["flops"] / (peaks["tc"] * 1e12)
    if t_hbm >= t_tc:
        achieved = work["split_bytes"] / t_split / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s"}
    else:
        achieved = work["flops"] / t_split / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["tc"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = ncu_traffic(args.config)
    roof["kernel"] = "attn_fwd_kernel"
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json burst figure)" \
        if peaks["source"] == "measured" else "fallback"
    t_call_roof = max(work["call_bytes"] / (peaks["hbm"] * 1e9), t_tc)
    value_us = mean_call * 1e3

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        us, dt, nrows, threads, reps = oracle_sample(w, budget_s=15.0)
        cpu = {"value": us, "unit": "us/call", "cores": threads, "kind": "oracle",
               "sample": f"{nrows} of {R} query tokens (all {s.h_q} heads) x {reps} "
                         f"repetitions, {dt:.1f} s, extrapolated to the full call by "
                         f"visible keys"}

    line = {
        "metric": METRIC, "value": value_us, "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_call,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.config, "h_q": s.h_q, "h_kv": s.h_kv, "d": s.d,
                   "branches": w.num_branches, "q_rows": int(R), "prefix_len": s.prefix_len,
                   "suffix_tokens": int(w.suffix_lens.sum()), "page_size": s.page_size,
                   "causal": s.causal, "work_units": int(len(units)),
                   "persistent_ctas": int(len(cta_first) - 1), "partial_blocks": n_parts,
                   "l2": "flushed between timed calls (write 2x L2, then read 2x L2)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "call_roofline": {"t_roof_us": t_call_roof * 1e6, "frac": t_call_roof / (value_us * 1e-6),
                          "bytes": work["call_bytes"], "flops": work["flops"]},
        "split_kernel_us": mean_split * 1e3,
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_call * args.steps, "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

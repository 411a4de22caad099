"""The benchmark's work accounting against the oracle's visible-pair count (CPU only)."""
import numpy as np
import pytest

import bench
import oracle
from shared_prefix_fan_gb300.workloads import WORKLOADS, draw, small_spec


@pytest.mark.parametrize("name", ["tiny", "decode", "batching", "wide"])
def test_visible_pairs_match_oracle(name):
    w = draw(WORKLOADS[name])
    s = w.spec
    assert bench.visible_pairs(w) == oracle.count_pairs(s.prefix_len, w.suffix_lens, w.q_rows,
                                                        s.h_q, s.causal)


def test_noncausal_pairs():
    w = draw(small_spec(causal=False, q_rows=[3, 0, 5], suffix_lens=[1, 4, 9]))
    s = w.spec
    assert bench.visible_pairs(w) == oracle.count_pairs(s.prefix_len, w.suffix_lens, w.q_rows,
                                                        s.h_q, False)


def test_decode_bytes():
    w = draw(WORKLOADS["decode"])
    work = bench.algorithmic_work(w)
    assert work["kv_bytes"] == (32768 + 8 * 512) * 8 * 128 * 2 * 2
    assert work["flops"] == 4 * 128 * 64 * 8 * (32768 + 512)


def test_kernel_fingerprint_ignores_comments_only():
    """The ncu traffic stays attached to a kernel whose comments changed, and
    is dropped as soon as its code changes."""
    code = "int f(int a) {\n  return a + 1;  // add one\n}\n/* block\n comment */\n"
    assert bench.source_code_text(code) == bench.source_code_text(
        "int f(int a) { return a + 1; }  // other words\n")
    assert bench.source_code_text(code) != bench.source_code_text("int f(int a) { return a + 2; }")
    assert bench.source_code_text('asm("ld.global.v4.s32 {%0}, [%1];");') == \
        'asm("ld.global.v4.s32 {%0}, [%1];");'


def test_roofline_object_bound_and_fractions():
    """Decode is HBM bound and batching tensor bound under the measured peaks;
    the fraction is achieved / peak and the algorithmic work is carried along."""
    peaks = dict(hbm=6775.3, tc=1900.5, tc_sustained=1691.5, source="measured")
    w = draw(WORKLOADS["decode"])
    work = bench.algorithmic_work(w)
    r = bench.roofline_of(work, peaks, 33.8e-6, "decode")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - work["split_bytes"] / 33.8e-6 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 6775.3) < 1e-12
    assert r["algorithmic_bytes"] == work["split_bytes"]
    wb = draw(WORKLOADS["batching"])
    rb = bench.roofline_of(bench.algorithmic_work(wb), peaks, 76.5e-6, "batching")
    assert rb["bound"] == "tensor" and rb["unit"] == "TFLOP/s"
    assert abs(rb["frac_sustained"] - rb["achieved"] / 1691.5) < 1e-12


def test_workload_config_is_the_workload_only():
    """Both arms print the same `config`: the workload's sizes, no plan details."""
    w = draw(WORKLOADS["batching"])
    c = bench.workload_config(w, 1)
    assert c["workload"] == "batching" and c["q_rows"] == 160 and c["branches"] == 8
    assert c["prefix_len"] == 16384 and c["suffix_tokens"] == 8 * 256 and c["page_size"] == 64
    assert c["parallelism"] == "single GPU" and "l2" in c
    assert not any(k in c for k in ("work_units", "persistent_ctas", "partial_blocks"))
    assert bench.workload_config(w, 4)["parallelism"] == "replicas x4"


def test_per_config_parsing():
    assert bench.parse_per_config("all") == ["decode", "tiny", "batching", "wide", "prefill"]
    assert bench.parse_per_config("none") == []
    assert bench.parse_per_config("wide, tiny") == ["wide", "tiny"]
    with pytest.raises(SystemExit):
        bench.parse_per_config("decode,nonsense")


def test_traffic_is_reported_only_for_the_captured_kernel_source(tmp_path, monkeypatch):
    """profiles/traffic.json entries carry the kernel source fingerprint; a
    mismatch (the kernel changed since the capture) reports no traffic."""
    import json
    import os
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = bench.kernel_source_sha()
    (prof / "traffic.json").write_text(json.dumps({
        "decode": {"kernel": "attn_fwd_kernel", "source_sha": sha, "dram_bytes_per_launch": 123.0},
        "wide": {"kernel": "attn_fwd_kernel", "source_sha": "0" * 16, "dram_bytes_per_launch": 9.0}}))
    real_join = os.path.join

    def join(*parts):  # profiles/ under tmp_path, sources from the repository
        if len(parts) >= 2 and parts[1] == "profiles":
            return real_join(str(tmp_path), *parts[1:])
        return real_join(*parts)

    monkeypatch.setattr(bench.os.path, "join", join)
    assert bench.ncu_traffic("decode") == 123.0
    assert bench.ncu_traffic("wide") is None
    assert bench.ncu_traffic("prefill") is None


@pytest.mark.parametrize("spec", [
    WORKLOADS["tiny"],
    small_spec(q_rows=[3, 0, 5, 1], suffix_lens=[20, 4, 33, 1], page_size=16, prefix_len=48,
               permute_suffix=True, seed=11),
], ids=["tiny", "ragged"])
def test_new_token_rows_are_the_append_positions(spec):
    """The resident-cache leg of the bench re-appends each query token's own
    K/V row: the rows new_token_rows names must be exactly where the oracle's
    append (before = S - T, add = T) writes them."""
    w = draw(spec)
    s = w.spec
    table = oracle.fork(w.prefix_pages, w.suffix_lens, s.page_size, w.free_pages,
                        w.max_pages_per_branch)
    pages, slots = bench.new_token_rows(w, table)
    R = w.total_rows
    rng = np.random.default_rng(5)
    k_new = rng.integers(1, 2**15, size=(R, s.h_kv, s.d), dtype=np.uint16)
    v_new = rng.integers(1, 2**15, size=(R, s.h_kv, s.d), dtype=np.uint16)
    T = np.asarray(w.q_rows, np.int32)
    kp, vp = oracle.kv_append(k_new, v_new, w.k_pool, w.v_pool, table, s.prefix_len,
                              np.asarray(w.suffix_lens, np.int32) - T, T)
    assert np.array_equal(kp[pages, :, slots, :], k_new)
    assert np.array_equal(vp[pages, :, slots, :], v_new)
    kp[pages, :, slots, :] = w.k_pool[pages, :, slots, :]   # nothing else was written
    vp[pages, :, slots, :] = w.v_pool[pages, :, slots, :]
    assert np.array_equal(kp, w.k_pool) and np.array_equal(vp, w.v_pool)

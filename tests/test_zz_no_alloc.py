"""fanout_attn_noalloc: the attention call for callers that must not allocate
device memory during a call (an engine that owns all device memory through its
own pool, code that cannot afford cudaFree's device-wide synchronisation, or
code running where allocation is not allowed). It keeps its work plan and
split partials in the library's fixed scratch array instead of a cudaMalloc'd
workspace. Checked against fanout_attn and the fp64 oracle, through the C ABI,
on two calls in a row with different problems (the shared array keeps the
previous call's contents), on consecutive decode steps, for the clear
rejection of a problem too big for the array, and for the refusal of a stream
that is being captured.

This file is collected last on purpose (pytest orders files by name)."""
import numpy as np
import pytest
import torch

from shared_prefix_fan_gb300 import binding
from shared_prefix_fan_gb300.workloads import WORKLOADS, draw
from tests.gpu_helpers import TOL_LSE, TOL_MAX_O, TOL_MEAN_O, DevWorkload

pytestmark = pytest.mark.gpu


def _noalloc(dw, out, lse):
    s = dw.w.spec
    return binding.attn_noalloc(dw.q, dw.k, dw.v, dw.table, s.prefix_len, dw.w.suffix_lens,
                                dw.w.q_rows, s.h_q, s.h_kv, s.page_size, s.scale, s.causal,
                                out, lse)


def _close(a_out, a_lse, b_out, b_lse):
    d = (a_out.double() - b_out.double()).abs()
    assert d.max().item() <= TOL_MAX_O and d.mean().item() <= TOL_MEAN_O
    assert (a_lse.double() - b_lse.double()).abs().max().item() <= TOL_LSE


def test_noalloc_matches_fanout_attn_on_two_calls():
    from tests.gpu_helpers import compare, oracle_ref

    for name in ("decode", "batching"):   # two calls in a row, different plans
        dw = DevWorkload(draw(WORKLOADS[name]))
        ref_out, ref_lse = dw.run()
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _noalloc(dw, out, lse) == binding.OK
        assert binding.last_error() == binding.OK
        _close(out, lse, ref_out, ref_lse)
        # and against the fp64 oracle, so a fault both entries share shows too
        compare(out, lse, *oracle_ref(dw.w), what=f"no-alloc {name}")


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")   # nothing was captured: the point
def test_noalloc_refuses_a_capturing_stream():
    """Each call copies its plan into the array from host memory that lives
    only for the call, so a call on a stream being captured is refused with
    nothing done (and the stream stays usable)."""
    dw = DevWorkload(draw(WORKLOADS["tiny"]))
    out = torch.zeros((dw.w.total_rows, dw.w.spec.h_q, 128), device="cuda")
    lse = torch.zeros((dw.w.total_rows, dw.w.spec.h_q), device="cuda")
    assert _noalloc(dw, out, lse) == binding.OK   # first call on the device: set-up
    torch.cuda.synchronize()
    out.zero_()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    s = dw.w.spec
    with torch.cuda.stream(stream):
        graph.capture_begin()
        try:
            rc = binding.attn_noalloc(dw.q, dw.k, dw.v, dw.table, s.prefix_len,
                                      dw.w.suffix_lens, dw.w.q_rows, s.h_q, s.h_kv, s.page_size,
                                      s.scale, s.causal, out, lse, stream=stream)
        finally:
            graph.capture_end()
    assert rc == binding.EUNSUPPORTED
    torch.cuda.synchronize()
    assert (out == 0).all().item()


def test_noalloc_rejects_problem_beyond_scratch():
    dw = DevWorkload(draw(WORKLOADS["batching"]))
    out = torch.zeros((dw.w.total_rows, dw.w.spec.h_q, 128), device="cuda")
    lse = torch.zeros((dw.w.total_rows, dw.w.spec.h_q), device="cuda")
    try:
        # 10 partial slots x 160 tokens x 64 heads x 520 B > the 32 MiB array
        binding.set_option(binding.OPT_SPLITS, 8)
        assert _noalloc(dw, out, lse) == binding.ENOMEM
    finally:
        binding.set_option(binding.OPT_SPLITS, 0)
    torch.cuda.synchronize()
    assert (out == 0).all().item()   # nothing ran


def test_noalloc_long_prefill():
    """A long prefill: fanout_attn cuts a few query blocks to even out the last
    wave (their partials are merged); the fixed scratch array cannot hold those
    partials, so the no-allocation entry plans without the cuts. Both give the
    same attention."""
    dw = DevWorkload(draw(WORKLOADS["prefill"]))
    ref_out, ref_lse = dw.run()
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    assert _noalloc(dw, out, lse) == binding.OK
    assert binding.last_error() == binding.OK
    _close(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("q_rows", [[1, 1, 1, 1], [8, 8, 8]], ids=["one_token", "eight_tokens"])
def test_noalloc_decode_steps(q_rows):
    """Decode steps through the no-allocation entry: it keeps the device's last
    plan while the suffix lengths move within their tiles (and plans anew when
    a range gains a tile); every step matches the fp64 oracle. With eight new
    tokens per branch each suffix range ends at its last token's causal
    position, which moves with every step."""
    import dataclasses

    import oracle
    from shared_prefix_fan_gb300.workloads import small_spec
    from tests.gpu_helpers import compare

    S0 = np.array([100, 90, 110, 100][:len(q_rows)], dtype=np.int32)
    grows = [0, 1, 2, 7, 40]
    spec = small_spec(h_q=64, h_kv=8, page_size=64, prefix_len=2048, q_rows=q_rows,
                      suffix_lens=[int(x) for x in S0 + max(grows)], permute_prefix=True,
                      permute_suffix=True, seed=78)
    dw = DevWorkload(draw(spec))
    w_max = dw.w
    for grow in grows:
        S = S0 + grow
        dw.w = dataclasses.replace(w_max, suffix_lens=S)
        out = torch.full((dw.w.total_rows, spec.h_q, 128), float("nan"), device="cuda")
        lse = torch.full((dw.w.total_rows, spec.h_q), float("nan"), device="cuda")
        assert _noalloc(dw, out, lse) == binding.OK
        assert binding.last_error() == binding.OK
        ref = oracle.attn(dw.w.q, dw.w.k_pool, dw.w.v_pool, dw.table_host, spec.prefix_len, S,
                          dw.w.q_rows, spec.h_q, spec.h_kv, spec.page_size, spec.scale, spec.causal)
        compare(out, lse, *ref, what=f"no-alloc step +{grow}")


def test_noalloc_without_lse():
    """lse = NULL through the no-allocation entry: out as with lse."""
    dw = DevWorkload(draw(WORKLOADS["decode"]))
    ref_out, ref_lse = dw.run()
    out = torch.full_like(ref_out, float("nan"))
    assert _noalloc(dw, out, None) == binding.OK
    assert binding.last_error() == binding.OK
    d = (out.double() - ref_out.double()).abs()
    assert d.max().item() <= TOL_MAX_O and d.mean().item() <= TOL_MEAN_O

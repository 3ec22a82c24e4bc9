"""The event-trace (-DGQA_TRACE) build of the library: it builds and exports
what the header declares plus gqa_trace_attach (CPU); on the GPU its results
are bit-identical to the release build's, and every CTA's stamps follow the
order in which the pipeline's steps depend on one another (one SM clock, so
stamps of different warps of a CTA compare).  The epilogue's stamps of the
last item are kept in shared memory and written at the end; slots a mode
does not stamp (the in-cluster merge's, with the combine) hold whatever that
memory held, and are not read."""
import ctypes

import numpy as np
import pytest
import torch

import gqa_decode_blackwell_gb300 as g
from gqa_decode_blackwell_gb300 import build as gbuild
from gqa_decode_blackwell_gb300 import workloads

# event indices of the trace layout [CTA][event][block], as the kernel writes them
TR_START, TR_PROD_K, TR_PROD_PLAN, TR_PROD_Q = 0, 3, 5, 6
TR_MMA_K, TR_MMA_QK, TR_MMA_P, TR_MMA_PV = 8, 9, 10, 12
TR_SM_S, TR_SM_PF = 16, 20
TR_EP_L, TR_EP_PV, TR_EP_O, TR_EP_CW, TR_EP_SENT, TR_EP_FULL, TR_EP_MERGED, TR_EP_EXIT = range(23, 31)
TR_EP_COMPUTED, TR_END, TR_EVENTS, BLOCKS = 15, 31, 32, 64


@pytest.fixture(scope="module")
def trace_lib():
    gbuild.build()
    gbuild.build_trace()
    lib = g.load_library(gbuild.TRACE_LIB)
    lib.gqa_trace_attach.argtypes = [ctypes.c_void_p]
    lib.gqa_trace_attach.restype = ctypes.c_int
    return lib


def test_trace_build_exports(trace_lib):
    for n in g.header_functions():
        assert hasattr(trace_lib, n), n
    assert hasattr(trace_lib, "gqa_trace_attach")


def _call(L, inp, out, lse, splits, causal):
    desc = g.make_desc(inp.q, inp.k_cache, causal=causal, out_dtype=out.dtype)
    need = g.gqa_decode_workspace_size(inp.q, inp.k_cache, splits, causal=causal, out_dtype=out.dtype)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=out.device)
    rc = L.gqa_decode_attn(ctypes.byref(desc), inp.q.data_ptr(), inp.k_cache.data_ptr(), inp.v_cache.data_ptr(),
                           inp.seqlens.data_ptr(), out.data_ptr(), lse.data_ptr(), splits, ws.data_ptr(), ws.numel(),
                           torch.cuda.current_stream().cuda_stream)
    assert rc == g.GQA_OK, rc


@pytest.mark.gpu
@pytest.mark.parametrize("name,splits", [("llama8b", 0), ("spec", 0), ("llama70b", 8), ("tiny", 4)])
def test_trace_stamps_follow_the_pipeline(trace_lib, name, splits):
    dev = torch.device("cuda:0")
    cfg = workloads.CONFIGS[name]
    inp = workloads.make_inputs(cfg).to(dev)
    odt = torch.float32 if cfg.out_dtype == "fp32" else torch.bfloat16
    ref_out = torch.empty(inp.q.shape, dtype=odt, device=dev)
    ref_lse = torch.empty(inp.q.shape[:3], dtype=torch.float32, device=dev)
    _call(g.lib(), inp, ref_out, ref_lse, splits, cfg.causal)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(nsm * TR_EVENTS * BLOCKS, dtype=torch.int64, device=dev)
    out, lse = torch.empty_like(ref_out), torch.empty_like(ref_lse)
    assert trace_lib.gqa_trace_attach(buf.data_ptr()) == g.GQA_OK
    try:
        _call(trace_lib, inp, out, lse, splits, cfg.causal)
        torch.cuda.synchronize()
    finally:
        trace_lib.gqa_trace_attach(None)
    assert trace_lib.gqa_decode_get_error(1) == g.GQA_OK
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), name

    desc = g.make_desc(inp.q.cpu(), inp.k_cache.cpu(), causal=cfg.causal, out_dtype=odt)
    num_ctas, mode, _, _ = g.gqa_decode_plan(desc, inp.seqlens.cpu().tolist(), splits, nsm, max_items=1)
    t = buf.view(nsm, TR_EVENTS, BLOCKS).cpu().numpy().astype(np.int64)
    working = [c for c in range(num_ctas) if t[c, TR_PROD_PLAN, 0] != 0]
    assert working, name
    assert all(t[c, TR_START, 0] == 0 for c in range(num_ctas, nsm))  # no CTA beyond the grid
    threads = (96 + 128 * (2 if cfg.q_tokens * cfg.q_heads // cfg.kv_heads <= 16 else 4))
    for c in working:
        a = t[c]
        # Orders that hold by construction: a thread's own stamps in program
        # order, and a stamp taken before the action that releases another
        # role (Q issued -> K0 issued, K0 seen -> score MMAs -> S seen ->
        # P arrival -> P seen by the value issuer) against that role's later
        # stamps; the teardown stamp after the CTA barrier bounds them all.
        chains = [
            [a[TR_START, 0], a[TR_PROD_PLAN, 0], a[TR_PROD_Q, 0], a[TR_PROD_K, 0]],   # producer
            [a[TR_PROD_Q, 0], a[TR_MMA_K, 0], a[TR_MMA_QK, 0]],                      # score issuer
            [a[TR_MMA_K, 0], a[TR_SM_S, 0], a[TR_SM_PF, 0]],                         # softmax
            [a[TR_SM_S, 0], a[TR_MMA_P, 0], a[TR_MMA_PV, 0]],                        # value issuer
        ]
        for chain in chains:
            assert all(x > 0 for x in chain), (name, c, chain)
            assert all(x <= y for x, y in zip(chain, chain[1:])), (name, c, chain)
            assert max(chain) <= a[TR_END, 0], (name, c, chain)
        assert a[TR_END, 1] == threads // 32, (name, c)        # every warp reached the teardown
        ep = [a[TR_EP_L, 0], a[TR_EP_PV, 0], a[TR_EP_O, 0]]
        if mode == 2:  # in-cluster merge: the merge's steps of the last item
            ep += [a[TR_EP_CW, 0], a[TR_EP_SENT, 0], a[TR_EP_FULL, 0], a[TR_EP_COMPUTED, 0], a[TR_EP_MERGED, 0]]
        else:
            ep += [a[TR_EP_SENT, 0]]
        ep += [a[TR_EP_EXIT, 0], a[TR_END, 0]]
        assert all(x > 0 for x in ep), (name, c, mode, ep)
        assert all(x <= y for x, y in zip(ep, ep[1:])), (name, c, mode, ep)


# ------------------------------------------------------------------ trace tool
def test_trace_tool_events_match_the_kernel():
    """gqa_decode_blackwell_gb300.trace names the kernel's TraceEvent values."""
    import os
    import re

    from gqa_decode_blackwell_gb300 import trace

    src = open(os.path.join(os.path.dirname(g.__file__), "csrc", "decode_kernel.cuh")).read()
    enum = src[src.index("enum TraceEvent"):]
    enum = enum[:enum.index("};")]
    pairs = dict((k, int(v)) for k, v in re.findall(r"TR_([A-Z0-9_]+)\s*=\s*(\d+)", enum))
    pairs.pop("EVENTS")
    assert pairs == {k: v for k, v in trace.EVENTS.items() if k != "EP_COMPUTED"}
    assert trace.NUM_EVENTS == 32 and trace.BLOCKS == int(re.search(r"kTraceBlocks = (\d+)", src).group(1))
    # the merge's compute stamp is flushed to the one free slot
    assert "(ev0) + i_ : 15," in src and trace.EVENTS["EP_COMPUTED"] == 15


def test_trace_tool_summary_of_a_synthetic_trace():
    from gqa_decode_blackwell_gb300 import trace

    E = trace.EVENTS
    t = np.zeros((4, trace.NUM_EVENTS, trace.BLOCKS), dtype=np.int64)
    for c, base in ((0, 1000), (1, 5000)):       # two working CTAs, six blocks each
        a = t[c]
        a[E["START"], 0] = base
        a[E["PROD_PLAN"], 0] = base + 100
        a[E["PROD_K"], 0] = base + 200
        a[E["MMA_K"], 0] = base + 300
        for g in range(6):
            s = base + 1000 + 500 * g
            a[E["MMA_QK"], g] = s - 50
            a[E["SM_S"], g], a[E["SM_LD"], g], a[E["SM_X"], g] = s, s + 10, s + 30
            a[E["SM_PE"], g], a[E["SM_PF"], g] = s + 60, s + 100
        a[E["END"], 0] = base + 1000 + 500 * 5 + 100 + 777
    summ = trace.summarize(t)
    assert summ["ctas"] == 2
    assert summ["start_up"]["first item"] == 100 and summ["start_up"]["first K landed"] == 300
    assert summ["softmax_per_block"] == {"S load": 10, "vote": 20, "exponent": 30, "P store": 40, "period": 500}
    assert summ["first_block"] == 100 and summ["last_P_full_to_end"] == 777


@pytest.mark.gpu
def test_trace_tool_on_the_speculative_workload():
    from gqa_decode_blackwell_gb300 import trace

    dev = torch.device("cuda:0")
    cfg = workloads.CONFIGS["spec"]
    inp = workloads.make_inputs(cfg).to(dev)
    out = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(inp.q.shape[:3], dtype=torch.float32, device=dev)
    t = trace.capture(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, out, lse, 0, causal=cfg.causal)
    summ = trace.summarize(t)
    assert summ["ctas"] == 128  # two pieces per (batch, KV head) pair, merged in clusters of two
    steps = summ["softmax_per_block"]
    assert all(v is not None and v > 0 for v in steps.values()), summ
    assert steps["period"] >= steps["S load"] + steps["vote"] + steps["exponent"] + steps["P store"], summ
    assert summ["last_P_full_to_end"] > 0 and summ["start_up"]["first K landed"] > 0, summ

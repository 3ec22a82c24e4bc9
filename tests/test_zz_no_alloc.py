"""gqa_decode_attn_static_workspace: the decode entry point for callers that
cannot allocate device memory where they call it (plugins confined to a host
framework's arena, runtimes with a fixed start-up footprint, paths that cannot
take cudaMalloc's device-wide synchronisation).  It must give the results of
gqa_decode_attn with a caller workspace, on consecutive calls that reuse the
library's one static workspace, and must refuse problems too big for it.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_decode_blackwell_gb300 as g
from gqa_decode_blackwell_gb300 import build as gbuild
from gqa_decode_blackwell_gb300 import workloads
from tests.tolerances import LSE_TOL, OUT_TOL

pytestmark = pytest.mark.gpu

STATIC_BYTES = 32 * 1024 * 1024
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build()
    g.gqa_decode_get_error(clear=True)


def _static_call(inp, out, lse, splits, causal, reduction="combine"):
    """The new entry point, straight through the C ABI."""
    desc = g.make_desc(inp.q, inp.k_cache, causal=causal, out_dtype=out.dtype, reduction=reduction)
    return g.lib().gqa_decode_attn_static_workspace(
        ctypes.byref(desc), inp.q.data_ptr(), inp.k_cache.data_ptr(), inp.v_cache.data_ptr(),
        inp.seqlens.data_ptr(), out.data_ptr(), lse.data_ptr(), splits,
        torch.cuda.current_stream().cuda_stream)


def _with_caller_workspace(inp, splits, causal, out_dtype, reduction="combine"):
    out, lse = g.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, num_splits=splits, causal=causal,
                        out_dtype=out_dtype, reduction=reduction)
    return out, lse


def _ragged_cut_down():
    """A short ragged batch whose pairs are cut into fewer pieces, some
    splits empty, than the 70B call before it left in the array: the merge
    then reads slots this call did not write, which must not matter."""
    cfg = workloads.shrink(workloads.CONFIGS["ragged"], batch=6, ragged=(1, 3000))
    inp = workloads.make_inputs(cfg)
    inp.seqlens[:2] = torch.tensor([1, 129], dtype=torch.int32)   # fewer blocks than splits
    return cfg, inp


def test_static_workspace_matches_caller_workspace_on_consecutive_calls():
    """Consecutive calls share the static array.  Both paths run the same
    plan and the same kernels, so their outputs must be bit-identical; the
    stated tolerance (2e-2 / 1e-3) would hide a stale slot that leaks in.
    The split partials go through the array with the combine kernel as the
    merge (the in-cluster merge needs no workspace at all: its case checks
    that the entry point still gives the caller-workspace result)."""
    cases = [("llama8b", 0), ("spec", 0), ("llama70b", 8), ("ragged-cut", 8), ("ragged-cut", 0), ("llama8b", 0)]
    for name, splits in cases:
        if name == "ragged-cut":
            cfg, inp = _ragged_cut_down()
            inp = inp.to(DEV)
        else:
            cfg = workloads.CONFIGS[name]
            inp = workloads.make_inputs(cfg).to(DEV)
        need = g.gqa_decode_workspace_size(inp.q, inp.k_cache, splits, causal=cfg.causal, reduction="combine")
        assert 0 < need <= STATIC_BYTES
        ref_out, ref_lse = _with_caller_workspace(inp, splits, cfg.causal, torch.bfloat16)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _static_call(inp, out, lse, splits, cfg.causal) == g.GQA_OK
        torch.cuda.synchronize()
        assert g.gqa_decode_get_error(clear=True) == g.GQA_OK
        assert not torch.isnan(out).any() and not torch.isnan(lse).any(), name
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), (name, splits)
        # within the stated tolerance as well (trivially, once bit-identical)
        d_out = (out.double() - ref_out.double()).abs().max().item()
        d_lse = (lse.double() - ref_lse.double()).abs().max().item()
        assert d_out <= OUT_TOL and d_lse <= LSE_TOL, (name, d_out, d_lse)


def test_static_workspace_refuses_problems_larger_than_it():
    # 64 splits x 1024 rows x 128 floats alone fill the 32 MiB array
    B, Hq, Hkv, d, s_max = 16, 64, 8, 128, 128
    q = torch.randn(B, 1, Hq, d, device=DEV).to(torch.bfloat16)
    k = torch.randn(B, s_max, Hkv, d, device=DEV).to(torch.bfloat16)
    sl = torch.full((B,), s_max, dtype=torch.int32, device=DEV)
    inp = workloads.DecodeInputs(None, q, k, k, sl, 0.0)
    assert g.gqa_decode_workspace_size(q, k, 64, reduction="combine") > STATIC_BYTES
    out = torch.full((B, 1, Hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, 1, Hq), float("nan"), device=DEV)
    assert _static_call(inp, out, lse, 64, False) == g.GQA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and torch.isnan(lse).all()   # nothing was launched
    # the same problem with fewer splits fits and runs
    assert _static_call(inp, out, lse, 8, False) == g.GQA_OK
    torch.cuda.synchronize()
    ref_out, ref_lse = _with_caller_workspace(inp, 8, False, torch.bfloat16)
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_static_workspace_with_in_cluster_merge():
    """Problems the automatic selection merges inside thread-block clusters
    need no workspace; the entry point then simply runs them."""
    cfg = workloads.CONFIGS["llama8b"]
    inp = workloads.make_inputs(cfg).to(DEV)
    assert g.gqa_decode_workspace_size(inp.q, inp.k_cache, 0, reduction="auto") == 0
    ref_out, ref_lse = _with_caller_workspace(inp, 0, False, torch.bfloat16, reduction="auto")
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _static_call(inp, out, lse, 0, False, reduction="auto") == g.GQA_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)

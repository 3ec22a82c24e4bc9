"""The bounds-checked (-DGQA_DEBUG) build of the library: it builds and
exports what the header declares (CPU), and on the GPU its checks never fire
on the workloads and their edge cases while its results stay bit-identical
to the release build's (the checks only skip writes that would leave their
buffer)."""
import ctypes
import math

import pytest
import torch

import gqa_decode_blackwell_gb300 as g
from gqa_decode_blackwell_gb300 import build as gbuild
from gqa_decode_blackwell_gb300 import workloads


@pytest.fixture(scope="module")
def debug_lib():
    gbuild.build()
    gbuild.build_debug()
    return g.load_library(gbuild.DEBUG_LIB)


def test_debug_build_exports_every_header_function(debug_lib):
    for n in g.header_functions():
        assert hasattr(debug_lib, n), n
    assert debug_lib.gqa_status_string(g.GQA_ERR_BOUNDS).decode() != "unknown status"


def _call(L, inp, out, lse, splits, causal, reduction, ws):
    desc = g.make_desc(inp.q, inp.k_cache, causal=causal, out_dtype=out.dtype, reduction=reduction)
    return L.gqa_decode_attn(ctypes.byref(desc), inp.q.data_ptr(), inp.k_cache.data_ptr(), inp.v_cache.data_ptr(),
                             inp.seqlens.data_ptr(), out.data_ptr(), lse.data_ptr(), splits,
                             None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(),
                             torch.cuda.current_stream().cuda_stream)


def _cases():
    dev = torch.device("cuda:0")
    out = []
    for name, splits, red in (("llama8b", 0, "auto"), ("llama70b", 8, "auto"), ("spec", 0, "auto"),
                              ("spec", 5, "combine"), ("tiny", 4, "auto")):
        cfg = workloads.CONFIGS[name]
        out.append((f"{name}-s{splits}-{red}", workloads.make_inputs(cfg).to(dev), splits, cfg.causal, red))
    cfg = workloads.shrink(workloads.CONFIGS["ragged"], batch=6, ragged=(1, 3000))
    inp = workloads.make_inputs(cfg)
    inp.seqlens[:2] = torch.tensor([0, 129], dtype=torch.int32)
    for splits, red in ((8, "combine"), (0, "auto"), (4, "cluster")):
        out.append((f"ragged-cut-s{splits}-{red}", inp.to(dev), splits, False, red))
    gen = torch.Generator().manual_seed(77)   # G = 6: LSE rows take plain stores
    q = torch.randn(3, 3, 12, 64, generator=gen).to(torch.bfloat16)
    k = torch.randn(3, 700, 2, 64, generator=gen).to(torch.bfloat16)
    v = torch.randn(3, 700, 2, 64, generator=gen).to(torch.bfloat16)
    sl = torch.tensor([700, 3, 300], dtype=torch.int32)
    odd = workloads.DecodeInputs(None, q, k, v, sl, 1 / math.sqrt(64)).to(dev)
    for splits, red in ((0, "auto"), (3, "combine"), (2, "cluster")):
        out.append((f"G6-s{splits}-{red}", odd, splits, True, red))
    gen = torch.Generator().manual_seed(78)   # head_dim 256, 32 columns
    q = torch.randn(1, 1, 32, 256, generator=gen).to(torch.bfloat16)
    k = torch.randn(1, 5000, 1, 256, generator=gen).to(torch.bfloat16)
    d256 = workloads.DecodeInputs(None, q, k, k.clone(), torch.tensor([5000], dtype=torch.int32), 1 / 16).to(dev)
    for splits, red in ((8, "combine"), (4, "cluster")):
        out.append((f"d256-s{splits}-{red}", d256, splits, False, red))
    return out


@pytest.mark.gpu
def test_debug_build_checks_stay_quiet_and_results_match(debug_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert debug_lib.gqa_decode_get_error(1) == g.GQA_OK
    for what, inp, splits, causal, red in _cases():
        for out_dtype in (torch.bfloat16, torch.float32):
            ref_out, ref_lse = g.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, num_splits=splits,
                                        causal=causal, out_dtype=out_dtype, reduction=red)
            out = torch.full_like(ref_out, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            wsb = g.gqa_decode_workspace_size(inp.q, inp.k_cache, splits, causal=causal, out_dtype=out_dtype,
                                              reduction=red)
            ws = torch.empty(wsb, dtype=torch.uint8, device=inp.q.device) if wsb else None
            assert _call(debug_lib, inp, out, lse, splits, causal, red, ws) == g.GQA_OK
            torch.cuda.synchronize()
            assert debug_lib.gqa_decode_get_error(1) == g.GQA_OK, what
            assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), (what, out_dtype)

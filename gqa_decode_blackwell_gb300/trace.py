"""Per-CTA event traces of the decode kernel, for measurement.

The -DGQA_TRACE build of the library (``build.build_trace()``) stamps the SM
clock (``clock64``) at each role's steps into a device buffer attached with
``gqa_trace_attach``: buffer[cta][event][block], uint64, with ``BLOCKS``
block slots per event (later blocks share the last slot).  Stamps of one CTA
share one clock and compare; stamps of different CTAs do not.

``capture`` runs one decode through the trace build and returns the buffer;
``summarize`` turns it into medians over the working CTAs of the start-up,
the per-block softmax phases and the drain after the last block, in cycles.

    python -m gqa_decode_blackwell_gb300.trace --config spec
"""
from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np

# The kernel's TraceEvent numbering (decode_kernel.cuh).
EVENTS = {
    "START": 0, "SETUP": 1, "PROD_WAIT": 2, "PROD_K": 3, "PROD_V": 4, "PROD_PLAN": 5, "PROD_Q": 6,
    "LENS": 7, "MMA_K": 8, "MMA_QK": 9, "MMA_P": 10, "MMA_V": 11, "MMA_PV": 12, "ITER": 13,
    "PROD_T0": 14, "EP_COMPUTED": 15, "SM_S": 16, "SM_LD": 17, "SM_X": 18, "SM_PE": 19, "SM_PF": 20,
    "SM_E0": 21, "SM_E1": 22, "EP_L": 23, "EP_PV": 24, "EP_O": 25, "EP_CW": 26, "EP_SENT": 27,
    "EP_FULL": 28, "EP_MERGED": 29, "EP_EXIT": 30, "END": 31,
}
NUM_EVENTS = 32
BLOCKS = 64


def _lib():
    from . import build, load_library

    build.build()
    build.build_trace()
    L = load_library(build.TRACE_LIB)
    L.gqa_trace_attach.argtypes = [ctypes.c_void_p]
    L.gqa_trace_attach.restype = ctypes.c_int
    return L


def capture(q, k_cache, v_cache, seqlens, out, lse, num_splits: int = 0, *, causal: bool = False,
            reduction: str = "auto", calls: int = 2) -> np.ndarray:
    """Runs gqa_decode_attn `calls` times through the trace build (the last
    call's stamps remain) and returns the stamps as int64 [SMs, 32, 64].
    The tensors are CUDA tensors as for ``gqa_decode_attn``."""
    import torch

    from . import GQA_OK, GQAError, gqa_decode_workspace_size, make_desc

    L = _lib()
    dev = q.device
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    buf = torch.zeros(nsm * NUM_EVENTS * BLOCKS, dtype=torch.int64, device=dev)
    desc = make_desc(q, k_cache, causal=causal, out_dtype=out.dtype, reduction=reduction)
    need = gqa_decode_workspace_size(q, k_cache, num_splits, causal=causal, out_dtype=out.dtype,
                                     reduction=reduction)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    if L.gqa_trace_attach(buf.data_ptr()) != GQA_OK:
        raise RuntimeError("gqa_trace_attach failed")
    try:
        for _ in range(calls):
            rc = L.gqa_decode_attn(ctypes.byref(desc), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   seqlens.data_ptr(), out.data_ptr(), 0 if lse is None else lse.data_ptr(),
                                   num_splits, ws.data_ptr(), ws.numel(), stream)
            if rc != GQA_OK:
                raise GQAError(rc, "gqa_decode_attn (trace build)")
        torch.cuda.synchronize(dev)
    finally:
        L.gqa_trace_attach(None)
    rc = L.gqa_decode_get_error(1)
    if rc != GQA_OK:
        raise GQAError(rc, "trace build: device error word")
    return buf.view(nsm, NUM_EVENTS, BLOCKS).cpu().numpy()


def _median(vals):
    vals = [v for v in vals if v is not None]
    return float(np.median(vals)) if vals else None


def summarize(t: np.ndarray) -> dict:
    """Medians over the CTAs that found a work item (cycles of each CTA's own
    clock): start-up from the grid dependency, the steady-state softmax
    phases of blocks 2.. (before the stamps' block slots run out), an item's
    first block, and the drain of the last block."""
    E = EVENTS
    working = [c for c in range(t.shape[0]) if t[c, E["START"], 0] and t[c, E["PROD_PLAN"], 0]]
    rel = {"first item": [], "first K issued": [], "first K landed": [], "first S seen": [],
           "first P full": [], "end": []}
    phases = {"S load": [], "vote": [], "exponent": [], "P store": [], "period": []}
    first_block, drain = [], []
    for c in working:
        a = t[c]
        s0 = a[E["START"], 0]
        for key, ev in (("first item", "PROD_PLAN"), ("first K issued", "PROD_K"), ("first K landed", "MMA_K"),
                        ("first S seen", "SM_S"), ("first P full", "SM_PF"), ("end", "END")):
            rel[key].append(int(a[E[ev], 0] - s0) if a[E[ev], 0] else None)
        if a[E["SM_S"], 0] and a[E["SM_PF"], 0]:
            first_block.append(int(a[E["SM_PF"], 0] - a[E["SM_S"], 0]))
        blocks = int((a[E["MMA_QK"]] != 0).sum())
        for g in range(2, min(blocks, BLOCKS) - 1):
            row = [a[E[e], g] for e in ("SM_S", "SM_LD", "SM_X", "SM_PE", "SM_PF")] + [a[E["SM_S"], g + 1]]
            if not all(row):
                continue
            ss, ld, x, pe, pf, nxt = (int(v) for v in row)
            phases["S load"].append(ld - ss)
            phases["vote"].append(x - ld)
            phases["exponent"].append(pe - x)
            phases["P store"].append(pf - pe)
            phases["period"].append(nxt - ss)
        last = min(blocks, BLOCKS) - 1
        if 0 <= last and a[E["SM_PF"], last] and a[E["END"], 0] and blocks <= BLOCKS:
            drain.append(int(a[E["END"], 0] - a[E["SM_PF"], last]))
    return {
        "ctas": len(working),
        "start_up": {k: _median(v) for k, v in rel.items()},
        "softmax_per_block": {k: _median(v) for k, v in phases.items()},
        "first_block": _median(first_block),
        "last_P_full_to_end": _median(drain),
    }


def main(argv=None):
    import torch

    from . import workloads

    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--config", default="spec", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--splits", type=int, default=None, help="num_splits (default: the workload's first)")
    ap.add_argument("--reduction", default="auto", choices=["auto", "combine", "cluster"])
    args = ap.parse_args(argv)
    cfg = workloads.CONFIGS[args.config]
    inp = workloads.make_inputs(cfg).to(torch.device("cuda", 0))
    odt = torch.float32 if cfg.out_dtype == "fp32" else torch.bfloat16
    out = torch.empty(inp.q.shape, dtype=odt, device=inp.q.device)
    lse = torch.empty(inp.q.shape[:3], dtype=torch.float32, device=inp.q.device)
    splits = cfg.num_splits[0] if args.splits is None else args.splits
    t = capture(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, out, lse, splits, causal=cfg.causal,
                reduction=args.reduction)
    print(json.dumps(summarize(t), indent=1))


if __name__ == "__main__":
    main()

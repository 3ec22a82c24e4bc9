#!/usr/bin/env python3
"""GQA decode benchmark on GB300: one JSON line on rank 0.

A step is one gqa_decode_attn call (split-KV decode kernel + LSE combine)
over one batch of seeded synthetic input already resident in HBM.  Steps
cycle through a rotating pool of distinct KV caches larger than L2 and are
replayed from CUDA graphs of back-to-back calls.  Defaults: the long-context
ragged workload (B4, 64/8 heads, d128, lengths uniform in [1024, 131072],
bf16; the largest of the five workloads), automatic splitting, one GPU.
With torchrun, every rank runs an independent replica (the work does not
shard with an exchange step) and the slowest rank's time is used.

Timing: `value` is the mean over the K timed steps (one CUDA-event pair
around them).  Beside it, `pages_method` repeats the measurement the way
"Building a Faster GQA Decode Kernel for Blackwell SM100" ("Performance
against FA4") times its kernels: the fastest of 3 round medians, 7 graph
replays per round, rounds of the full call and of the decode kernel alone
interleaved.

--impl reference times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gqa_decode_blackwell_gb300 import workloads  # noqa: E402

METRIC = "decode attn µs/call & achieved KV-read HBM GB/s (fraction of GB300 peak)"
FALLBACK_HBM_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = ["decode_kernel.cuh", "sm103_ptx.cuh", "plan.cuh"]


# ------------------------------------------------------------------ helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity for one process)."""
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def _code_only(text: str) -> str:
    """C++ source with its comments removed and whitespace runs collapsed:
    what the compiler sees, so that editing a comment keeps a profile valid."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":  # literal: copied up to its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest() -> str:
    """Digest of the decode kernel's code (comments and layout excluded)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gqa_decode_blackwell_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def ncu_fields(workload: str):
    """The machine-read fields ("- key: `value`" lines) of the committed ncu
    summary of the decode kernel on `workload`, and its path, if the summary
    was taken on the current kernel source; else (None, why)."""
    path = os.path.join(PROFILES, f"decode_kernel_{workload}.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None, "no ncu summary for this workload"
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            v = v.strip()
            if v.startswith("`") and "`" in v[1:]:  # the quoted value, without any remark after it
                v = v[1:v.index("`", 1)]
            fields[k.strip()] = v
    if fields.get("kernel_source_sha256") != kernel_source_digest():
        return None, "kernel changed since the ncu capture"
    return fields, os.path.relpath(path, ROOT)


def ncu_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source."""
    fields, src = ncu_fields(workload)
    if fields is None:
        return None, src
    try:
        return float(fields["dram_bytes_per_launch"]), src
    except (KeyError, ValueError):
        return None, "summary has no dram_bytes_per_launch"


def ncu_tensor_pct(workload: str):
    """The decode kernel's tensor-pipe utilisation (sm__pipe_tensor_cycles_active,
    % of peak sustained over the launch) from the committed ncu summary, if
    it was taken on the current kernel source; else None."""
    fields, _ = ncu_fields(workload)
    try:
        return float(fields["tensor_pipe_active_pct"]) if fields is not None else None
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ["uuid", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.samples = []
        self.window = None
        self.proc = None
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = [s for t, s in self.samples if len(s) == len(self.FIELDS)]
        if self.uuid:
            mine = [s for s in rows if self.uuid.replace("GPU-", "") in s[0]]
            rows = mine or rows
        t0, t1 = self.window or (0, float("inf"))
        inside = [s for (t, s) in self.samples if t0 - 0.25 <= t <= t1 + 0.25 and s in rows]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in use for i in range(4) if s[4 + i].lower().startswith("active")})

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[1]) for s in use if num(s[1]) is not None]
        mx = [num(s[2]) for s in use if num(s[2]) is not None]
        pw = [num(s[3]) for s in use if num(s[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------- our kernels
class GraphSteps:
    """Runs n decode calls as replays of CUDA graphs of `per` back-to-back calls."""

    def __init__(self, call, per: int, stream):
        self.call, self.per, self.stream = call, per, stream
        self.graphs = {}

    def _graph(self, n):
        if n not in self.graphs:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(gr, stream=self.stream):
                    for j in range(n):
                        self.call(j)
            self.graphs[n] = gr
        return self.graphs[n]

    def prepare(self, n: int):
        """Captures the graphs run(n) replays, so that no capture (host work
        with the GPU idle) falls inside a timed region."""
        full, rem = divmod(n, self.per)
        if full:
            self._graph(self.per)
        if rem:
            self._graph(rem)

    def run(self, n: int):
        full, rem = divmod(n, self.per)
        if full:
            gf = self._graph(self.per)
            for _ in range(full):
                gf.replay()
        if rem:
            self._graph(rem).replay()

    def replay_times_ms(self, replays: int, stream):
        """Per-call times of `replays` replays of the pool graph, each timed
        with its own CUDA-event pair on `stream`."""
        gf = self._graph(self.per)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
        for a, b in evs:
            a.record(stream)
            gf.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) / self.per for a, b in evs]


def pages_method(steps: GraphSteps, dec_steps: GraphSteps, stream, rounds: int = 3, replays: int = 7):
    """Fastest of `rounds` round medians of `replays` timed graph replays,
    rounds of the full call and of the decode kernel alone interleaved."""
    call, dec = [], []
    for _ in range(rounds):
        call.append(statistics.median(steps.replay_times_ms(replays, stream)))
        dec.append(statistics.median(dec_steps.replay_times_ms(replays, stream)))
    return min(call), min(dec)


def live_copy_pieces(dst, src, lens):
    """(destination, source) pairs for one end-to-end step: all of q and of
    the lengths, and rows [0, L_b) of each sequence's key and value cache
    ([B, capacity, Hkv, d]; a sequence's live rows are one contiguous run).
    dst and src are (q, k_cache, v_cache, seqlens) tuples of equal shapes."""
    (dq, dk, dv, ds), (hq, hk, hv, hs) = dst, src
    return [(dq, hq), (ds, hs)] + [(dc[b, :n], hc[b, :n]) for dc, hc in ((dk, hk), (dv, hv))
                                   for b, n in enumerate(lens) if n > 0]


def bench_ours(args, cfg, world, rank, local):
    import gqa_decode_blackwell_gb300 as g
    from gqa_decode_blackwell_gb300 import build as gbuild

    gbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    splits = args.splits
    in_dtype = torch.float16 if args.dtype == "fp16" else torch.bfloat16
    out_dtype = torch.float32 if cfg.out_dtype == "fp32" else in_dtype
    if args.len_div > 1:
        cfg = workloads.shrink(cfg, seqlen=max(1, cfg.seqlen // args.len_div),
                               ragged=None if cfg.ragged is None else
                               tuple(max(1, x // args.len_div) for x in cfg.ragged))
    host = workloads.make_inputs(cfg, dtype=in_dtype)
    kv_bytes = host.kv_bytes()
    alloc_bytes = host.k_cache.numel() * 2 * 2
    pool = max(2, math.ceil(args.pool_mb * 2**20 / alloc_bytes) + 1)
    base = host.to(dev)
    copies = [base] + [workloads.DecodeInputs(cfg, base.q.clone(), base.k_cache.clone(), base.v_cache.clone(),
                                              base.seqlens.clone(), base.scale) for _ in range(pool - 1)]
    out = torch.empty(base.q.shape, dtype=out_dtype, device=dev)
    lse = torch.empty(base.q.shape[:3], dtype=torch.float32, device=dev)
    red = args.reduction
    ws_bytes = g.gqa_decode_workspace_size(base.q, base.k_cache, splits, causal=cfg.causal, out_dtype=out_dtype,
                                           reduction=red)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    nc, mode, slots, _ = g.gqa_decode_plan(g.make_desc(base.q, base.k_cache, causal=cfg.causal, out_dtype=out_dtype,
                                                       reduction=red),
                                           host.seqlens.tolist(), splits, 0, max_items=1)
    launches_per_step = 1 + (1 if slots > 0 else 0)

    def attn(j):
        c = copies[j % pool]
        g.gqa_decode_attn(c.q, c.k_cache, c.v_cache, c.seqlens, out, lse, splits, ws, causal=cfg.causal,
                          reduction=red)

    def split_only(j):
        c = copies[j % pool]
        g.gqa_decode_attn_split(c.q, c.k_cache, c.v_cache, c.seqlens, out, lse, splits, ws, causal=cfg.causal,
                                reduction=red)

    stream = torch.cuda.Stream(device=dev)
    for j in range(pool):  # eager once per copy: kernel attributes, tensor maps
        attn(j)
    torch.cuda.synchronize()
    if g.gqa_decode_get_error(clear=True) != g.GQA_OK:
        raise RuntimeError("decode reported a device error during warm-up")
    steps = GraphSteps(attn, pool, stream)
    dec_steps = GraphSteps(split_only, pool, stream)
    steps.run(pool)
    dec_steps.run(pool)
    torch.cuda.synchronize()

    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.6)
    cur = torch.cuda.current_stream(dev)
    steps.prepare(args.steps)
    dec_steps.prepare(args.steps)
    steps.run(args.warmup)
    torch.cuda.synchronize()
    barrier(world, dev)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record(cur)
    steps.run(args.steps)
    ev1.record(cur)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world, dev)
    if clocks:
        clocks.mark(t0, t1)
    ms_step = ev0.elapsed_time(ev1) / args.steps
    ms_step_max = reduce_max(ms_step, world, dev)

    # decode kernel alone (same plan, same launches), for the roofline
    dec_n = args.steps
    dec_steps.run(min(args.warmup, pool))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    dec_steps.run(dec_n)
    e1.record(cur)
    torch.cuda.synchronize()
    ms_decode = e0.elapsed_time(e1) / dec_n
    pm_call, pm_dec = pages_method(steps, dec_steps, cur)
    if clocks:
        clocks.stop()
    if g.gqa_decode_get_error(clear=True) != g.GQA_OK:
        raise RuntimeError("decode reported a device error in the timed region")

    # Eager calls (no graph): host time per C-ABI call, measured on the
    # ctypes call with its arguments prepared once (argument checks, plan,
    # tensor maps, launches), and the device time per call of the same run.
    import ctypes

    lib = g.lib()
    desc = g.make_desc(base.q, base.k_cache, causal=cfg.causal, out_dtype=out_dtype, reduction=red)
    argsets = [(ctypes.byref(desc), c.q.data_ptr(), c.k_cache.data_ptr(), c.v_cache.data_ptr(),
                c.seqlens.data_ptr(), out.data_ptr(), lse.data_ptr(), splits, ws.data_ptr(),
                ws.numel(), cur.cuda_stream) for c in copies]
    n_eager = 200
    for j in range(2 * pool):
        lib.gqa_decode_attn(*argsets[j % pool])
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    q0.record(cur)
    for j in range(n_eager):
        lib.gqa_decode_attn(*argsets[j % pool])
    host_us = (time.perf_counter() - h0) * 1e6 / n_eager
    q1.record(cur)
    torch.cuda.synchronize()
    eager = {"host_us_per_call": round(host_us, 3), "us_per_call": round(q0.elapsed_time(q1) * 1e3 / n_eager, 3),
             "calls": n_eager}
    if g.gqa_decode_get_error(clear=True) != g.GQA_OK:
        raise RuntimeError("decode reported a device error in the eager calls")

    # end to end through the C ABI with pinned host buffers: each step copies
    # q, the lengths and every sequence's live key/value rows (positions
    # [0, L_b), the ones the call reads; rows past a length are left as they
    # are on the device), runs the call and reads out and lse back.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hs = (x.pin_memory() for x in (host.q, host.k_cache, host.v_cache, host.seqlens))
        dq, dk, dv, ds = (torch.empty_like(x, device=dev) for x in (hq, hk, hv, hs))
        pieces = live_copy_pieces((dq, dk, dv, ds), (hq, hk, hv, hs), host.seqlens.tolist())
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(src.numel() * src.element_size() for _, src in pieces)
        d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

        def e2e_step():
            for dst, src in pieces:
                dst.copy_(src, non_blocking=True)
            g.gqa_decode_attn(dq, dk, dv, ds, out, lse, splits, ws, causal=cfg.causal, reduction=red)
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world, dev)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(cur)
        for _ in range(args.e2e_steps):
            e2e_step()
        a1.record(cur)
        torch.cuda.synchronize()
        ms_e2e = reduce_max(a0.elapsed_time(a1) / args.e2e_steps, world, dev)
        # the copied-in result must equal, bit for bit, a call on the
        # device-resident inputs (the rows left uncopied are never read)
        g.gqa_decode_attn(base.q, base.k_cache, base.v_cache, base.seqlens, out, lse, splits, ws,
                          causal=cfg.causal, reduction=red)
        torch.cuda.synchronize()
        same = all(torch.equal(a.contiguous().view(torch.uint8), b.cpu().contiguous().view(torch.uint8))
                   for a, b in ((h_out, out), (h_lse, lse)))
        if not same or g.gqa_decode_get_error(clear=True) != g.GQA_OK:
            raise RuntimeError("end-to-end result differs from the call on device-resident inputs")
        e2e = {"value": round(world * kv_bytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(ms_e2e, 4), "steps": args.e2e_steps, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "copies": "q, lengths and each sequence's live K/V rows from pinned host memory, one stream",
               "checked": "bit-identical to the call on device-resident inputs"}

    peak, peak_kind = measured_peak()
    achieved = kv_bytes / (ms_decode * 1e-3) / 1e9
    if args.len_div == 1:
        traffic, traffic_src = ncu_traffic(cfg.name)
        tensor_pct = ncu_tensor_pct(cfg.name)
    else:
        traffic, traffic_src = None, "lengths divided for a profiling capture"
        tensor_pct = None
    roofline = {"bound": "hbm", "kernel": "gqa_decode_kernel", "achieved": round(achieved, 2), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "traffic": traffic, "traffic_source": traffic_src, "tensor_pipe_active_pct": tensor_pct,
                "us_per_launch": round(ms_decode * 1e3, 3), "algorithmic_bytes_per_launch": kv_bytes}
    value = world * kv_bytes / (ms_step_max * 1e-3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(host, cfg, args.cpu_seconds)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step_max, 5), "us_per_call": round(ms_step_max * 1e3, 3),
        "frac_of_peak": round(value / world / peak, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16" if args.dtype == "fp16" else "bf16",
        "data": f"synthetic: seeded randn rounded to {args.dtype}",
        "config": {"workload": cfg.name, "description": cfg.description, "batch": cfg.batch,
                   "q_tokens": cfg.q_tokens, "q_heads": cfg.q_heads, "kv_heads": cfg.kv_heads,
                   "head_dim": cfg.head_dim, "seqlen": cfg.seqlen if cfg.ragged is None else "ragged",
                   "seqlens_sum": int(host.seqlens.sum().item()), "kv_bytes_per_step": kv_bytes,
                   "len_div": args.len_div,
                   "num_splits": "auto" if splits == 0 else splits,
                   "plan": ["splits", "balanced", "splits merged in clusters"][mode], "reduction": red,
                   "ctas": nc, "partial_slots": slots,
                   "l2": f"rotating pool of {pool} KV caches ({pool * alloc_bytes / 1e6:.0f} MB) > 129 MB L2",
                   "launch": f"CUDA graphs of {pool} back-to-back calls, PDL between kernels",
                   "parallelism": f"replicas x{world}"},
        "pages_method": {"us_per_call": round(pm_call * 1e3, 3), "decode_kernel_us": round(pm_dec * 1e3, 3),
                         "gbs": round(kv_bytes / (pm_call * 1e-3) / 1e9, 2),
                         "frac_of_peak": round(kv_bytes / (pm_call * 1e-3) / 1e9 / peak, 4),
                         "how": "fastest of 3 round medians, 7 graph replays of the pool per round, "
                                "full-call and decode-only rounds interleaved"},
        "eager": eager,
        "roofline": roofline, "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary() if clocks else None, "e2e": e2e, "cpu_baseline": cpu,
    }
    return result


def cpu_baseline(host, cfg, seconds):
    import oracle

    cores = len(os.sched_getaffinity(0))
    orc = oracle.load()
    t = time.perf_counter()
    orc.decode(host.q, host.k_cache, host.v_cache, host.seqlens, causal=cfg.causal, nthreads=cores)
    one = time.perf_counter() - t
    reps = max(1, min(1000, int(seconds / max(one, 1e-6))))
    t = time.perf_counter()
    for _ in range(reps):
        orc.decode(host.q, host.k_cache, host.v_cache, host.seqlens, causal=cfg.causal, nthreads=cores)
    dt = time.perf_counter() - t
    return {"value": round(reps * host.kv_bytes() / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": f"the whole {cfg.name} workload, {reps} repetitions ({dt:.1f} s)"}


# ------------------------------------------------------------ reference arm
def bench_reference(args, cfg):
    import oracle

    orc = oracle.load()
    cores = len(os.sched_getaffinity(0))
    host = workloads.make_inputs(cfg, dtype=torch.float16 if args.dtype == "fp16" else torch.bfloat16)
    B = cfg.batch
    per_b = [int(L) * cfg.kv_heads * cfg.head_dim * 4 for L in host.seqlens.tolist()]

    def step(i):
        b = i % B
        orc.decode(host.q[b:b + 1], host.k_cache[b:b + 1], host.v_cache[b:b + 1], host.seqlens[b:b + 1],
                   causal=cfg.causal, nthreads=cores)
        return per_b[b]

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    nbytes = sum(step(i) for i in range(args.steps))
    dt = time.perf_counter() - t
    value = nbytes / dt / 1e9
    sample = f"one sequence (all heads) of the {cfg.name} workload per step"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded randn rounded to bf16",
        "config": {"workload": cfg.name, "description": cfg.description, "kv_bytes_per_step_mean": sum(per_b) / B},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="ragged", choices=sorted(workloads.CONFIGS) + ["all"],
                    help="the workload; 'all' prints one JSON line for each of the five in turn")
    ap.add_argument("--len-div", type=int, default=1,
                    help="divide the workload's KV lengths by this (smaller profiling captures only)")
    ap.add_argument("--splits", type=int, default=None, help="0 = automatic (default: the config's first)")
    ap.add_argument("--pool-mb", type=float, default=512.0)
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16", help="element type of q, k and v")
    ap.add_argument("--reduction", choices=["auto", "combine", "cluster"], default="auto",
                    help="how split partials are merged (auto: the library's selection)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    args = ap.parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    names = list(workloads.CONFIG_ORDER) if args.config == "all" else [args.config]
    splits_arg = args.splits
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            for name in names:
                cfg = workloads.CONFIGS[name]
                args.splits = cfg.num_splits[0] if splits_arg is None else splits_arg
                print(json.dumps(bench_reference(args, cfg)), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        for name in names:
            cfg = workloads.CONFIGS[name]
            args.splits = cfg.num_splits[0] if splits_arg is None else splits_arg
            res = bench_ours(args, cfg, world, rank, local)
            if rank == 0:
                print(json.dumps(res), flush=True)
            del res
            torch.cuda.empty_cache()
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""GPU parity: the sm_103a kernels, called through the C ABI, against the fp64
oracle on the same seeded inputs.

Tolerances: max |O_gpu - O_oracle| <= 2e-2 (bf16 or fp32 output) and
max |lse_gpu - lse_oracle| <= 1e-3, with -inf LSEs matching exactly.  Beside
that stated bar every comparison also asserts a regression bound a few times
the error these kernels show: per element |dO| <= REG_ABS (REG_LONG on the
long workloads) + one 16-bit ulp of |O_oracle| (for 16-bit outputs; the
rounding of the output itself) and
|dlse| <= REG_LSE, so that a change which stays under the stated bar but
breaks part of the arithmetic (a lost block at long lengths) still fails.
Setting GQA_PARITY_LOG=<path> appends each comparison's errors to a JSON-lines
file.
"""
import functools
import json
import math
import os

import numpy as np
import pytest
import torch

import gqa_decode_blackwell_gb300 as g
import oracle
from gqa_decode_blackwell_gb300 import build as gbuild
from gqa_decode_blackwell_gb300 import workloads
# the stated bar and the regression bounds, derived from the kernel's arithmetic
from tests.tolerances import LSE_TOL, OUT_TOL, REG_ABS, REG_LONG, REG_LSE

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build()
    g.gqa_decode_get_error(clear=True)
    yield
    assert g.gqa_decode_get_error(clear=True) in (g.GQA_OK,)


def ulp16(x, dtype):
    """One ulp of a 16-bit float type at |x| (0 for fp32 outputs)."""
    if dtype == torch.float32:
        return np.zeros_like(x)
    mant = 7 if dtype == torch.bfloat16 else 10
    ax = np.maximum(np.abs(x), 2.0 ** -126 if dtype == torch.bfloat16 else 2.0 ** -14)
    return np.exp2(np.floor(np.log2(ax)) - mant)


def _log(record):
    path = os.environ.get("GQA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(record) + "\n")


def assert_close(out, lse, ref_out, ref_lse, what="", reg_abs=REG_ABS, reg_lse=REG_LSE):
    o = out.detach().double().cpu().numpy()
    l = lse.detach().double().cpu().numpy()
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    inf_ref = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), inf_ref), f"{what}: -inf LSE pattern differs"
    diff = np.abs(o - ref_out)
    err_o = float(diff.max()) if o.size else 0.0
    err_l = float(np.abs(l[~inf_ref] - ref_lse[~inf_ref]).max()) if (~inf_ref).any() else 0.0
    # error beyond the rounding of the output to its 16-bit type
    excess = diff - ulp16(ref_out, out.dtype)
    err_x = float(excess.max()) if o.size else 0.0
    rms = float(np.sqrt(np.mean(ref_out ** 2))) if o.size else 0.0
    _log({"what": what, "dtype": str(out.dtype), "max_dO": err_o, "max_dO_beyond_ulp": err_x,
          "max_dlse": err_l, "rms_O": rms})
    assert err_o <= OUT_TOL and err_l <= LSE_TOL, f"{what}: max|dO| {err_o:.3e}, max|dlse| {err_l:.3e}"
    assert err_x <= reg_abs and err_l <= reg_lse, \
        f"{what}: regression bound: max(|dO| - ulp) {err_x:.3e} > {reg_abs:.1e} or max|dlse| {err_l:.3e} > {reg_lse:.1e}"
    return err_o, err_l


def run_gpu(inp, splits, out_dtype=torch.bfloat16, causal=False, scale=0.0, reduction="auto"):
    d = inp if inp.q.is_cuda else inp.to(DEV)
    out, lse = g.decode(d.q, d.k_cache, d.v_cache, d.seqlens, num_splits=splits, causal=causal, scale=scale,
                        out_dtype=out_dtype, reduction=reduction)
    torch.cuda.synchronize()
    assert g.gqa_decode_get_error(clear=True) == g.GQA_OK
    return out, lse


@functools.lru_cache(maxsize=2)
def config_case(name):
    cfg = workloads.CONFIGS[name]
    inp = workloads.make_inputs(cfg)
    ref = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, causal=cfg.causal)
    return cfg, inp.to(DEV), ref


# (workload, num_splits, reduction): the automatic choices, then the in-cluster
# merge forced on and the combine kernel forced on for every workload
FULL = [("tiny", 1, "auto"), ("tiny", 4, "auto"), ("tiny", 0, "auto"), ("llama8b", 0, "auto"),
        ("llama8b", 1, "auto"), ("llama8b", 16, "auto"), ("llama70b", 8, "auto"), ("llama70b", 0, "auto"),
        ("spec", 0, "auto"), ("spec", 1, "auto"), ("spec", 5, "auto"), ("ragged", 0, "auto"), ("ragged", 8, "auto"),
        ("tiny", 0, "cluster"), ("tiny", 4, "combine"), ("llama8b", 0, "cluster"), ("llama8b", 0, "combine"),
        ("llama8b", 4, "cluster"), ("llama70b", 8, "cluster"), ("llama70b", 0, "cluster"), ("spec", 0, "cluster"),
        ("spec", 0, "combine"), ("spec", 2, "cluster"), ("ragged", 0, "cluster"), ("ragged", 8, "cluster")]


@pytest.mark.parametrize("name,splits,reduction", FULL, ids=[f"{n}-s{s}-{r}" for n, s, r in FULL])
def test_config_full_size(name, splits, reduction):
    """Every element of every config at full size (the oracle is C, fp64, threaded)."""
    cfg, inp, (ref_out, ref_lse) = config_case(name)
    out_dtype = torch.float32 if cfg.out_dtype == "fp32" else torch.bfloat16
    out, lse = run_gpu(inp, splits, out_dtype, cfg.causal, reduction=reduction)
    assert_close(out, lse, ref_out, ref_lse, f"{name} splits={splits} {reduction}",
                 reg_abs=REG_ABS if name == "tiny" else REG_LONG)
    again = run_gpu(inp, splits, out_dtype, cfg.causal, reduction=reduction)
    assert torch.equal(out, again[0]) and torch.equal(lse, again[1]), "not bit-identical on repeat"


def _nan_tail_inputs(lens, s_max, nq, Hq, Hkv, d, seed, dtype=torch.bfloat16):
    gen = torch.Generator().manual_seed(seed)
    B = len(lens)
    q = torch.randn(B, nq, Hq, d, generator=gen).to(dtype)
    k = torch.randn(B, s_max, Hkv, d, generator=gen).to(dtype)
    v = torch.randn(B, s_max, Hkv, d, generator=gen).to(dtype)
    for b, L in enumerate(lens):   # cache positions past the sequence hold NaN
        k[b, max(L, 0):] = float("nan")
        v[b, max(L, 0):] = float("nan")
    return q, k, v, torch.tensor(lens, dtype=torch.int32)


# head columns nq * G: 2, 4, 8 and 12 (16-column kernels: the second 8-column
# softmax warpgroup partly or wholly padding), 16, 18 and 20 (32-column
# kernels whose last warpgroup holds only padding) and 32
EDGE = [(64, 4, 1, False), (64, 8, 4, True), (128, 4, 1, False), (128, 8, 1, False), (128, 8, 4, True),
        (128, 16, 2, True), (64, 2, 1, False), (128, 12, 1, False), (128, 16, 1, False), (64, 5, 4, True),
        (64, 6, 3, True), (256, 4, 1, False), (256, 8, 1, True), (256, 16, 2, True), (256, 6, 3, True)]


@pytest.mark.parametrize("d,G,nq,causal", EDGE, ids=[f"d{a}-G{b}-nq{c}-{'c' if e else 'n'}" for a, b, c, e in EDGE])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_edge_lengths_and_poisoned_tail(d, G, nq, causal, splits):
    """Lengths 1, 127, 128, 129, 4097 and 0; every cache position past a
    sequence's end is NaN, so any read of it (or 0 * NaN) would show."""
    lens = [1, 127, 128, 129, 4097, 0, nq]
    Hkv = 2
    q, k, v, sl = _nan_tail_inputs(lens, 4200, nq, G * Hkv, Hkv, d, seed=100 + d + G + nq)
    ref_out, ref_lse = oracle.decode(q, k, v, sl, causal=causal)
    out, lse = run_gpu(workloads.DecodeInputs(None, q, k, v, sl, 1 / math.sqrt(d)).to(DEV), splits,
                       torch.float32, causal)
    assert_close(out, lse, ref_out, ref_lse, f"edge d={d} G={G} nq={nq} causal={causal} splits={splits}")


@pytest.mark.parametrize("d,G,nq,causal", EDGE, ids=[f"d{a}-G{b}-nq{c}-{'c' if e else 'n'}" for a, b, c, e in EDGE])
@pytest.mark.parametrize("splits", [0, 2, 4, 8])
def test_edge_lengths_cluster_merge(d, G, nq, causal, splits):
    """The same poisoned-tail edge lengths with the in-cluster merge forced:
    pieces past a short sequence's blocks are empty and must drop out."""
    lens = [1, 127, 128, 129, 4097, 0, nq]
    Hkv = 2
    q, k, v, sl = _nan_tail_inputs(lens, 4200, nq, G * Hkv, Hkv, d, seed=100 + d + G + nq)
    ref_out, ref_lse = oracle.decode(q, k, v, sl, causal=causal)
    inp = workloads.DecodeInputs(None, q, k, v, sl, 1 / math.sqrt(d)).to(DEV)
    for out_dtype in (torch.float32, torch.bfloat16):
        out, lse = run_gpu(inp, splits, out_dtype, causal, reduction="cluster")
        assert_close(out, lse, ref_out, ref_lse,
                     f"cluster edge d={d} G={G} nq={nq} causal={causal} splits={splits} {out_dtype}")


def test_lse_off_16_bytes_cluster_merge():
    """An lse output that is only 4-byte aligned: the merged LSEs take plain stores."""
    lens = [300, 5, 129, 1000]
    q, k, v, sl = _nan_tail_inputs(lens, 1000, 1, 16, 2, 128, seed=9)
    ref_out, ref_lse = oracle.decode(q, k, v, sl)
    d = workloads.DecodeInputs(None, q, k, v, sl, 0).to(DEV)
    out = torch.empty(d.q.shape, dtype=torch.bfloat16, device=DEV)
    lse_store = torch.empty(d.q.shape[:3].numel() + 1, device=DEV)
    lse = lse_store[1:].view(d.q.shape[:3])
    g.gqa_decode_attn(d.q, d.k_cache, d.v_cache, d.seqlens, out, lse, 4, None, reduction="cluster")
    torch.cuda.synchronize()
    assert g.gqa_decode_get_error(clear=True) == g.GQA_OK
    assert_close(out, lse, ref_out, ref_lse, "cluster merge, lse at +4 bytes")


def test_more_splits_than_blocks():
    q, k, v, sl = _nan_tail_inputs([300, 5, 129], 300, 1, 8, 2, 128, seed=7)
    ref = oracle.decode(q, k, v, sl)
    for splits in (16, 64):
        out, lse = run_gpu(workloads.DecodeInputs(None, q, k, v, sl, 0).to(DEV), splits, torch.bfloat16)
        assert_close(out, lse, *ref, f"splits={splits}")


def test_scale_override_and_bf16_fp32_outputs():
    cfg = workloads.shrink(workloads.CONFIGS["llama8b"], batch=2, seqlen=700)
    inp = workloads.make_inputs(cfg)
    ref = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, scale=0.3)
    for dt in (torch.bfloat16, torch.float32):
        out, lse = run_gpu(inp, 0, dt, scale=0.3)
        assert_close(out, lse, *ref, f"scale 0.3 {dt}")


@pytest.mark.parametrize("reduction", ["auto", "combine", "cluster"])
def test_deterministic_bitwise(reduction):
    cfg, inp, _ = config_case("llama8b")
    a = run_gpu(inp, 0, reduction=reduction)
    b = run_gpu(inp, 0, reduction=reduction)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_splitkv_partials_then_combine():
    cfg = workloads.shrink(workloads.CONFIGS["spec"], batch=5, seqlen=1000)
    inp = workloads.make_inputs(cfg)
    inp.seqlens[:] = torch.tensor([1000, 513, 4, 129, 257], dtype=torch.int32)
    S = 3
    begin, end = oracle.split_ranges(inp.seqlens.tolist(), S)
    parts = [oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, causal=True, pos_begin=begin[s],
                           pos_end=end[s]) for s in range(S)]
    ref_full = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, causal=True)
    d = inp.to(DEV)
    B, nq, Hq, D = d.q.shape
    o_part = torch.full((S, B, nq, Hq, D), float("nan"), device=DEV)
    lse_part = torch.empty(S, B, nq, Hq, device=DEV)
    g.gqa_decode_splitkv(d.q, d.k_cache, d.v_cache, d.seqlens, S, o_part, lse_part, causal=True)
    torch.cuda.synchronize()
    for s in range(S):
        ref_o, ref_l = parts[s]
        valid = ~np.isneginf(ref_l)
        o = o_part[s].double().cpu().numpy()
        l = lse_part[s].double().cpu().numpy()
        assert np.array_equal(np.isneginf(l), ~valid)
        assert np.abs(o[valid] - ref_o[valid]).max() <= OUT_TOL
        assert np.abs(l[valid] - ref_l[valid]).max() <= LSE_TOL
    out = torch.empty(B, nq, Hq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, nq, Hq, device=DEV)
    g.gqa_decode_combine(o_part, lse_part, out, lse)
    torch.cuda.synchronize()
    assert_close(out, lse, *ref_full, "splitkv + combine")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_combine_against_oracle(d, out_dtype):
    rng = np.random.default_rng(d)
    S, rows = 7, 300
    o = rng.standard_normal((S, rows, d)).astype(np.float32)
    l = (rng.standard_normal((S, rows)) * 3).astype(np.float32)
    l[rng.random((S, rows)) < 0.3] = -np.inf
    l[:, :5] = -np.inf                       # rows with no valid split
    o[np.broadcast_to(np.isneginf(l)[..., None], o.shape)] = np.nan   # must never be read
    ref_out, ref_lse = oracle.combine(o, l)
    ref_out = np.nan_to_num(ref_out)
    out = torch.empty(rows, d, dtype=out_dtype, device=DEV)
    lse = torch.empty(rows, device=DEV)
    g.gqa_decode_combine(torch.from_numpy(o).to(DEV), torch.from_numpy(l).to(DEV), out, lse)
    torch.cuda.synchronize()
    assert_close(out, lse, ref_out, ref_lse, "combine")


def test_head_map_golden_on_gpu():
    with open(os.path.join(GOLDEN, "gqa_head_groups.json")) as f:
        gold = json.load(f)
    for ex in gold["examples"]:
        Hq, Hkv = ex["num_qo_heads"], ex["num_kv_heads"]
        if Hq // Hkv > 32:
            continue
        gen = torch.Generator().manual_seed(3)
        q = torch.randn(1, 1, Hq, 128, generator=gen).to(torch.bfloat16)
        k = torch.randn(1, 200, Hkv, 128, generator=gen).to(torch.bfloat16)
        v = torch.arange(1, Hkv + 1, dtype=torch.float32).view(1, 1, Hkv, 1).expand(1, 200, Hkv, 128)
        v = v.contiguous().to(torch.bfloat16)
        out, _ = run_gpu(workloads.DecodeInputs(None, q, k, v, torch.tensor([200], dtype=torch.int32), 0), 0,
                         torch.float32)
        got = [int(round(float(out[0, 0, hq, 0]))) - 1 for hq in range(Hq)]
        assert got == ex["kv_head_of_q_head"]


@pytest.mark.parametrize("reduction", ["auto", "combine"])
def test_graph_capture_and_replay(reduction):
    """Captured once, replayed on new inputs (auto: the in-cluster merge,
    clusters of four on this shape)."""
    cfg = workloads.shrink(workloads.CONFIGS["llama8b"], batch=4, seqlen=1500)
    a = workloads.make_inputs(cfg).to(DEV)
    b = workloads.make_inputs(cfg, seed=99)
    ref_b = oracle.decode(b.q, b.k_cache, b.v_cache, b.seqlens)
    out = torch.empty(a.q.shape, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(a.q.shape[:3], device=DEV)
    ws_bytes = g.gqa_decode_workspace_size(a.q, a.k_cache, 0, reduction=reduction)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=DEV)
    # warm-up outside capture
    g.gqa_decode_attn(a.q, a.k_cache, a.v_cache, a.seqlens, out, lse, 0, ws, reduction=reduction)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.gqa_decode_attn(a.q, a.k_cache, a.v_cache, a.seqlens, out, lse, 0, ws, reduction=reduction)
    a.q.copy_(b.q); a.k_cache.copy_(b.k_cache); a.v_cache.copy_(b.v_cache); a.seqlens.copy_(b.seqlens)
    graph.replay()
    torch.cuda.synchronize()
    assert_close(out, lse, *ref_b, "graph replay")


def test_bad_seqlen_is_clamped_and_flagged():
    q, k, v, sl = _nan_tail_inputs([50, 90], 100, 1, 4, 1, 64, seed=5)
    k[:] = torch.randn(k.shape).to(torch.bfloat16)
    v[:] = torch.randn(v.shape).to(torch.bfloat16)
    bad = torch.tensor([500, -3], dtype=torch.int32)
    ref = oracle.decode(q, k, v, [100, 0])
    d = workloads.DecodeInputs(None, q, k, v, bad, 0).to(DEV)
    out, lse = g.decode(d.q, d.k_cache, d.v_cache, d.seqlens, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert g.gqa_decode_get_error(clear=True) == g.GQA_ERR_BAD_SEQLEN
    assert_close(out, lse, *ref, "clamped lengths")


def test_timeout_selftest_reports_and_context_survives():
    """A bounded wait on a barrier nothing completes returns an error status;
    the context stays usable for the next decode."""
    g.gqa_decode_selftest_timeout(20000)
    assert g.gqa_decode_get_error(clear=True) == g.GQA_ERR_TIMEOUT
    assert g.gqa_decode_get_error(clear=True) == g.GQA_OK
    cfg, inp, ref = config_case("tiny")
    out, lse = run_gpu(inp, 4, torch.float32)
    assert_close(out, lse, *ref, "after timeout")


def test_empty_batch():
    q = torch.empty(0, 1, 8, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.empty(0, 16, 2, 128, dtype=torch.bfloat16, device=DEV)
    sl = torch.empty(0, dtype=torch.int32, device=DEV)
    out = torch.empty(0, 1, 8, 128, dtype=torch.bfloat16, device=DEV)
    g.gqa_decode_attn(q, k, k, sl, out)
    torch.cuda.synchronize()


@pytest.mark.parametrize("reduction", ["auto", "combine"])
def test_split_then_merge_equals_attn(reduction):
    cfg, inp, ref = config_case("llama8b")
    out = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(inp.q.shape[:3], device=DEV)
    ws_bytes = g.gqa_decode_workspace_size(inp.q, inp.k_cache, 0, reduction=reduction)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=DEV)
    g.gqa_decode_attn_split(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, out, lse, 0, ws, reduction=reduction)
    g.gqa_decode_attn_merge(inp.q, inp.k_cache, out, lse, 0, ws, reduction=reduction)
    torch.cuda.synchronize()
    assert_close(out, lse, *ref, "split + merge")
    a_out, a_lse = run_gpu(inp, 0, reduction=reduction)
    assert torch.equal(out, a_out) and torch.equal(lse, a_lse)


def _random_batch(B, s_max, nq, Hq, Hkv, d, seed, lo=0):
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(lo, s_max + 1, (B,), generator=gen).to(torch.int32)
    q = torch.randn(B, nq, Hq, d, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, s_max, Hkv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, s_max, Hkv, d, generator=gen).to(torch.bfloat16)
    return workloads.DecodeInputs(None, q, k, v, lens, 0)


def test_many_items_per_cta_walk_the_plan_iterator():
    """400 sequences x 4 KV heads x 16 splits = 25600 items: more than a CTA's
    shared-memory item list holds, so the kernel walks its plan iterator."""
    inp = _random_batch(400, 300, 1, 8, 4, 128, seed=31)
    ref = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens)
    out, lse = run_gpu(inp, 16, torch.float32)
    assert_close(out, lse, *ref, "25600 split items")


@pytest.mark.parametrize("splits", [0, 3, 4])
def test_batch_larger_than_shared_length_table(splits):
    """600 sequences: lengths are read from global memory and the automatic
    mode uses fixed splits."""
    inp = _random_batch(600, 200, 2, 8, 2, 64, seed=32, lo=1)
    ref = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, causal=True)
    out, lse = run_gpu(inp, splits, torch.bfloat16, causal=True)
    assert_close(out, lse, *ref, f"B=600 splits={splits}")


def test_one_long_pair_more_than_64_pieces():
    """One sequence on one KV head, 256 blocks over 152 CTAs: the balanced plan
    cuts it into more pieces than the 64 the combine keeps in registers, so
    the combine takes its many-splits loop."""
    inp = _random_batch(1, 32768, 1, 4, 1, 128, seed=41, lo=32768)
    desc = g.make_desc(inp.q, inp.k_cache)
    C, mode, slots, items = g.gqa_decode_plan(desc, inp.seqlens.tolist(), 0, 0)
    assert mode == 1 and max(int(r[7]) for r in items) > 64
    ref = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens)
    out, lse = run_gpu(inp, 0, torch.float32)
    assert_close(out, lse, *ref, "one pair, 256 blocks")


# ------------------------------------------------- long-length block addressing
def _hot_block_inputs(lens, s_max, nq, Hq, Hkv, d, hot, seed):
    """Keys of one 128-position block per (b, KV head) point along q (equal
    scores of ~22.6), every other key is small noise (scores ~N(0, 0.01)): the softmax
    mass of the hot block outweighs the rest by >10^6, so O is close to the
    mean of V over that block and any mis-addressed K or V block shows as an
    O.(1) error.  Cache positions past a sequence's end hold NaN."""
    gen = torch.Generator().manual_seed(seed)
    B = len(lens)
    q = torch.ones(B, nq, Hq, d).to(torch.bfloat16)
    k = (torch.randn(B, s_max, Hkv, d, generator=gen) * 0.1)
    v = torch.randn(B, s_max, Hkv, d, generator=gen)
    for b in range(B):
        for h in range(Hkv):
            blk = hot[b][h]
            k[b, blk * 128:(blk + 1) * 128, h, :] = 2.0 * math.sqrt(128 / d)
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    for b, L in enumerate(lens):
        k[b, L:] = float("nan")
        v[b, L:] = float("nan")
    return q, k, v, torch.tensor(lens, dtype=torch.int32)


LONG = [
    # d, nq, G, causal, lens, hot blocks per (b, h)
    (128, 1, 4, False, [131072, 100003, 65537], [[0, 1023], [781, 390], [512, 257]]),
    (64, 2, 4, True, [70001, 33333, 129], [[546, 0], [260, 100], [1, 0]]),
]


@pytest.mark.parametrize("case", range(len(LONG)), ids=[f"d{c[0]}-nq{c[1]}" for c in LONG])
@pytest.mark.parametrize("splits,reduction", [(0, "auto"), (1, "auto"), (8, "auto"), (64, "auto"),
                                              (0, "cluster"), (8, "cluster")])
def test_long_sequence_block_addressing(case, splits, reduction):
    d, nq, G, causal, lens, hot = LONG[case]
    Hkv = 2
    q, k, v, sl = _hot_block_inputs(lens, max(lens), nq, G * Hkv, Hkv, d, hot, seed=500 + case)
    key = (case,)
    if key not in _LONG_REF:
        _LONG_REF.clear()
        _LONG_REF[key] = oracle.decode(q, k, v, sl, causal=causal)
    ref_out, ref_lse = _LONG_REF[key]
    # closed form, independent of the oracle: for the first new token, O is
    # the mean of V over the hot block's visible rows (equal scores there; the
    # other keys carry < 1e-5 of the mass)
    for b, L in enumerate(lens):
        vis0 = L - (nq - 1) if causal else L
        for h in range(Hkv):
            lo, hi = hot[b][h] * 128, min((hot[b][h] + 1) * 128, vis0)
            if hi <= lo:
                continue
            mean_v = v[b, lo:hi, h, :].double().mean(0).numpy()
            assert np.abs(ref_out[b, 0, h * G:(h + 1) * G, :] - mean_v).max() < 1e-3, (b, h)
    inp = workloads.DecodeInputs(None, q, k, v, sl, 1 / math.sqrt(d)).to(DEV)
    out, lse = run_gpu(inp, splits, torch.float32, causal, reduction=reduction)
    assert_close(out, lse, ref_out, ref_lse, f"long d={d} nq={nq} splits={splits} {reduction}", reg_abs=REG_LONG)


_LONG_REF = {}


# ------------------------------------------------------------- head_dim 256
# The page's split-reduction trace shape ("Building a Faster GQA Decode Kernel
# for Blackwell SM100", "The final split reduction trace"): batch 1, one query
# token, 32 query heads on one KV head, 32768 positions, eight splits, head
# dimension 256 -- and a 16-column shape with ragged lengths.
@functools.lru_cache(maxsize=1)
def d256_case(which):
    inp = workloads.head_dim_256_inputs(which)
    ref = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens)
    return inp.to(DEV), ref


D256 = [(0, 8, "auto"), (0, 8, "combine"), (0, 0, "auto"), (0, 1, "auto"), (0, 4, "cluster"),
        (1, 0, "auto"), (1, 3, "auto"), (1, 4, "cluster"), (1, 0, "cluster")]


@pytest.mark.parametrize("which,splits,reduction", D256, ids=[f"c{w}-s{s}-{r}" for w, s, r in D256])
def test_head_dim_256(which, splits, reduction):
    """head_dim 256: K and V blocks stream as two 128-element d-halves, the
    scores accumulate over both, O lives in two TMEM accumulators."""
    inp, (ref_out, ref_lse) = d256_case(which)
    for out_dtype in (torch.bfloat16, torch.float32):
        out, lse = run_gpu(inp, splits, out_dtype, reduction=reduction)
        assert_close(out, lse, ref_out, ref_lse, f"d256 case {which} splits={splits} {reduction} {out_dtype}",
                     reg_abs=REG_LONG)
    again = run_gpu(inp, splits, torch.float32, reduction=reduction)
    assert torch.equal(out, again[0]) and torch.equal(lse, again[1])


def test_head_dim_256_splitkv_then_combine():
    inp, (ref_out, ref_lse) = d256_case(1)
    B, nq, Hq, D = inp.q.shape
    S = 5
    o_part = torch.full((S, B, nq, Hq, D), float("nan"), device=DEV)
    lse_part = torch.empty(S, B, nq, Hq, device=DEV)
    g.gqa_decode_splitkv(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, S, o_part, lse_part)
    out = torch.empty(B, nq, Hq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, nq, Hq, device=DEV)
    g.gqa_decode_combine(o_part, lse_part, out, lse)
    torch.cuda.synchronize()
    assert_close(out, lse, ref_out, ref_lse, "d256 splitkv + combine", reg_abs=REG_LONG)


# ------------------------------------------------------------------ fp16 inputs
@functools.lru_cache(maxsize=2)
def fp16_case(name):
    cfg = workloads.CONFIGS[name]
    inp = workloads.make_inputs(cfg, dtype=torch.float16)
    ref = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, causal=cfg.causal)
    return cfg, inp.to(DEV), ref


FP16 = [("llama8b", 0, torch.float16), ("llama8b", 1, torch.float16), ("spec", 0, torch.float16),
        ("spec", 5, torch.float32), ("tiny", 4, torch.float16), ("ragged", 0, torch.float32),
        ("llama8b", 16, torch.float16)]


@pytest.mark.parametrize("name,splits,out_dtype", FP16, ids=[f"{n}-s{s}-{str(o)[6:]}" for n, s, o in FP16])
def test_fp16_inputs_full_size(name, splits, out_dtype):
    """fp16 q, k, v (P enters the value MMA in fp16) at full config size,
    with fp16 and fp32 outputs."""
    cfg, inp, (ref_out, ref_lse) = fp16_case(name)
    out, lse = run_gpu(inp, splits, out_dtype, cfg.causal)
    assert out.dtype == out_dtype
    assert_close(out, lse, ref_out, ref_lse, f"fp16 {name} splits={splits} out={out_dtype}",
                 reg_abs=REG_ABS if name == "tiny" else REG_LONG)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp16_edge_lengths_and_poisoned_tail(d):
    lens = [1, 127, 128, 129, 4097, 0, 4]
    q, k, v, sl = _nan_tail_inputs(lens, 4200, 4, 16, 2, d, seed=300 + d, dtype=torch.float16)
    ref = oracle.decode(q, k, v, sl, causal=True)
    for splits in (0, 3):
        out, lse = run_gpu(workloads.DecodeInputs(None, q, k, v, sl, 1 / math.sqrt(d)).to(DEV), splits,
                           torch.float16, True)
        assert_close(out, lse, *ref, f"fp16 edge d={d} splits={splits}")


def test_fp16_splitkv_then_combine_to_fp16():
    cfg = workloads.shrink(workloads.CONFIGS["llama8b"], batch=3, seqlen=900)
    inp = workloads.make_inputs(cfg, dtype=torch.float16)
    ref = oracle.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens)
    d = inp.to(DEV)
    B, nq, Hq, D = d.q.shape
    S = 4
    o_part = torch.empty((S, B, nq, Hq, D), device=DEV)
    lse_part = torch.empty(S, B, nq, Hq, device=DEV)
    g.gqa_decode_splitkv(d.q, d.k_cache, d.v_cache, d.seqlens, S, o_part, lse_part)
    out = torch.empty(B, nq, Hq, D, dtype=torch.float16, device=DEV)
    lse = torch.empty(B, nq, Hq, device=DEV)
    g.gqa_decode_combine(o_part, lse_part, out, lse)
    torch.cuda.synchronize()
    assert_close(out, lse, *ref, "fp16 splitkv + combine")


def test_mixed_types_are_rejected():
    cfg = workloads.shrink(workloads.CONFIGS["llama8b"], batch=1, seqlen=256)
    inp = workloads.make_inputs(cfg).to(DEV)
    with pytest.raises(ValueError):
        g.decode(inp.q.to(torch.float16), inp.k_cache, inp.v_cache, inp.seqlens)
    # a 16-bit output of the other 16-bit type
    with pytest.raises(g.GQAError) as e:
        g.decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, out_dtype=torch.float16)
    assert e.value.status == g.GQA_ERR_UNSUPPORTED

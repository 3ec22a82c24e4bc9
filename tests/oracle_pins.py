"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` handle and raises
``AssertionError`` when the handle disagrees with a fact fixed by the pages
or by mathematics: closed forms, invariants, exact special cases, a library
special case (PyTorch SDPA in fp64) and the pages' own worked GQA example.
``test_oracle_pins.py`` runs them on the real oracle; ``test_oracle_mutants.py``
runs them on builds with one planted mistake each and requires that some pin
rejects every mutant.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle as oracle_mod

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _rand_bf16(gen, *shape, scale=1.0):
    return (torch.randn(*shape, generator=gen) * scale).to(torch.bfloat16)


def _int_bf16(gen, lo, hi, *shape):
    """Small integers: exact in bf16, so shifted/scaled copies stay exact."""
    return torch.randint(lo, hi + 1, shape, generator=gen).to(torch.bfloat16)


# ------------------------------------------------------------ brute force
def pin_bruteforce_tiny(orc):
    """Tiny shapes against a pure-Python loop over the definition."""
    gen = torch.Generator().manual_seed(11)
    B, nq, Hq, Hkv, d, S_max = 2, 2, 4, 2, 4, 8
    q = _rand_bf16(gen, B, nq, Hq, d)
    k = _rand_bf16(gen, B, S_max, Hkv, d)
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    seqlens = [5, 8]
    for causal in (False, True):
        out, lse = orc.decode(q, k, v, seqlens, causal=causal, nthreads=2)
        qf, kf, vf = q.double().tolist(), k.double().tolist(), v.double().tolist()
        scale = 1.0 / math.sqrt(d)
        for b in range(B):
            L = seqlens[b]
            for t in range(nq):
                for hq in range(Hq):
                    h = hq // (Hq // Hkv)
                    keys = [j for j in range(L) if (not causal) or j <= L - nq + t]
                    scores = [scale * sum(qf[b][t][hq][x] * kf[b][j][h][x] for x in range(d)) for j in keys]
                    mx = max(scores)
                    ws = [math.exp(s - mx) for s in scores]
                    z = sum(ws)
                    ref = [sum(w * vf[b][j][h][x] for w, j in zip(ws, keys)) / z for x in range(d)]
                    assert np.allclose(out[b, t, hq], ref, rtol=0, atol=1e-12), (b, t, hq)
                    assert abs(lse[b, t, hq] - (mx + math.log(z))) < 1e-12


# ------------------------------------------------------- library special case
def _sdpa_reference(q, k, v, seqlens, causal):
    """PyTorch SDPA in fp64 with enable_gqa and an explicit bottom-right mask."""
    B, nq, Hq, d = q.shape
    outs = []
    for b in range(B):
        L = int(seqlens[b])
        qb = q[b].double().permute(1, 0, 2).unsqueeze(0)            # [1, Hq, nq, d]
        kb = k[b, :L].double().permute(1, 0, 2).unsqueeze(0)        # [1, Hkv, L, d]
        vb = v[b, :L].double().permute(1, 0, 2).unsqueeze(0)
        mask = None
        if causal:
            j = torch.arange(L).view(1, L)
            t = torch.arange(nq).view(nq, 1)
            mask = (j <= (L - nq + t)).view(1, 1, nq, L)
        ob = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, enable_gqa=True)
        outs.append(ob[0].permute(1, 0, 2))                          # [nq, Hq, d]
    return torch.stack(outs).numpy()


def pin_sdpa(orc, causal=False, shape=(2, 1, 8, 2, 16, 37), seqlens=None, seed=12):
    B, nq, Hq, Hkv, d, S_max = shape
    gen = torch.Generator().manual_seed(seed)
    q = _rand_bf16(gen, B, nq, Hq, d)
    k = _rand_bf16(gen, B, S_max, Hkv, d)
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    if seqlens is None:
        seqlens = [S_max - 3 * b for b in range(B)]
    out, _ = orc.decode(q, k, v, seqlens, causal=causal, nthreads=4)
    ref = _sdpa_reference(q, k, v, seqlens, causal)
    err = float(np.abs(out - ref).max())
    assert err < 1e-10, f"oracle vs SDPA fp64: max abs err {err}"


def pin_fp16_widening(orc):
    """Every one of the 65536 fp16 bit patterns widens to numpy's float16 value
    (an independent IEEE binary16 implementation); NaN patterns stay NaN."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.elem(int(x), True) for x in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_sdpa_fp16(orc):
    """fp16 inputs against SDPA in fp64 on the same fp16 values."""
    gen = torch.Generator().manual_seed(21)
    B, nq, Hq, Hkv, d, S_max = 2, 2, 8, 2, 16, 31
    q = torch.randn(B, nq, Hq, d, generator=gen).to(torch.float16)
    k = (torch.randn(B, S_max, Hkv, d, generator=gen) * 3).to(torch.float16)
    v = torch.randn(B, S_max, Hkv, d, generator=gen).to(torch.float16)
    seqlens = [31, 20]
    out, _ = orc.decode(q, k, v, seqlens, causal=True, nthreads=4)
    ref = _sdpa_reference(q, k, v, seqlens, True)
    err = float(np.abs(out - ref).max())
    assert err < 1e-10, f"fp16 oracle vs SDPA fp64: max abs err {err}"


def pin_sdpa_all(orc):
    pin_sdpa(orc, causal=False)
    pin_sdpa(orc, causal=True, shape=(3, 4, 8, 2, 16, 29), seqlens=[29, 17, 4])
    # The correctness recipe of "Flash Attention 4 - warp-role choreography and
    # the edges" (section "Does it actually compute attention?"): B=1, S=1024,
    # Hq=32, Hkv=8, D=128 against SDPA with GQA enabled.
    pin_sdpa(orc, causal=False, shape=(1, 1, 32, 8, 128, 1024), seqlens=[1024], seed=13)


# ---------------------------------------------------------------- closed forms
def pin_identical_keys(orc):
    """All keys equal: softmax is uniform, O = mean of V over the visible keys,
    lse = s + ln|J|."""
    gen = torch.Generator().manual_seed(14)
    B, nq, Hq, Hkv, d, S_max = 2, 1, 4, 2, 8, 12
    q = _rand_bf16(gen, B, nq, Hq, d)
    k0 = _rand_bf16(gen, 1, 1, Hkv, d)
    k = k0.expand(B, S_max, Hkv, d).contiguous()
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    seqlens = [12, 7]
    out, lse = orc.decode(q, k, v, seqlens)
    for b, L in enumerate(seqlens):
        for hq in range(Hq):
            h = hq // (Hq // Hkv)
            mean = v[b, :L, h].double().mean(0).numpy()
            assert np.allclose(out[b, 0, hq], mean, atol=1e-12, rtol=0)
            s = float((q[b, 0, hq].double() * k0[0, 0, h].double()).sum()) / math.sqrt(d)
            assert abs(lse[b, 0, hq] - (s + math.log(L))) < 1e-12


def pin_causal_counts(orc):
    """Zero keys with the causal mask: token t of nq new tokens sees exactly
    L - nq + t + 1 keys (bottom-right alignment), so lse_t = ln(L - nq + t + 1)
    and O_t is the mean of V over that prefix."""
    gen = torch.Generator().manual_seed(15)
    B, nq, Hq, Hkv, d, S_max = 2, 4, 4, 2, 8, 10
    q = _rand_bf16(gen, B, nq, Hq, d)
    k = torch.zeros(B, S_max, Hkv, d, dtype=torch.bfloat16)
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    seqlens = [10, 6]
    out, lse = orc.decode(q, k, v, seqlens, causal=True)
    for b, L in enumerate(seqlens):
        for t in range(nq):
            n = L - nq + t + 1
            for hq in range(Hq):
                h = hq // (Hq // Hkv)
                assert abs(lse[b, t, hq] - math.log(n)) < 1e-12, (b, t, hq, lse[b, t, hq], n)
                assert np.allclose(out[b, t, hq], v[b, :n, h].double().mean(0).numpy(), atol=1e-12, rtol=0)


def pin_dominant_score(orc):
    """One key equal to 50 q dominates: O = V of that key to 1e-12.  Its score
    is hundreds, so an oracle that does not subtract the max overflows."""
    gen = torch.Generator().manual_seed(16)
    B, nq, Hq, Hkv, d, S_max = 1, 1, 2, 1, 64, 9
    q = _int_bf16(gen, -2, 2, B, nq, Hq, d)
    q[0, 0, 1] = q[0, 0, 0]
    k = _int_bf16(gen, -1, 1, B, S_max, Hkv, d)
    jstar = 5
    k[0, jstar, 0] = (q[0, 0, 0].float() * 50).to(torch.bfloat16)
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    out, lse = orc.decode(q, k, v, [S_max])
    for hq in range(Hq):
        assert np.allclose(out[0, 0, hq], v[0, jstar, 0].double().numpy(), atol=1e-12, rtol=0)
        s = float((q[0, 0, hq].double() * k[0, jstar, 0].double()).sum()) / math.sqrt(d)
        assert s > 100.0 and abs(lse[0, 0, hq] - s) < 1e-9


def pin_single_and_empty(orc):
    """L = 1 gives O = V_0 and lse = s_0; L = 0 gives O = 0 and lse = -inf.
    The cache is longer than L so that reading past L would be visible."""
    gen = torch.Generator().manual_seed(17)
    B, nq, Hq, Hkv, d, S_max = 2, 1, 2, 1, 8, 4
    q = _rand_bf16(gen, B, nq, Hq, d)
    k = _rand_bf16(gen, B, S_max, Hkv, d)
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    out, lse = orc.decode(q, k, v, [1, 0])
    for hq in range(Hq):
        assert np.allclose(out[0, 0, hq], v[0, 0, 0].double().numpy(), atol=1e-15, rtol=0)
        s0 = float((q[0, 0, hq].double() * k[0, 0, 0].double()).sum()) / math.sqrt(d)
        assert abs(lse[0, 0, hq] - s0) < 1e-12
        assert np.all(out[1, 0, hq] == 0.0) and lse[1, 0, hq] == -math.inf


def pin_rows_sum_to_one(orc):
    """exp(s_j - lse) summed over the visible keys is 1 for every row."""
    gen = torch.Generator().manual_seed(18)
    B, nq, Hq, Hkv, d, S_max = 2, 2, 4, 2, 16, 33
    q = _rand_bf16(gen, B, nq, Hq, d, scale=2.0)
    k = _rand_bf16(gen, B, S_max, Hkv, d)
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    seqlens = [33, 20]
    for causal in (False, True):
        _, lse = orc.decode(q, k, v, seqlens, causal=causal)
        for b, L in enumerate(seqlens):
            for t in range(nq):
                hi = L - nq + t + 1 if causal else L
                for hq in range(Hq):
                    h = hq // (Hq // Hkv)
                    s = (k[b, :hi, h].double() @ q[b, t, hq].double()).numpy() / math.sqrt(d)
                    assert abs(np.exp(s - lse[b, t, hq]).sum() - 1.0) < 1e-12


def pin_shift_and_scale_invariance(orc):
    """With q = e_0, adding c to key component 0 shifts every score by
    scale*c: O is unchanged and lse moves by exactly scale*c.  V + 1 moves O
    by 1; 2V doubles O.  Integer inputs keep every shifted copy exact."""
    gen = torch.Generator().manual_seed(19)
    B, nq, Hq, Hkv, d, S_max = 1, 1, 2, 1, 16, 21
    q = torch.zeros(B, nq, Hq, d, dtype=torch.bfloat16)
    q[..., 0] = 1.0
    k = _int_bf16(gen, -4, 4, B, S_max, Hkv, d)
    v = _int_bf16(gen, -4, 4, B, S_max, Hkv, d)
    out, lse = orc.decode(q, k, v, [S_max])
    k2 = k.clone()
    k2[..., 0] = k2[..., 0] + 8
    out2, lse2 = orc.decode(q, k2, v, [S_max])
    assert np.allclose(out2, out, atol=1e-12, rtol=0)
    assert np.allclose(lse2 - lse, 8.0 / math.sqrt(d), atol=1e-12, rtol=0)
    out3, lse3 = orc.decode(q, k, (v.float() + 1).to(torch.bfloat16), [S_max])
    assert np.allclose(out3, out + 1.0, atol=1e-12, rtol=0) and np.allclose(lse3, lse, atol=0, rtol=0)
    out4, _ = orc.decode(q, k, (v.float() * 2).to(torch.bfloat16), [S_max])
    assert np.allclose(out4, 2.0 * out, atol=1e-12, rtol=0)


# ------------------------------------------------------------- GQA golden
def pin_head_map_golden(orc):
    """The pages' worked GQA examples (tests/golden/gqa_head_groups.json):
    with 32 query heads on 8 KV heads, query head hq reads KV head hq // 4.
    Each KV head gets a constant V, so O of query head hq equals its KV head's
    constant."""
    with open(os.path.join(GOLDEN, "gqa_head_groups.json")) as f:
        gold = json.load(f)
    for ex in gold["examples"]:
        Hq, Hkv = ex["num_qo_heads"], ex["num_kv_heads"]
        assert Hq // Hkv == ex["gqa_ratio"]
        gen = torch.Generator().manual_seed(20)
        d, S_max = 8, 5
        q = _rand_bf16(gen, 1, 1, Hq, d)
        k = _rand_bf16(gen, 1, S_max, Hkv, d)
        v = torch.arange(1, Hkv + 1, dtype=torch.float32).view(1, 1, Hkv, 1).expand(1, S_max, Hkv, d)
        v = v.contiguous().to(torch.bfloat16)
        out, _ = orc.decode(q, k, v, [S_max])
        got = [int(round(float(out[0, 0, hq, 0]))) - 1 for hq in range(Hq)]
        assert got == ex["kv_head_of_q_head"], (ex, got)


# ------------------------------------------------------------ split + combine
def pin_split_then_combine(orc):
    """Splitting the keys into contiguous ranges, attending within each and
    merging the partials reproduces the unsplit result (1e-12), including
    empty splits and an empty sequence."""
    gen = torch.Generator().manual_seed(21)
    B, nq, Hq, Hkv, d, S_max = 4, 2, 4, 2, 16, 45
    q = _rand_bf16(gen, B, nq, Hq, d, scale=2.0)
    k = _rand_bf16(gen, B, S_max, Hkv, d)
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    seqlens = [45, 17, 3, 0]
    for causal in (False, True):
        full, full_lse = orc.decode(q, k, v, seqlens, causal=causal)
        for S in (1, 2, 3, 4, 8):
            begin, end = oracle_mod.split_ranges(seqlens, S, block=4)
            parts = [orc.decode(q, k, v, seqlens, causal=causal, pos_begin=begin[s], pos_end=end[s])
                     for s in range(S)]
            o_part = np.stack([p[0] for p in parts])
            l_part = np.stack([p[1] for p in parts])
            assert np.isneginf(l_part).any() or S == 1
            out, lse = orc.combine(o_part, l_part)
            assert np.allclose(out, full, atol=1e-12, rtol=0), (causal, S)
            fin = np.isfinite(full_lse)
            assert np.array_equal(fin, np.isfinite(lse))
            assert np.allclose(lse[fin], full_lse[fin], atol=1e-12, rtol=0)


# Key ranges of the documented split partition, worked out by hand from its
# definition (the one gqa_decode_splitkv states): sequence b of length L has
# nblk = ceil(L / block) blocks and splits = clamp(ceil(nblk / min_blocks), 1, S)
# splits; split s < splits covers blocks [floor(s*nblk/splits),
# floor((s+1)*nblk/splits)), i.e. positions [128*lo, min(128*hi, L)), and the
# splits past `splits` are empty ([0, 0)).  Entries: (L, S, min_blocks, block)
# -> [(begin, end) of split 0, 1, ..., S-1].
SPLIT_TABLE = [
    ((0, 1, 1, 128), [(0, 0)]),
    ((0, 3, 1, 128), [(0, 0), (0, 0), (0, 0)]),
    ((1, 1, 1, 128), [(0, 1)]),
    ((1, 3, 1, 128), [(0, 1), (0, 0), (0, 0)]),
    ((128, 3, 1, 128), [(0, 128), (0, 0), (0, 0)]),
    ((129, 1, 1, 128), [(0, 129)]),
    ((129, 3, 1, 128), [(0, 128), (128, 129), (0, 0)]),
    ((129, 8, 1, 128), [(0, 128), (128, 129)] + [(0, 0)] * 6),
    ((1000, 1, 1, 128), [(0, 1000)]),
    # nblk = 8 over 3 splits: floor(8/3) = 2, floor(16/3) = 5
    ((1000, 3, 1, 128), [(0, 256), (256, 640), (640, 1000)]),
    ((1000, 8, 1, 128), [(128 * s, 128 * (s + 1)) for s in range(7)] + [(896, 1000)]),
    # at least 3 blocks a split: ceil(8/3) = 3 splits even when 8 are allowed
    ((1000, 8, 3, 128), [(0, 256), (256, 640), (640, 1000)] + [(0, 0)] * 5),
    ((129, 8, 3, 128), [(0, 129)] + [(0, 0)] * 7),
    # 4-position blocks: L = 10 has 3 blocks, floor(3/2) = 1
    ((10, 2, 1, 4), [(0, 4), (4, 10)]),
    ((10, 5, 1, 4), [(0, 4), (4, 8), (8, 10), (0, 0), (0, 0)]),
]


def pin_split_ranges(orc, split_ranges=None):
    """The oracle's split partition (oracle.split_ranges) against the table
    above, worked by hand from the partition's definition, one sequence at a
    time and all of them in one batch; plus the properties any reading of it
    must have: the non-empty ranges are contiguous, block-aligned, cover
    [0, L) exactly and number min(S, ceil(nblk / min_blocks)) (at least 1)."""
    fn = oracle_mod.split_ranges if split_ranges is None else split_ranges
    for (L, S, mb, blk), want in SPLIT_TABLE:
        begin, end = fn([L], S, block=blk, min_blocks=mb)
        got = [(int(begin[s, 0]), int(end[s, 0])) for s in range(S)]
        assert got == want, ((L, S, mb, blk), got, want)
    # a batch gives each sequence its own partition
    for S, mb, blk in ((3, 1, 128), (8, 1, 128), (8, 3, 128)):
        rows = [(key, want) for key, want in SPLIT_TABLE if key[1:] == (S, mb, blk)]
        lens = [key[0] for key, _ in rows]
        begin, end = fn(lens, S, block=blk, min_blocks=mb)
        for i, (_, want) in enumerate(rows):
            assert [(int(begin[s, i]), int(end[s, i])) for s in range(S)] == want
    # properties on a sweep
    for L in list(range(0, 600, 7)) + [1023, 1024, 1025, 131072]:
        for S in (1, 2, 3, 4, 5, 8, 16, 64):
            nblk = -(-L // 128)
            begin, end = fn([L], S)
            ranges = [(int(begin[s, 0]), int(end[s, 0])) for s in range(S)]
            n_live = min(S, max(nblk, 1))
            live, dead = ranges[:n_live], ranges[n_live:]
            assert all(r == (0, 0) for r in dead), (L, S, ranges)
            assert live[0][0] == 0 and live[-1][1] == L, (L, S, ranges)
            for (b0, e0), (b1, _) in zip(live, live[1:]):
                assert e0 == b1 and b1 % 128 == 0, (L, S, ranges)
            sizes = [-(-(e - b) // 128) for b, e in live]
            if L > 0:
                assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1, (L, S, ranges)


def pin_lse_logsumexp(orc):
    """The LSE at moderate sizes (several hundred keys, ragged and empty rows,
    both mask modes) against scipy's logsumexp of fp64 scores from a numpy
    matmul: ln sum_j exp(scale * q . k_j) over the visible keys, -inf when
    there are none."""
    from scipy.special import logsumexp

    gen = torch.Generator().manual_seed(23)
    B, nq, Hq, Hkv, d, S_max = 4, 3, 8, 2, 32, 300
    G = Hq // Hkv
    q = _rand_bf16(gen, B, nq, Hq, d, scale=2.0)
    k = _rand_bf16(gen, B, S_max, Hkv, d)
    v = _rand_bf16(gen, B, S_max, Hkv, d)
    seqlens = [300, 1, 0, 177]
    scale = 1.0 / math.sqrt(d)
    qn, kn = q.double().numpy(), k.double().numpy()
    for causal in (False, True):
        _, lse = orc.decode(q, k, v, seqlens, causal=causal, nthreads=4)
        for b, L in enumerate(seqlens):
            for t in range(nq):
                vis = L if not causal else max(0, min(L, L - nq + t + 1))
                for hq in range(Hq):
                    if vis == 0:
                        assert np.isneginf(lse[b, t, hq]), (b, t, hq, causal)
                        continue
                    sc = scale * (kn[b, :vis, hq // G, :] @ qn[b, t, hq, :])
                    ref = float(logsumexp(sc))
                    assert abs(lse[b, t, hq] - ref) < 1e-12, (b, t, hq, causal, lse[b, t, hq], ref)


def pin_combine_closed_forms(orc):
    gen = np.random.default_rng(22)
    d, rows = 8, 3
    o1 = gen.standard_normal((rows, d))
    o2 = gen.standard_normal((rows, d))
    a = gen.standard_normal(rows)
    # equal weights: the average, lse + ln 2
    out, lse = orc.combine(np.stack([o1, o2]), np.stack([a, a]))
    assert np.allclose(out, (o1 + o2) / 2, atol=1e-14) and np.allclose(lse, a + math.log(2), atol=1e-14)
    # weights 1 : 3
    out, lse = orc.combine(np.stack([o1, o2]), np.stack([a, a + math.log(3)]))
    assert np.allclose(out, (o1 + 3 * o2) / 4, atol=1e-14) and np.allclose(lse, a + math.log(4), atol=1e-14)
    # an empty split is skipped
    out, lse = orc.combine(np.stack([o1, np.full_like(o2, np.nan)]), np.stack([a, np.full(rows, -np.inf)]))
    assert np.allclose(out, o1, atol=1e-15) and np.allclose(lse, a, atol=1e-15)
    # every split empty: zero output, -inf lse
    out, lse = orc.combine(np.stack([o1, o2]), np.full((2, rows), -np.inf))
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


ALL_PINS = [
    pin_bruteforce_tiny,
    pin_sdpa_all,
    pin_fp16_widening,
    pin_sdpa_fp16,
    pin_identical_keys,
    pin_causal_counts,
    pin_dominant_score,
    pin_single_and_empty,
    pin_rows_sum_to_one,
    pin_shift_and_scale_invariance,
    pin_head_map_golden,
    pin_split_then_combine,
    pin_split_ranges,
    pin_lse_logsumexp,
    pin_combine_closed_forms,
]

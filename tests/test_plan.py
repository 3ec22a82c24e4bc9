"""Host-side planning: the work decomposition the decode kernel walks
(plan.cuh, enumerated through gqa_decode_plan) covers every KV block of every
(batch, KV head) pair exactly once, with consistent partial slots and piece
counts (CPU only)."""
import collections

import numpy as np
import pytest

import gqa_decode_blackwell_gb300 as g
import oracle
from gqa_decode_blackwell_gb300 import build as gbuild


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()


def _desc(B, Hkv, s_max, G=4, nq=1, d=128, reduction=g.GQA_REDUCE_COMBINE):
    """The kernel-reduction plans by default (the in-cluster merge has tests of its own below)."""
    return g.gqa_desc_t(B, nq, Hkv * G, Hkv, d, s_max, 0.0, 0, 0, 0, reduction)


def _blocks(L):
    return (max(L, 0) + 127) // 128


def _units(nblk, X):
    return nblk + X if nblk > 0 else 0


# Grid and item units X of the balanced plan: with k >= 2 SMs per (batch, KV
# head) pair and at most 32 blocks per CTA (cache capacity <= 32 k blocks),
# k CTAs per pair and X = 0; otherwise every SM, and X = 1 for the 16-column
# kernels (nq * G <= 16), 3 for the 32-column ones.
def _grid_and_item_units(pairs, sm, G, nq, s_max):
    k = sm // pairs if pairs > 0 else 0
    if k >= 2 and _blocks(s_max) <= 32 * k:
        return k * pairs, 0
    return sm, (1 if nq * G <= 16 else 3)


def check_balanced(seqlens, Hkv, s_max, sm, G=4, nq=1):
    """Balanced plan: every pair costs its blocks plus X item units; the
    units, in pair order (batch-major), are cut into C contiguous ranges."""
    grid, X = _grid_and_item_units(len(seqlens) * Hkv, sm, G, nq, s_max)
    desc = _desc(len(seqlens), Hkv, s_max, G=G, nq=nq)
    C, mode, slots, items = g.gqa_decode_plan(desc, seqlens, 0, sm)
    assert mode == 1
    lens = [min(max(int(L), 0), s_max) for L in seqlens]
    U = sum(_units(_blocks(L), X) for L in lens) * Hkv
    assert C == max(1, min(grid, len(lens) * Hkv * _units(_blocks(s_max), X)))
    C_eff = max(1, min(C, U))

    def cta_of(u):  # the largest c with floor(c * U / C_eff) <= u
        return ((u + 1) * C_eff - 1) // U
    # unit order: pair (b, h) starts at v_first, its X item units come first
    v_first, v = {}, 0
    for b, L in enumerate(lens):
        for h in range(Hkv):
            v_first[(b, h)] = v
            v += _units(_blocks(L), X)
    assert v == U
    vload = collections.Counter(cta_of(u) for u in range(U))
    cover = collections.Counter()
    per_pair = collections.defaultdict(list)
    per_cta = collections.Counter()
    for c, b, h, b0, b1, slot, first, npieces in items:
        per_pair[(b, h)].append((c, b0, b1, slot, first, npieces))
        per_cta[c] += b1 - b0
        for blk in range(b0, b1):
            cover[(b, h, blk)] += 1
            assert cta_of(v_first[(b, h)] + X + blk) == c
    # every unit exactly once
    expect = {(b, h, k) for b, L in enumerate(lens) for h in range(Hkv) for k in range(_blocks(L))}
    assert set(cover) == expect and all(v == 1 for v in cover.values())
    # every pair visited, pieces consistent
    for b, L in enumerate(lens):
        for h in range(Hkv):
            pieces = per_pair[(b, h)]
            assert len(pieces) >= 1
            n = len(pieces)
            assert all(p[5] == n for p in pieces)
            assert sum(p[4] for p in pieces) == 1
            if n == 1:
                assert pieces[0][3] == -1
            else:
                assert sorted(p[3] for p in pieces) == list(range(n))
                assert n <= slots
            # pieces are contiguous and in CTA order
            ordered = sorted(pieces)
            assert ordered[0][1] == 0 and ordered[-1][2] == _blocks(L)
            for a, z in zip(ordered, ordered[1:]):
                assert a[2] == z[1]
    # only the first C_eff CTAs work; their loads in units differ by at most one
    assert all(c < C_eff for c in per_cta)
    if U > 0:
        loads = [vload.get(c, 0) for c in range(C_eff)]
        assert max(loads) - min(loads) <= 1
        assert sum(per_cta.values()) == U - X * Hkv * sum(1 for L in lens if L > 0)


@pytest.mark.parametrize("G,nq", [(4, 1), (8, 4)])
@pytest.mark.parametrize("seed", range(24))
def test_balanced_plan_random(seed, G, nq):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    Hkv = int(rng.choice([1, 2, 8]))
    s_max = int(rng.integers(1, 5000))
    lens = rng.integers(-5, s_max + 1, size=B)
    lens[rng.random(B) < 0.2] = 0
    sm = int(rng.choice([1, 3, 16, 152]))
    check_balanced(lens.tolist(), Hkv, s_max, sm, G, nq)
    # the same lengths in a much larger cache: fewer units than CTAs
    check_balanced(lens.tolist(), Hkv, s_max * 7, 152, G, nq)


@pytest.mark.parametrize("lens,Hkv,s_max,sm,G,nq", [
    ([0, 0, 0], 2, 128, 152, 4, 1),         # nothing to read: every pair is an empty item
    ([200], 2, 4200, 152, 4, 1),            # fewer units than CTAs, pairs cut in two
    ([129], 1, 4200, 152, 4, 1),
    ([1, 127, 128, 129, 4097, 0, 1], 2, 4200, 152, 4, 1),
    ([5000, 0, 3], 1, 5000, 16, 4, 1),
    ([1], 1, 1, 152, 4, 1),                 # one unit, one CTA
    ([512], 1, 512, 152, 4, 1),             # tiny config: 4 units
    ([4096] * 8, 8, 4096, 152, 4, 1),       # Llama-8B-shaped
    ([8192] * 16, 8, 8192, 152, 8, 1),      # 70B-shaped
    ([2048] * 32, 2, 2048, 152, 8, 4),      # speculative: 32 columns
    ([131072, 1024, 70000, 0], 8, 131072, 152, 4, 1),
    ([0, 300, 0, 0, 129, 0], 3, 300, 5, 4, 1),
])
def test_balanced_plan_cases(lens, Hkv, s_max, sm, G, nq):
    check_balanced(lens, Hkv, s_max, sm, G, nq)


@pytest.mark.parametrize("B,Hkv,L,G,nq,ctas,pieces", [
    (8, 8, 4096, 4, 1, 128, 2),     # Llama-8B-shaped: 64 pairs, two CTAs each
    (32, 2, 2048, 8, 4, 128, 2),    # speculative
    (4, 8, 8192, 8, 1, 128, 4),     # 32 pairs, four CTAs each
    (16, 8, 8192, 8, 1, 152, None), # 128 pairs on 152 SMs: every SM
    (4, 8, 131072, 8, 1, 152, None),  # long sequences: every SM
])
def test_balanced_plan_equal_lengths_one_item_per_cta(B, Hkv, L, G, nq, ctas, pieces):
    """Equal lengths with two or more SMs per pair: every CTA gets one item of
    the same size, every pair the same number of pieces."""
    C, mode, slots, items = g.gqa_decode_plan(_desc(B, Hkv, L, G=G, nq=nq), [L] * B, 0, 152)
    assert mode == 1 and C == ctas
    if pieces is not None:
        per_cta = collections.Counter(int(r[0]) for r in items)
        assert len(per_cta) == ctas and set(per_cta.values()) == {1}
        assert {int(r[4]) - int(r[3]) for r in items} == {(L // 128) // pieces}
        assert {int(r[7]) for r in items} == {pieces}
    check_balanced([L] * B, Hkv, L, 152, G, nq)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 8, 64])
def test_split_plan_matches_documented_partition(S):
    rng = np.random.default_rng(S)
    B, Hkv, s_max = 6, 2, 1000
    lens = rng.integers(0, s_max + 1, size=B).tolist()
    lens[0] = 1
    desc = _desc(B, Hkv, s_max)
    C, mode, slots, items = g.gqa_decode_plan(desc, lens, S, 152)
    assert mode == 0 and C == min(152, B * Hkv * S)
    begin, end = oracle.split_ranges(lens, S, block=128)
    seen = set()
    for c, b, h, b0, b1, slot, first, npieces in items:
        w = (b * Hkv + h) * S + (slot if slot >= 0 else 0)
        assert w % C == c
        s = slot if slot >= 0 else 0
        assert (S == 1) == (slot == -1)
        assert min(b0 * 128, lens[b]) == begin[s, b] or b0 == b1
        assert min(b1 * 128, lens[b]) == end[s, b]
        seen.add((b, h, s))
    assert len(seen) == B * Hkv * S


def test_auto_falls_back_to_splits_for_huge_batches():
    lens = [300] * 1500
    C, mode, slots, items = g.gqa_decode_plan(_desc(1500, 1, 300), lens, 0, 152)
    assert mode == 0


def test_balanced_plan_can_exceed_64_pieces_per_pair():
    """A long sequence on few KV heads is cut over (nearly) every CTA: far
    more than 64 pieces for one pair, which the combine must merge beyond its
    64-slot fast path."""
    C, mode, slots, items = g.gqa_decode_plan(_desc(1, 1, 32768), [32768], 0, 152)
    assert mode == 1 and slots == 152
    assert 140 <= max(int(r[7]) for r in items) <= 152
    check_balanced([32768], 1, 32768, 152)


def test_balanced_plan_needs_int32_prefix_sums():
    """512 sequences of up to 2^30 positions would overflow the balanced
    plan's int32 prefix sums of units: the fixed-splits plan takes over."""
    C, mode, slots, items = g.gqa_decode_plan(_desc(512, 1, 1 << 30), [1] * 512, 0, 152, max_items=0)
    assert mode == 0
    C, mode, slots, items = g.gqa_decode_plan(_desc(512, 1, 1 << 20), [1] * 512, 0, 152, max_items=0)
    assert mode == 1


# ------------------------------------------------------- in-cluster merge
def _cluster_k_auto(pairs, sm, s_max):
    """The automatic choice: k = the largest power of two <= min(8, sm // pairs,
    blocks), taken when k >= 2, the cache spans at most 32 k blocks, the k *
    pairs CTAs are at least 64, each streams at most 3 blocks more than a CTA
    of the balanced plan (sm // pairs per pair, at most one per block), and
    k <= 4 or k * pairs <= 64; else 0 (the combine kernel)."""
    per_pair = sm // pairs
    lim = min(per_pair, _blocks(s_max))
    k = 1
    while 2 * k <= lim and k < 8:
        k *= 2
    nb = _blocks(s_max)
    bal = min(per_pair * pairs, pairs * nb)
    extra = -(-nb // k) - (-(-pairs * nb // bal))
    if k >= 2 and nb <= 32 * k and extra <= 3 and (k <= 4 or pairs * k <= 64) and k * pairs >= 64:
        return k
    return 0


def check_cluster(lens, Hkv, s_max, sm, k, G=4, nq=1, num_splits=0, reduction=g.GQA_REDUCE_AUTO):
    """Cluster plan: k fixed splits per pair; CTA q*k + j holds piece j of the
    pairs q, q + Q, ... of cluster q (Q = grid / k clusters), with the
    documented partition of each sequence into min(k, blocks) splits."""
    desc = _desc(len(lens), Hkv, s_max, G=G, nq=nq, reduction=reduction)
    C, mode, slots, items = g.gqa_decode_plan(desc, lens, num_splits, sm)
    pairs = len(lens) * Hkv
    assert mode == 2 and slots == 0
    Q = max(1, min(pairs, sm // k))
    assert C == Q * k
    begin, end = oracle.split_ranges(lens, k, block=128)
    seen = collections.Counter()
    for c, b, h, b0, b1, slot, first, npieces in items:
        q, j = divmod(int(c), k)
        pair = b * Hkv + h
        assert pair % Q == q and slot == j
        L = min(max(lens[b], 0), s_max)
        if b0 < b1:
            assert (b0 * 128, min(b1 * 128, L)) == (begin[j, b], end[j, b])
        else:
            assert begin[j, b] == end[j, b] == 0 or L == 0
        seen[(b, h, j)] += 1
    assert set(seen) == {(b, h, j) for b in range(len(lens)) for h in range(Hkv) for j in range(k)}
    assert set(seen.values()) == {1}
    # The merge exchanges item by item: the k CTAs of a cluster must take the
    # same pairs in the same order (items are listed in processing order).
    order = collections.defaultdict(list)
    for c, b, h, *_ in items:
        order[int(c)].append((int(b), int(h)))
    for q in range(Q):
        assert all(order[q * k + j] == order[q * k] for j in range(1, k))


@pytest.mark.parametrize("B,Hkv,L,G,nq,k", [
    (8, 8, 4096, 4, 1, 2),      # Llama-8B-shaped: 64 pairs, clusters of two
    (32, 2, 2048, 8, 4, 2),     # speculative
    (8, 1, 1024, 4, 1, 8),      # 8 pairs x 8 <= 64 CTAs, 8 blocks each
    (1, 8, 4096, 4, 1, 8),      # 8 pairs x 8 = 64 CTAs
    (4, 8, 8192, 8, 1, 4),      # 32 pairs, 64 blocks <= 32 x 4
])
def test_auto_selects_cluster_merge_for_short_sequences(B, Hkv, L, G, nq, k):
    assert _cluster_k_auto(B * Hkv, 152, L) == k
    check_cluster([L] * B, Hkv, L, 152, k, G, nq)


@pytest.mark.parametrize("B,Hkv,L,G,nq,mode", [
    (16, 8, 8192, 8, 1, 1),     # 70B-shaped: one SM per pair, balanced plan + combine
    (4, 8, 131072, 8, 1, 1),    # ragged long context: 1024 blocks > 32 x 4
    (1, 1, 65536, 4, 1, 1),     # one long sequence
    (1, 1, 32768, 4, 1, 1),     # one pair: 8 CTAs would be far fewer than the balanced plan's 152
    (1, 2, 4096, 4, 1, 1),      # 2 pairs: 16 CTAs against 64
    (1, 1, 512, 8, 1, 1),       # tiny: a cluster of 4 CTAs is below 64
])
def test_auto_keeps_combine_for_long_sequences_or_many_pairs(B, Hkv, L, G, nq, mode):
    assert _cluster_k_auto(B * Hkv, 152, L) == 0
    C, m, slots, items = g.gqa_decode_plan(_desc(B, Hkv, L, G=G, nq=nq, reduction=g.GQA_REDUCE_AUTO), [L] * B, 0,
                                          152)
    assert m == mode and slots > 0


@pytest.mark.parametrize("S,pairs,expect", [
    (2, 64, 2), (2, 400, 2), (2, 63, 0), (2, 1, 0), (4, 64, 0), (4, 400, 0), (8, 8, 0), (8, 128, 0), (3, 4, 0),
    (16, 2, 0), (1, 4, 0),
])
def test_explicit_split_counts_follow_the_measured_selection(S, pairs, expect):
    """An explicit split count merges in the cluster for 2 splits on at least
    128 CTAs (where it measured faster); other counts use the combine kernel."""
    lens = [2000] * pairs
    C, mode, slots, items = g.gqa_decode_plan(_desc(pairs, 1, 2000, reduction=g.GQA_REDUCE_AUTO), lens, S, 152)
    if expect:
        assert mode == 2 and slots == 0
        check_cluster(lens, 1, 2000, 152, expect, num_splits=S)
    else:
        assert mode == 0


@pytest.mark.parametrize("S", [2, 4, 8])
def test_forced_cluster_merge_with_ragged_lengths(S):
    rng = np.random.default_rng(S)
    lens = rng.integers(0, 3000, size=23).tolist()
    lens[:3] = [0, 1, 129]          # empty, one block, fewer blocks than splits
    check_cluster(lens, 3, 3000, 152, S, num_splits=S, reduction=g.GQA_REDUCE_CLUSTER)


def test_forced_cluster_merge_many_pairs_is_persistent():
    """128 pairs x 8 pieces on 152 SMs: 19 clusters of eight, each walking
    its pairs one after another."""
    check_cluster([8192] * 16, 8, 8192, 152, 8, G=8, num_splits=8, reduction=g.GQA_REDUCE_CLUSTER)


def test_forced_cluster_merge_automatic_split_count():
    # ragged-like: 32 pairs on 152 SMs -> 4 CTAs per pair
    check_cluster([131072, 1024, 70000, 5], 8, 131072, 152, 4, reduction=g.GQA_REDUCE_CLUSTER)
    # more pairs than SMs: one CTA per pair, nothing to merge
    C, mode, slots, items = g.gqa_decode_plan(_desc(200, 1, 300, reduction=g.GQA_REDUCE_CLUSTER), [300] * 200, 0, 152)
    assert mode == 0 and slots == 0 and C == 152 and all(int(r[5]) == -1 for r in items)


@pytest.mark.parametrize("S", [3, 5, 16, 64])
def test_forced_cluster_merge_rejects_other_split_counts(S):
    L = g.lib()
    import ctypes
    desc = _desc(2, 2, 1000, reduction=g.GQA_REDUCE_CLUSTER)
    nc, mode, slots, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    sl = np.array([1000, 1000], dtype=np.int32)
    rc = L.gqa_decode_plan(ctypes.byref(desc), sl.ctypes.data, S, 152, ctypes.byref(nc), ctypes.byref(mode),
                           ctypes.byref(slots), None, 0, ctypes.byref(n))
    assert rc == g.GQA_ERR_UNSUPPORTED


def test_unknown_reduction_mode_is_invalid():
    import ctypes
    desc = _desc(2, 2, 1000, reduction=7)
    nc, mode, slots, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    sl = np.array([1000, 1000], dtype=np.int32)
    rc = g.lib().gqa_decode_plan(ctypes.byref(desc), sl.ctypes.data, 0, 152, ctypes.byref(nc), ctypes.byref(mode),
                                 ctypes.byref(slots), None, 0, ctypes.byref(n))
    assert rc == g.GQA_ERR_INVALID_ARG

"""Host model of the decode kernel's mbarrier protocol.

The kernel's warps synchronise through mbarriers waited on by phase parity:
a wait for phase k returns once the barrier's completed-phase count c has a
parity different from k's.  That is only the intended answer when c is k or
k + 1 at the time of the wait; with c = k - 1 the wait passes a phase early,
with c = k + 2 it blocks on a phase that has already completed.

This module replays the protocol of one CTA (producer, score-MMA issuer,
value-MMA issuer, softmax warpgroup) under random interleavings: TMA loads land
in any order, the MMAs of one issuing thread complete in issue order, each
agent advances whenever its wait is satisfied.  A CTA's blocks belong to work
items (some empty); at the end of each item the softmax warpgroup hands a
staging buffer (two of them, OUT_FULL / OUT_EMPTY) to the value-MMA thread,
which writes the item out and releases the previous item's buffer.  Every wait is checked against
the rule above.  The K/V ring layout is a parameter so that the check also
shows why K and V need rings of their own: with one shared ring whose depth
is odd, a stage's previous tile can belong to the other issuer and still be
in flight when a wait starts.
"""
import random

import pytest


class Bar:
    def __init__(self):
        self.c = 0  # completed phases


class Violation(Exception):
    pass


def split_rings(ns):
    nsk, nsv = (ns + 1) // 2, ns // 2

    def k_slot(g, G):
        return g % nsk, g // nsk

    def v_slot(g, G):
        return nsk + g % nsv, g // nsv

    return k_slot, v_slot


def shared_ring(ns):
    # issue order K0 K1 V0 K2 V1 ...: K(g) is tile 2g-1 (g > 0), V(g) is tile
    # 2g+2, the last V is tile 2G-1
    def k_slot(g, G):
        t = 0 if g == 0 else 2 * g - 1
        return t % ns, t // ns

    def v_slot(g, G):
        t = 2 * g + 2 if g + 1 < G else 2 * g + 1
        return t % ns, t // ns

    return k_slot, v_slot


def run_cta(ns, G, layout, rng, tail_wait=True, items=None):
    """One CTA with G blocks in `items` (block counts, default one item);
    raises Violation on an unsound parity wait or a deadlock."""
    if items is None:
        items = [G]
    assert sum(items) == G
    k_slot, v_slot = layout(ns)
    out_full, out_empty = [Bar(), Bar()], [Bar(), Bar()]
    ring_full = [Bar() for _ in range(ns)]
    ring_empty = [Bar() for _ in range(ns)]
    s_full, s_empty = [Bar(), Bar()], [Bar(), Bar()]
    p_full, p_empty = [Bar(), Bar()], [Bar(), Bar()]
    landing = []                 # TMA loads in flight: barriers to complete
    mma_q = {"qk": [], "pv": []}  # commits of each issuer, completed in order
    # producer's issue counts per stage, to detect two loads in one stage
    in_flight = [0] * ns

    def wait(bar, k, what):
        """Generator step: yields until the hardware predicate holds."""
        while True:
            passes = (bar.c & 1) != (k & 1)
            if passes:
                if bar.c != k + 1:
                    raise Violation(f"{what}: wait for phase {k} passed at c={bar.c}")
                return
            if bar.c >= k + 2:
                raise Violation(f"{what}: wait for phase {k} blocks at c={bar.c}")
            yield

    def producer():
        order = []
        for g in range(G):
            order.append(("K", g))
            if g > 0:
                order.append(("V", g - 1))
        if G > 0:
            order.append(("V", G - 1))
        for kind, g in order:
            stage, ph = (k_slot if kind == "K" else v_slot)(g, G)
            # free once the previous tile of the stage was released
            if ph > 0:
                yield from wait(ring_empty[stage], ph - 1, f"producer {kind}{g}")
            if in_flight[stage]:
                raise Violation(f"producer {kind}{g}: stage {stage} still loading")
            in_flight[stage] += 1
            landing.append(stage)

    def qk():
        for g in range(G):
            sl = g & 1
            if g >= 2:
                yield from wait(s_empty[sl], (g >> 1) - 1, f"qk S_EMPTY {g}")
            stage, ph = k_slot(g, G)
            yield from wait(ring_full[stage], ph, f"qk RING_FULL K{g}")
            mma_q["qk"].append(s_full[sl])
            mma_q["qk"].append(ring_empty[stage])

    def pv():
        g = 0
        for k, nb in enumerate(items):
            for _ in range(nb):
                sl = g & 1
                yield from wait(p_full[sl], g >> 1, f"pv P_FULL {g}")
                stage, ph = v_slot(g, G)
                yield from wait(ring_full[stage], ph, f"pv RING_FULL V{g}")
                mma_q["pv"].append(p_empty[sl])
                mma_q["pv"].append(ring_empty[stage])
                g += 1
            # write item k out; item k-1's buffer has been read
            yield from wait(out_full[k & 1], k >> 1, f"pv OUT_FULL item {k}")
            if k >= 1:
                out_empty[(k - 1) & 1].c += 1

    def softmax():
        g = 0
        for k, nb in enumerate(items):
            for _ in range(nb):
                sl = g & 1
                yield from wait(s_full[sl], g >> 1, f"softmax S_FULL {g}")
                s_empty[sl].c += 1
                if g >= 2:
                    yield from wait(p_empty[sl], (g >> 1) - 1, f"softmax P_EMPTY {g}")
                if tail_wait:  # zeroing the rows of V past the sequence end
                    stage, ph = v_slot(g, G)
                    yield from wait(ring_full[stage], ph, f"softmax tail V{g}")
                p_full[sl].c += 1
                g += 1
            if nb > 0:  # epilogue: the item's last value MMA has completed
                gl = g - 1
                yield from wait(p_empty[gl & 1], gl >> 1, f"softmax epilogue P_EMPTY {gl}")
            if k >= 2:  # staging buffer of item k-2 released
                yield from wait(out_empty[k & 1], (k >> 1) - 1, f"softmax OUT_EMPTY item {k}")
            out_full[k & 1].c += 1

    agents = {"producer": producer(), "qk": qk(), "pv": pv(), "softmax": softmax()}
    live = dict(agents)
    for _ in range(200000):
        moves = [("agent", n) for n in live]
        moves += [("land", i) for i in range(len(landing))]
        moves += [("mma", q) for q in mma_q if mma_q[q]]
        if not live and not landing and not any(mma_q.values()):
            return
        kind, x = rng.choice(moves)
        if kind == "agent":
            try:
                next(live[x])
            except StopIteration:
                del live[x]
        elif kind == "land":
            stage = landing.pop(x)
            in_flight[stage] -= 1
            ring_full[stage].c += 1
        else:
            mma_q[x].pop(0).c += 1
    raise Violation("no progress")


@pytest.mark.parametrize("ns", list(range(4, 13)))
def test_split_rings_sound(ns):
    rng = random.Random(1000 + ns)
    for trial in range(600):
        run_cta(ns, rng.randint(1, 12), split_rings, rng)


def random_items(rng, G):
    """G blocks cut into items, with empty items mixed in."""
    items, left = [], G
    while left > 0 or rng.random() < 0.2:
        if rng.random() < 0.15:
            items.append(0)
            continue
        nb = rng.randint(1, max(1, left)) if left > 0 else 0
        items.append(nb)
        left -= nb
        if left == 0 and rng.random() < 0.7:
            break
    return items


@pytest.mark.parametrize("ns", [4, 5, 6, 12])
def test_item_handoff_sound(ns):
    """Several items per CTA, empty ones included: staging handoff and the
    epilogue's wait on the last value MMA stay sound and free of deadlock."""
    rng = random.Random(77 + ns)
    for trial in range(500):
        G = rng.randint(0, 12)
        items = random_items(rng, G)
        run_cta(ns, G, split_rings, rng, items=items)


def test_shared_ring_with_odd_depth_is_unsound():
    """The model finds the early pass that a shared ring of odd depth allows."""
    for ns in (3, 5):
        rng = random.Random(7 + ns)
        found = False
        for _ in range(2000):
            try:
                run_cta(ns, 10, shared_ring, rng, tail_wait=False)
            except Violation as e:
                assert "qk RING_FULL" in str(e) or "producer" in str(e)
                found = True
                break
        assert found, f"no violation found for shared ring depth {ns}"


def test_shared_ring_with_even_depth_holds_in_the_model():
    rng = random.Random(3)
    for _ in range(300):
        run_cta(6, rng.randint(1, 12), shared_ring, rng, tail_wait=False)

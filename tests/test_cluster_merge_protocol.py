"""Host model of the decode kernel's in-cluster merge handshake.

The k CTAs of a thread-block cluster take the same work items in the same
order (CTA q*k + j holds piece j of every pair of cluster q).  For each item,
the softmax warpgroup of every CTA sends two things into a staging buffer of
each CTA of the cluster: its normalised rows of the columns that CTA owns, and
the LSEs of its columns.  Both go by st.async and complete transaction bytes on
the receiver's PEER_FULL barrier of that buffer.

The receiver then posts the expected bytes itself (one expect-tx arrival),
waits on PEER_FULL, and merges the k pieces.  Except after its last item, each
of its four warps then arrives on that buffer's PEER_EMPTY barrier in every CTA
of the cluster, so 4 k arrivals complete a phase.  A sender waits on PEER_EMPTY
before it writes into a buffer again (NB = 2 buffers, used in turn).

Before leaving, a CTA waits for the PEER_EMPTY phases that no later staging
wait consumed, which covers every item but the last.  It then meets the others
at a relaxed cluster barrier.  That barrier orders no memory operation, so a
message still in flight past it could land in a CTA that has already left.

The model runs the k CTAs and every message in flight (data pieces and remote
arrivals) under random interleavings. It checks that:
- each parity wait follows the mbarrier rule that test_pipeline_protocol also
  checks: a wait on phase p starts with p or p + 1 phases completed;
- a piece lands in a buffer only after its receiver has merged the item that
  buffer held before, and a merge reads k pieces of its own item;
- no message reaches a CTA before it has initialised its barriers or after it
  has left, and every CTA leaves (no deadlock).
Mutants of the protocol show that these checks are not vacuous.

The model is sequentially consistent.  With two buffers, a sender cannot get
two items ahead of a receiver even without the staging wait, because it needs
the receiver's pieces of the item in between.  The staging wait's other role,
as the release/acquire edge that orders a receiver's reads before the sender's
next writes, is outside such a model.  With one buffer the wait is what keeps
a sender from overwriting a piece not merged yet, and a mutant shows it.
"""
import random

import pytest

NB = 2          # staging buffers per warpgroup
WARPS = 4       # warps of the softmax warpgroup; each arrives on PEER_EMPTY
ROWS, LSES = 96, 16  # bytes of a piece's rows and of its LSEs (any positive sizes)


class Violation(Exception):
    pass


class Barrier:
    """An mbarrier phase: `count` arrivals and a transaction byte count that
    may go negative while bytes land before the expect-tx arrival."""

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.c = 0  # completed phases

    def _complete_if_done(self):
        if self.pending == 0 and self.tx == 0:
            self.c += 1
            self.pending = self.count

    def arrive(self, expect_bytes=0):
        self.tx += expect_bytes
        self.pending -= 1
        self._complete_if_done()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._complete_if_done()


def parity_wait(bar, phase, what):
    """A predicate for a wait on `phase` of `bar` by parity, checking the rule
    each time it is polled."""

    def ready():
        if bar.c not in (phase, phase + 1):
            raise Violation(f"{what}: waits on phase {phase} with {bar.c} completed")
        return (bar.c & 1) != (phase & 1)

    return ready


class Cluster:
    def __init__(self, k, items, rng, mutant=None, nb=NB):
        self.k, self.items, self.rng, self.mutant, self.nb = k, items, rng, mutant, nb
        NB = nb
        self.full = [[Barrier(1) for _ in range(NB)] for _ in range(k)]
        self.empty = [[Barrier(WARPS * k) for _ in range(NB)] for _ in range(k)]
        # buf[receiver][buffer][sender] = [item of the rows, item of the LSEs]
        self.buf = [[[[None, None] for _ in range(k)] for _ in range(NB)] for _ in range(k)]
        self.merged = [[-1] * NB for _ in range(k)]  # last item merged out of each buffer
        self.initialised = [False] * k
        self.at_exit = [False] * k
        self.left = [False] * k
        self.inflight = []

    def deliver(self, msg):
        kind, tgt, ob, snd, item, part = msg
        NB = self.nb
        if self.left[tgt]:
            raise Violation(f"{kind} of item {item} from CTA {snd} lands in CTA {tgt} after it left")
        if not self.initialised[tgt]:
            raise Violation(f"{kind} lands in CTA {tgt} before its barriers are initialised")
        if kind == "piece":
            before = item - NB if item >= NB else -1
            if self.merged[tgt][ob] != before:
                raise Violation(f"item {item} from CTA {snd} overwrites buffer {ob} of CTA {tgt}, "
                                f"which last merged item {self.merged[tgt][ob]}")
            self.buf[tgt][ob][snd][part] = item
            self.full[tgt][ob].complete_tx(ROWS if part == 0 else LSES)
        else:
            self.empty[tgt][ob].arrive()

    def cta(self, j, n_items):
        """CTA j's softmax warpgroup: yields the predicate it waits on next
        (None: it may simply continue later)."""
        m, NB = self.mutant, self.nb
        self.initialised[j] = True  # barriers initialised, then the cluster arrive
        cluster_waited = False
        for i in range(n_items):
            ob, last = i % NB, i == n_items - 1
            if i >= NB and m != "no_staging_wait":
                phase = i // NB if m == "staging_parity" else i // NB - 1
                yield parity_wait(self.empty[j][ob], phase, f"CTA {j} staging wait, item {i}")
            if not cluster_waited and m != "no_init_wait":
                yield lambda: all(self.initialised)
            cluster_waited = True
            for part in (0, 1):  # rows to their owners, LSEs to every CTA
                for t in range(self.k):
                    self.inflight.append(("piece", t, ob, j, i, part))
            yield None
            expect = self.k * (ROWS + LSES) - (LSES if m == "expect_short" else 0)
            self.full[j][ob].arrive(expect)
            yield parity_wait(self.full[j][ob], i // NB, f"CTA {j} piece wait, item {i}")
            for s in range(self.k):
                if self.buf[j][ob][s] != [i, i]:
                    raise Violation(f"CTA {j} merges item {i} with {self.buf[j][ob][s]} from CTA {s}")
            self.merged[j][ob] = i
            if not last or m == "arrive_after_last":
                for w in range(WARPS):
                    for t in range(self.k):
                        self.inflight.append(("arrive", t, ob, j, i, w))
                    yield None
        if m != "no_exit_wait":
            for i in range(max(n_items - NB, 0), n_items - 1):
                yield parity_wait(self.empty[j][i % NB], i // NB, f"CTA {j} exit wait, item {i}")
        self.at_exit[j] = True
        yield lambda: all(self.at_exit)
        self.left[j] = True


def run_cluster(k, n_items, seed, mutant=None, extra_item_cta=None, nb=NB):
    """Runs one cluster to the end under a random schedule.  The bias towards
    delivering messages late or early is drawn per run."""
    rng = random.Random(seed)
    cl = Cluster(k, n_items, rng, mutant, nb)
    counts = [n_items + (1 if j == extra_item_cta else 0) for j in range(k)]
    gens = [cl.cta(j, counts[j]) for j in range(k)]
    preds = [None] * k
    done = [False] * k
    p_msg = rng.uniform(0.05, 0.95)
    while not all(done) or cl.inflight:
        agents = [j for j in range(k) if not done[j] and (preds[j] is None or preds[j]())]
        if not agents and not cl.inflight:
            raise Violation(f"deadlock: CTAs {[j for j in range(k) if not done[j]]} wait forever")
        if cl.inflight and (not agents or rng.random() < p_msg):
            cl.deliver(cl.inflight.pop(rng.randrange(len(cl.inflight))))
            continue
        j = rng.choice(agents)
        try:
            preds[j] = next(gens[j])
        except StopIteration:
            done[j] = True
    return cl


CASES = [(k, n, nb) for k in (2, 4, 8) for n in (1, 2, 3, 5) for nb in (1, 2)]


@pytest.mark.parametrize("k,n_items,nb", CASES)
def test_merge_handshake_is_sound(k, n_items, nb):
    for seed in range(40):
        cl = run_cluster(k, n_items, seed, nb=nb)
        assert all(cl.left)
        for j in range(k):  # every buffer was merged up to its last item
            for ob in range(nb):
                own = [i for i in range(n_items) if i % nb == ob]
                assert cl.merged[j][ob] == (own[-1] if own else -1)


@pytest.mark.parametrize("mutant,n_items,nb,expect", [
    # an arrival for the second-last item lands after its target has left
    ("no_exit_wait", 3, 2, "after it left"),
    # arrivals for the last item have no wait to cover them
    ("arrive_after_last", 2, 2, "after it left"),
    # one buffer: a sender rewrites it before its receiver has merged it
    ("no_staging_wait", 3, 1, "overwrites buffer"),
    # a wait on the wrong phase never passes (the kernel's bounded wait runs out)
    ("staging_parity", 3, 2, "deadlock|waits on phase"),
    # a piece reaches a CTA whose barriers are not set up yet
    ("no_init_wait", 1, 2, "before its barriers"),
    # the receiver expects fewer bytes than the k pieces carry: it merges too
    # early, or (all bytes in before the expect-tx) the phase never completes
    ("expect_short", 2, 2, "merges item|deadlock"),
])
def test_protocol_mutants_are_caught(mutant, n_items, nb, expect):
    import re

    caught = []
    for seed in range(200):
        try:
            run_cluster(4, n_items, seed, mutant, nb=nb)
        except Violation as e:
            caught.append(str(e))
    assert caught and all(re.search(expect, msg) for msg in caught), caught[:3]


def test_cluster_out_of_lockstep_deadlocks():
    """One CTA with an item more than the others waits for pieces nobody
    sends: in the kernel that wait runs out and sets the error word, which is
    why the plan must give a cluster's CTAs the same items in the same order."""
    with pytest.raises(Violation, match="deadlock"):
        run_cluster(2, 2, 0, extra_item_cta=1)

"""The adjuster (Rimuru, section "The adjuster: when to evict an expert, and which one?").

Part 1 pins the oracle to the section: its two printed examples (tests/golden), the hysteresis
gap and the cap, and hand-worked choices of which expert moves.  Part 2 checks libpmoe's native
adjuster against the oracle, change list by change list, on seeded random round sequences, and
its argument checks.  Everything here is host code: no GPU is needed.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle.adjuster import AdjusterOracle
from paged_moe_expert_gb300 import _lib, build
from paged_moe_expert_gb300.adjuster import Adjuster

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "adjuster_examples.json")

# Three layers of four experts.  Layer 1 ranks 1, 2, 3, 0; layer 2 is all ties (ranks 0..3).
PROBS = np.array([[0.40, 0.30, 0.20, 0.10],
                  [0.05, 0.50, 0.25, 0.20],
                  [0.25, 0.25, 0.25, 0.25]], dtype=np.float32)
CACHED = [2, 2, 3]  # pages: L0 e0 0-2, e1 3-5; L1 e1 6-8, e2 9-11; L2 e0 12-14, e1 15-17, e2 18-20


# ---- part 1: the oracle against the section ------------------------------------------------

def test_printed_examples():
    g = json.load(open(GOLDEN))
    for ex in g["examples"]:
        ev, add = AdjusterOracle.counts(ex["short_pages"], ex["free_pages"])
        assert (ev, add) == (ex["evict"], ex["add"]), ex["what"]
        if "pages_freed" in ex:
            assert ev * g["pages_per_expert"] == ex["pages_freed"]
            assert ex["pages_freed"] - ex["short_pages"] == ex["spare_after_cover"]


def count_pins_hold(C):
    """The count rule's pins, as a predicate so that planted mistakes can be run through it."""
    ok = C(0, 0) == (1, 0) and C(0, 1) == (1, 0)                 # fewer than 2 free: evict one
    ok &= all(C(0, F) == (0, 0) for F in range(2, 12))           # 2..9 free, and floor(<1) = 0
    ok &= C(0, 12) == (0, 1) and C(0, 23) == (0, 4) and C(0, 24) == (0, 5)
    ok &= C(0, 1000) == (0, 5)                                   # at most 5 per round
    # Shortfall wins over free pages; the evictions cover R_b + 1 pages with no whole expert
    # to spare.
    for R in range(1, 40):
        ev, add = C(R, 50)
        ok &= add == 0 and 3 * ev >= R + 1 and 3 * (ev - 1) < R + 1
    return bool(ok)


def test_hysteresis_gap_and_cap():
    assert count_pins_hold(AdjusterOracle.counts)


def test_grow_takes_the_most_probable_nominees():
    o = AdjusterOracle(PROBS, CACHED, offload_limit=3, num_pages=40)
    assert o.free_pages() == 19  # 21 pages hold the 7 cached experts
    # F_b = 19 -> add 3.  Nominees: L0 e2 (0.20), L1 e3 (0.20), L2 e3 (0.25); the L0/L1 tie goes
    # to layer 0.  Reserved pages are the lowest free ids, 21 upward.
    assert o.decide(0) == [[1, 2, 3, 21, 22, 23], [1, 0, 2, 24, 25, 26], [1, 1, 3, 27, 28, 29]]
    assert o.kept == [3, 3, 4] and o.free_pages() == 10
    assert o.decide(0) == []  # 10 free: inside the gap


def test_shrink_takes_the_least_probable_and_frees_after_the_pass():
    o = AdjusterOracle(PROBS, CACHED, offload_limit=3, num_pages=40)
    o.decide(0)
    o.end_forward()
    # Short 8 -> evict 3.  Last kept: L0 e2 (0.20), L1 e3 (0.20), L2 e3 (0.25).
    ch = o.decide(8)
    assert ch == [[-1, 0, 2, 24, 25, 26], [-1, 1, 3, 27, 28, 29], [-1, 2, 3, 21, 22, 23]]
    assert o.free_pages() == 10                    # still the running pass's
    assert o.page_table(0)[2] == [24, 25, 26]
    o.end_forward()
    assert o.free_pages() == 19 and o.page_table(0)[2] == [-1, -1, -1]
    assert o.kept == [2, 2, 3]


def test_precautionary_eviction_and_layer_tie():
    o = AdjusterOracle(PROBS, CACHED, offload_limit=3, num_pages=22)
    assert o.free_pages() == 1
    # F_b = 1 -> evict 1.  Last kept: L0 e1 (0.30), L1 e2 (0.25), L2 e2 (0.25): L1 wins the tie.
    assert o.decide(0) == [[-1, 1, 2, 9, 10, 11]]


def test_offload_limit_excludes_layers():
    o = AdjusterOracle(PROBS, CACHED, offload_limit=2, num_pages=40)
    # L0 and L1 already offload 2 experts: only L2 nominates.
    assert o.decide(1) == [[-1, 2, 2, 18, 19, 20]]
    o.end_forward()
    assert o.decide(5) == []  # now every layer offloads 2
    o.end_forward()


def test_ranking_ties_go_to_the_lower_expert():
    o = AdjusterOracle(PROBS, [0, 0, 0], offload_limit=4, num_pages=100)
    assert o.ranking[2] == [0, 1, 2, 3] and o.ranking[1] == [1, 2, 3, 0]


def check_invariants(o):
    seen = {}
    for p, own in enumerate(o.owner):
        if own is not None and own[0] == "expert":
            key = (own[1], own[2], own[3])
            assert key not in seen, "two pages for one matrix"
            seen[key] = p
    pend = set(o.pending)
    for l in range(o.L):
        kept = set(o.ranking[l][:o.kept[l]])
        holders = {e for (ll, e, j) in seen if ll == l}
        assert holders == kept | {e for (ll, e) in pend if ll == l}  # top slice, plus pending
        for e in holders:
            assert all((l, e, j) in seen for j in range(3))


def test_random_rounds_keep_the_invariants():
    rng = np.random.default_rng(1)
    for trial in range(20):
        L, E = int(rng.integers(1, 6)), int(rng.integers(1, 9))
        probs = rng.dirichlet(np.ones(E), size=L).astype(np.float32)
        cached = rng.integers(0, E + 1, size=L)
        o = AdjusterOracle(probs, cached, int(rng.integers(0, E + 1)),
                           3 * int(cached.sum()) + int(rng.integers(0, 30)))
        for _ in range(30):
            o.decide(int(rng.integers(0, 12)) if rng.random() < 0.4 else 0)
            check_invariants(o)
            o.end_forward()
            check_invariants(o)


def test_planted_mistakes_are_caught():
    """The pins above fail for plausible slips in the oracle (planted on the CPU only)."""
    def floor_evict(R_b, F_b):
        ev, add = AdjusterOracle.counts(R_b, F_b)
        return ((R_b + 1) // 3 if R_b > 0 else ev), add

    def no_extra_page(R_b, F_b):
        ev, add = AdjusterOracle.counts(R_b, F_b)
        return (math.ceil(R_b / 3) if R_b > 0 else ev), add

    def no_cap(R_b, F_b):
        ev, add = AdjusterOracle.counts(R_b, F_b)
        return ev, ((F_b - 9) // 3 if add else add)

    def grow_at_9(R_b, F_b):
        ev, add = AdjusterOracle.counts(R_b, F_b)
        return ev, (min(5, (F_b - 8) // 3) if R_b == 0 and F_b >= 9 else add)

    for m in (floor_evict, no_extra_page, no_cap, grow_at_9):
        assert not count_pins_hold(m), m.__name__

    class HighestEvicted(AdjusterOracle):  # shrink sorted the wrong way
        def decide(self, R_b, max_changes=None):
            self.probs = [[-p for p in row] for row in self.probs]
            try:
                return super().decide(R_b, max_changes)
            finally:
                self.probs = [[-p for p in row] for row in self.probs]

    class LaterLayerWinsTies(AdjusterOracle):
        def decide(self, R_b, max_changes=None):
            self.probs = [[p - 1e-9 * l for p in row] for l, row in enumerate(self.probs)]
            return super().decide(R_b, max_changes)

    assert HighestEvicted(PROBS, CACHED, 3, 22).decide(0) != [[-1, 1, 2, 9, 10, 11]]
    assert LaterLayerWinsTies(PROBS, CACHED, 3, 22).decide(0) != [[-1, 1, 2, 9, 10, 11]]


# ---- part 2: the native adjuster against the oracle ----------------------------------------

@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def same_state(a, o):
    assert a.free_pages() == o.free_pages()
    assert list(a.cached()) == o.kept
    for l in range(o.L):
        assert a.page_table(l).tolist() == o.page_table(l)


def test_native_matches_worked_examples(lib):
    a = Adjuster(PROBS, CACHED, 3, 40)
    assert a.decide(0).tolist() == [[1, 2, 3, 21, 22, 23], [1, 0, 2, 24, 25, 26], [1, 1, 3, 27, 28, 29]]
    a.end_forward()
    assert a.decide(8).tolist() == [[-1, 0, 2, 24, 25, 26], [-1, 1, 3, 27, 28, 29], [-1, 2, 3, 21, 22, 23]]
    assert a.free_pages() == 10
    a.end_forward()
    assert a.free_pages() == 19
    assert Adjuster(PROBS, CACHED, 3, 22).decide(0).tolist() == [[-1, 1, 2, 9, 10, 11]]


@pytest.mark.parametrize("seed", range(12))
def test_native_matches_oracle_on_random_rounds(lib, seed):
    rng = np.random.default_rng(100 + seed)
    L, E = int(rng.integers(1, 12)), int(rng.integers(1, 65))
    # Skewed per-layer popularity like a router's, with some exact ties.
    probs = rng.dirichlet(np.full(E, 0.3), size=L).astype(np.float32)
    probs[rng.random((L, E)) < 0.1] = np.float32(0.0)
    cached = rng.integers(0, E + 1, size=L)
    limit = int(rng.integers(0, E + 1))
    pages = 3 * int(cached.sum()) + int(rng.integers(0, 60))
    a, o = Adjuster(probs, cached, limit, pages), AdjusterOracle(probs, cached, limit, pages)
    same_state(a, o)
    lent = []
    for _ in range(40):
        r = rng.random()
        if r < 0.15 and a.free_pages() > 0:
            n = int(rng.integers(1, a.free_pages() + 1))
            got = a.lend(n).tolist()
            assert got == o.lend(n)
            lent += got
        elif r < 0.25 and lent:
            back = [lent.pop(int(rng.integers(0, len(lent)))) for _ in range(int(rng.integers(1, len(lent) + 1)))]
            a.give_back(back)
            o.give_back(back)
        R = int(rng.integers(1, 20)) if rng.random() < 0.35 else 0
        mc = int(rng.integers(0, L + 1)) if rng.random() < 0.2 else L
        assert a.decide(R, mc).tolist() == o.decide(R, mc)
        same_state(a, o)
        a.end_forward()
        o.end_forward()
        same_state(a, o)


def test_native_argument_checks(lib):
    with pytest.raises(_lib.PmoeError, match="INVALID_ARG"):
        Adjuster(PROBS, CACHED, 3, 20)                     # 21 pages needed
    with pytest.raises(_lib.PmoeError, match="INVALID_ARG"):
        Adjuster(PROBS, [5, 0, 0], 3, 40)                  # more than E cached
    bad = PROBS.copy()
    bad[1, 1] = np.nan
    with pytest.raises(_lib.PmoeError, match="finite"):
        Adjuster(bad, CACHED, 3, 40)
    a = Adjuster(PROBS, CACHED, 3, 40)
    with pytest.raises(_lib.PmoeError, match="INVALID_ARG"):
        a.decide(-1)
    a.decide(8)
    with pytest.raises(_lib.PmoeError, match="end_forward"):
        a.decide(0)                                        # evictions still pending
    a.end_forward()
    with pytest.raises(_lib.PmoeError):
        a.lend(a.free_pages() + 1)
    got = a.lend(2)
    with pytest.raises(_lib.PmoeError):
        a.give_back([got[0], got[0]])                      # listed twice
    with pytest.raises(_lib.PmoeError):
        a.give_back([0])                                   # an expert's page, not lent
    free = a.free_pages()
    a.give_back(got)
    assert a.free_pages() == free + 2
    with pytest.raises(_lib.PmoeError):
        a.page_table(3)


# ---- part 3: the round protocol around it (host bookkeeping of the elastic stack) -----------

def test_kv_round():
    from paged_moe_expert_gb300.pipeline import kv_round
    assert kv_round(0, 0, 5) == (0, 0, 0)
    assert kv_round(0, 10, 4) == (4, 0, 6)        # lend what is free, the rest is R_b
    assert kv_round(10, 3, 0) == (0, 7, 0)        # demand fell: give pages back
    assert kv_round(2, 5, 9) == (3, 0, 0)


def test_constant_kv_demand_is_met_within_a_few_rounds():
    """With the oracle adjuster and the round protocol (KV first, then the adjuster, pages of
    evicted experts free after the pass), a constant demand that the evictable experts can cover
    stops being short after a few rounds, and a demand that drops to zero lets the cache grow
    back until fewer than 12 pages are free (below that floor((F_b - 9) / 3) adds nothing)."""
    from paged_moe_expert_gb300.pipeline import kv_round
    rng = np.random.default_rng(5)
    L, E, limit = 6, 10, 6
    probs = rng.dirichlet(np.ones(E), size=L).astype(np.float32)
    o = AdjusterOracle(probs, [E] * L, limit, 3 * E * L + 4)
    held, shorts = 0, []
    for need in [60] * 12 + [0] * 30:
        take, back, short = kv_round(held, need, o.free_pages())
        held += take - back
        if take:
            o.lend(take)
        if back:
            lent = [p for p, own in enumerate(o.owner) if own == ("lent",)]
            o.give_back(lent[-back:])
        o.decide(short)
        o.end_forward()
        shorts.append(short)
    assert shorts[0] > 0 and shorts[11] == 0
    assert o.free_pages() < 12 and o.free_pages() == 4 + 3 * (E * L - sum(o.kept))
    assert sum(o.kept) < E * L  # 4 spare pages + 2 missing experts = 10 free: inside the gap


# ---- part 4: KV pages carved from lent expert pages (the unified pool) ----------------------

def expert_pages_in_use(a, L):
    used = set()
    for l in range(L):
        for row in a.page_table(l):
            used |= {int(p) for p in row if p >= 0}
    return used


def test_kv_pages_live_only_on_lent_pages(lib):
    from paged_moe_expert_gb300.pipeline import KVPages
    rng = np.random.default_rng(8)
    L, E, page, kvb = 3, 6, 64, 16                        # 4 KV pages per expert page
    probs = rng.dirichlet(np.ones(E), size=L).astype(np.float32)
    pages = 3 * E * L + 6
    a = Adjuster(probs, [E] * L, 4, pages)
    kv = KVPages(a, pages, page, kvb)
    # request 1 takes 5 KV pages: two expert pages lent, the request's pages share them
    assert kv.allocate(1, 5) == 0
    offs = kv.live()[1]
    assert len({o // page for o in offs}) == 2 and a.free_pages() == 4
    # request 2 has no page yet: it takes the free KV pages already split off (request 1's
    # second expert page) before another expert page is lent
    assert kv.allocate(2, 2) == 0
    assert {o // page for o in kv.live()[2]} == {max(o // page for o in offs)}
    before = a.free_pages()
    kv.release(1)
    assert a.free_pages() == before + 1                    # request 1's full page came back
    live = kv.live()[2]
    assert all(o // page not in expert_pages_in_use(a, L) for o in live)


def test_random_rounds_keep_kv_and_experts_apart(lib):
    from paged_moe_expert_gb300.pipeline import KVPages
    rng = np.random.default_rng(9)
    L, E, page, kvb = 4, 8, 64, 16
    probs = rng.dirichlet(np.full(E, 0.5), size=L).astype(np.float32)
    pages = 3 * E * L + 9
    a = Adjuster(probs, [E] * L, 5, pages)
    kv = KVPages(a, pages, page, kvb)
    active, nxt, waiting = {}, 0, {}
    for rnd in range(60):
        departures = [r for r in list(active) if rng.random() < 0.3]
        for r in departures:
            del active[r]
        arrivals = dict(waiting)
        waiting = {}
        for _ in range(int(rng.integers(0, 4))):
            arrivals[nxt] = int(rng.integers(1, 9))
            nxt += 1
        for r in departures:
            kv.release(r)
        short_kv = 0
        for r, n in arrivals.items():
            miss = kv.allocate(r, n)
            active[r] = True
            if miss:
                waiting[r] = miss
                short_kv += miss
        a.decide(-(-short_kv // kv.per_page))
        # experts (including the evicted ones still readable this pass) never share a page with KV
        kv_pages = {o // page for offs in kv.live().values() for o in offs}
        assert not kv_pages & expert_pages_in_use(a, L)
        spans = sorted(o for offs in kv.live().values() for o in offs)
        assert len(spans) == len(set(spans))
        a.end_forward()
    assert nxt > 0


def test_kv_pages_on_native_allocators_match_the_oracles(lib):
    """The same request rounds through KVPages (native adjuster and tiers) and through the same
    composition over the two oracles give the same KV offsets, change lists and free counts."""
    from oracle.tiers import EXPERT as O_EXPERT, KV as O_KV, TiersOracle
    from paged_moe_expert_gb300.pipeline import KVPages

    class OracleKV:
        def __init__(self, adj, pages, page, kvb):
            self.t = TiersOracle(pages * page, page, 0, kvb, 0)
            for p in range(pages):
                assert self.t.alloc(O_EXPERT) == p * page
            self.adj, self.page, self.req = adj, page, {}

        def allocate(self, rid, n):
            got = self.req.setdefault(rid, [])
            for i in range(n):
                off = self.t.alloc(O_KV, rid)
                if off is None and self.adj.free_pages() > 0:
                    p = self.adj.lend(1)[0]
                    self.t.free(O_EXPERT, p * self.page)
                    off = self.t.alloc(O_KV, rid)
                if off is None:
                    return n - i
                got.append(off)
            return 0

        def release(self, rid):
            for off in self.req.pop(rid, []):
                self.t.free(O_KV, off)
            c = self.t.stats()
            for _ in range(c[1] + c[2]):
                off = self.t.alloc(O_EXPERT)
                self.adj.give_back([off // self.page])

    rng = np.random.default_rng(12)
    L, E, page, kvb = 3, 8, 64, 16
    probs = rng.dirichlet(np.full(E, 0.5), size=L).astype(np.float32)
    pages = 3 * E * L + 7
    a, o = Adjuster(probs, [E] * L, 5, pages), AdjusterOracle(probs, [E] * L, 5, pages)
    kn, ko = KVPages(a, pages, page, kvb), OracleKV(o, pages, page, kvb)
    active, nxt = set(), 0
    for rnd in range(50):
        departures = [r for r in sorted(active) if rng.random() < 0.3]
        for r in departures:
            active.discard(r)
            kn.release(r)
            ko.release(r)
        short = 0
        for _ in range(int(rng.integers(0, 4))):
            n = int(rng.integers(1, 10))
            mn, mo = kn.allocate(nxt, n), ko.allocate(nxt, n)
            assert mn == mo
            short += mn
            active.add(nxt)
            nxt += 1
        assert kn.live() == {r: v for r, v in ko.req.items()}
        R = -(-short // (page // kvb))
        assert a.decide(R).tolist() == o.decide(R)
        assert a.free_pages() == o.free_pages()
        a.end_forward()
        o.end_forward()

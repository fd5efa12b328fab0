"""Three tiers of pages over one pool (Rimuru, section "One pool for data whose sizes differ by
orders of magnitude").

Part 1 pins the oracle to the section: the huge page size, the section's worked example of KV
pages carved from one expert page for three requests, the split order (split small pages first,
then an expert page, a huge page only through expert pages), the merge order, same-request
placement, and byte accounting over random sequences; planted mistakes fail the pins.  Part 2
checks libpmoe's native allocator against the oracle call by call.  Part 3: the memory views.
Host only: no GPU needed.
"""
import math

import numpy as np
import pytest
import torch

from oracle.tiers import CONV, EXPERT, KV, SSM, TiersOracle
from paged_moe_expert_gb300 import _lib, build
from paged_moe_expert_gb300 import tiers as tr

# ---- part 1: the oracle against the section ------------------------------------------------


def test_huge_page_is_the_lcm():
    assert TiersOracle(100, 6, ssm_page=4).huge == 12
    assert TiersOracle(100, 6).huge == 6                    # no SSM state: the expert page
    # a Qwen1.5-shaped expert page (5.77 MB = 11 * 512 KiB) with a 2 MiB SSM page: 4 expert
    # pages = 11 SSM pages per huge page
    assert TiersOracle(10 ** 9, 5767168, ssm_page=2097152).huge == 23068672 == 4 * 5767168 == 11 * 2097152


def worked_example(T):
    """Two expert-sized huge pages; KV pages of a quarter expert page."""
    t = T(2 * 8, 8, kv_page=2)
    got = [t.alloc(KV, owner) for owner in (1, 2, 3)]
    return t, got


def test_worked_example_three_requests_on_one_expert_page():
    t, got = worked_example(TiersOracle)
    assert got == [0, 2, 4]                                 # one split expert page serves all three
    t.free(KV, 0)
    t.free(KV, 2)                                           # requests 1 and 2 finish ...
    assert t.stats()[6] == 1                                # ... the page is still split
    assert t.alloc(EXPERT) == 8                             # an expert goes to the other page,
    assert t.alloc(EXPERT) is None                          # not into the freed KV space
    assert t.alloc(KV, 9) == 0                              # which still serves the KV cache
    t.free(KV, 0)
    t.free(KV, 4)                                           # the third request finishes:
    assert t.stats() == [8, 1, 0, 0, 1, 0, 0, 0]            # the page merged back, whole again


def test_small_pages_never_cut_straight_from_a_huge_page():
    t = TiersOracle(24, 6, ssm_page=4, kv_page=3)           # huge page 12 = two expert pages
    assert t.alloc(KV, 1) == 0
    # the huge page became two expert pages; one was split into KV pages, one is a free expert page
    assert t.stats() == [12, 1, 1, 0, 0, 0, 1, 1]
    assert t.alloc(SSM) == 12                               # SSM pages come from the other huge page
    assert t.stats()[1] == 0 and t.stats()[3] == 2


def test_split_order_small_then_expert_then_huge():
    t = TiersOracle(2 * 12, 6, ssm_page=4, kv_page=3)
    a = t.alloc(KV, 1)                                      # splits huge 0 -> expert pages 0, 6
    b = t.alloc(KV, 2)                                      # the free small page of page 0
    c = t.alloc(KV, 3)                                      # then the free expert page 6
    d = t.alloc(KV, 4)
    e = t.alloc(KV, 5)                                      # only now huge page 1
    assert (a, b, c, d, e) == (0, 3, 6, 9, 12)


def test_same_request_shares_a_split_page():
    t = TiersOracle(3 * 8, 8, kv_page=2)
    x = [t.alloc(KV, o) for o in (1, 2, 1, 2)]              # page 0 full: 0 2 4 6
    assert x == [0, 2, 4, 6]
    assert t.alloc(KV, 3) == 8                              # new split page 8
    t.free(KV, 2)                                           # request 2 frees a slot on page 0
    assert t.alloc(KV, 3) == 10                             # request 3 stays on its own page 8
    assert t.alloc(KV, 1) == 2                              # request 1 returns to page 0


def test_merge_upward_to_a_whole_huge_page():
    t = TiersOracle(12, 6, ssm_page=4, kv_page=3)
    k = t.alloc(KV, 1)
    e = t.alloc(EXPERT)
    assert t.stats()[1] == 0
    t.free(EXPERT, e)
    assert t.stats()[1] == 0                                # page 0 is still split
    t.free(KV, k)
    assert t.stats() == [12, 1, 0, 0, 0, 0, 0, 0]


def accounting(t):
    """Every byte of the whole huge pages is exactly one of: free huge, free middle, live middle,
    split expert page."""
    c = t.stats()
    H = c[0]
    used = c[1] * H + (c[2] + c[4] + c[6]) * t.size[EXPERT] + (c[3] + c[5]) * t.size[SSM]
    return used == len(t.pages) * H


def test_random_sequences_keep_pages_disjoint_and_bytes_accounted():
    rng = np.random.default_rng(2)
    for trial in range(40):
        e = int(rng.choice([6, 8, 12]))
        ssm = int(rng.choice([0, 4, 9]))
        kv = int(rng.choice([1, 2, 3]))
        kv = kv if e % kv == 0 else 1
        t = TiersOracle(int(rng.integers(1, 60)), e, ssm, kv, 2 if e % 2 == 0 else 0)
        kinds = [EXPERT, KV] + ([SSM] if ssm else []) + ([CONV] if t.size[CONV] else [])
        live = []
        for _ in range(80):
            if live and rng.random() < 0.45:
                k, off = live.pop(int(rng.integers(0, len(live))))
                t.free(k, off)
            else:
                k = int(rng.choice(kinds))
                off = t.alloc(k, int(rng.integers(0, 3)))
                if off is not None:
                    live.append((k, off))
            spans = sorted((off, off + t.size[k]) for k, off in live)
            assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
            assert all(0 <= s and e_ <= len(t.pages) * t.huge for s, e_ in spans)
            assert accounting(t)
        for k, off in live:
            t.free(k, off)
        assert t.stats()[1] == len(t.pages)                 # everything merged back


def test_planted_mistakes_are_caught():
    class StraightToKV(TiersOracle):                         # cuts a huge page into small pages
        def alloc(self, kind, owner=0):
            if kind == KV and not any(hp is not None for hp in self.pages):
                self.size[EXPERT], keep = self.huge, self.size[EXPERT]
                try:
                    return super().alloc(kind, owner)
                finally:
                    self.size[EXPERT] = keep
            return super().alloc(kind, owner)

    class NoAffinity(TiersOracle):
        def alloc(self, kind, owner=0):
            return super().alloc(kind, 0)

    class NoMerge(TiersOracle):
        def _give_middle(self, off):
            self._huge_of(off)["pages"][off] = "free"

    _never_straight(TiersOracle)
    with pytest.raises(AssertionError):
        _never_straight(StraightToKV)
    t = NoAffinity(3 * 8, 8, kv_page=2)
    [t.alloc(KV, o) for o in (1, 2, 1, 2)]
    t.alloc(KV, 3)
    t.free(KV, 2)
    assert t.alloc(KV, 3) != 10
    t = NoMerge(12, 6, ssm_page=4, kv_page=3)
    k = t.alloc(KV, 1)
    t.free(KV, k)
    assert t.stats() != [12, 1, 0, 0, 0, 0, 0, 0]


def _never_straight(T):
    t = T(24, 6, ssm_page=4, kv_page=3)
    t.alloc(KV, 1)
    assert t.stats() == [12, 1, 1, 0, 0, 0, 1, 1]


# ---- part 2: the native allocator against the oracle ---------------------------------------

@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


@pytest.mark.parametrize("seed", range(8))
def test_native_matches_oracle(lib, seed):
    rng = np.random.default_rng(50 + seed)
    for _ in range(25):
        e = int(rng.choice([6, 8, 12, 5767168]))
        ssm = int(rng.choice([0, 4, 9])) if e < 100 else int(rng.choice([0, 2097152]))
        kv = int(rng.choice([1, 2, 3])) if e < 100 else 131072 * 11
        kv = kv if e % kv == 0 else 0
        conv = 2 if e % 2 == 0 and rng.random() < 0.5 else 0
        huge = math.lcm(e, ssm) if ssm else e
        pool = huge * int(rng.integers(1, 6)) + int(rng.integers(0, 7))
        o, t = TiersOracle(pool, e, ssm, kv, conv), tr.Tiers(pool, e, ssm, kv, conv)
        kinds = [EXPERT] + ([SSM] if ssm else []) + ([KV] if kv else []) + ([CONV] if conv else [])
        live = []
        for _ in range(70):
            if live and rng.random() < 0.4:
                k, off = live.pop(int(rng.integers(0, len(live))))
                o.free(k, off)
                t.free(k, off)
            else:
                k, own = int(rng.choice(kinds)), int(rng.integers(0, 4))
                a = o.alloc(k, own)
                assert t.alloc(k, own) == a
                if a is not None:
                    live.append((k, a))
            assert t.stats() == o.stats()
        t.close()


def test_native_worked_example(lib):
    t, got = worked_example(tr.Tiers)
    assert got == [0, 2, 4]
    t.free(KV, 0)
    t.free(KV, 2)
    assert t.alloc(EXPERT) == 8 and t.alloc(EXPERT) is None and t.alloc(KV, 9) == 0
    t.free(KV, 0)
    t.free(KV, 4)
    assert t.stats() == [8, 1, 0, 0, 1, 0, 0, 0]


def test_native_argument_checks(lib):
    with pytest.raises(_lib.PmoeError, match="divide"):
        tr.Tiers(100, 6, kv_page=4)
    with pytest.raises(_lib.PmoeError, match="INVALID_ARG"):
        tr.Tiers(100, 0)
    t = tr.Tiers(24, 6, ssm_page=4, kv_page=3)
    with pytest.raises(_lib.PmoeError, match="no pages of this kind"):
        t.alloc(CONV)
    k = t.alloc(KV, 1)
    with pytest.raises(_lib.PmoeError, match="not a live page"):
        t.free(KV, k + 1)                                   # not a page boundary
    with pytest.raises(_lib.PmoeError, match="not a live page"):
        t.free(EXPERT, 0)                                   # split, not handed out as an expert
    with pytest.raises(_lib.PmoeError, match="not a live page"):
        t.free(KV, -3)
    before = t.stats()
    with pytest.raises(_lib.PmoeError):
        t.free(KV, 3)                                       # a free slot
    assert t.stats() == before
    t.free(KV, k)
    assert t.stats() == [12, 2, 0, 0, 0, 0, 0, 0]


# ---- part 3: the memory views ----------------------------------------------------------------



def test_views_share_the_pool_bytes(lib):
    d, f = 64, 128
    expert_page = f * d * 2                               # one bf16 matrix
    kv_page = 16 * 2 * 64 * 2                             # 16 tokens of K and V, 64 dims, bf16
    pool = torch.zeros(3 * expert_page, dtype=torch.uint8)
    t = tr.Tiers(pool.numel(), expert_page, kv_page=kv_page)
    e = t.alloc(EXPERT)
    w = tr.page_view(pool, e, expert_page, torch.bfloat16, (f, d))
    w.fill_(1.5)
    assert tr.expert_page_index(e, expert_page) == 0
    t.free(EXPERT, e)                                      # reclaimed: the KV view reuses the bytes
    k = t.alloc(KV, 7)
    assert k == e
    kv = tr.page_view(pool, k, kv_page, torch.bfloat16, (16, 2, 64))
    assert kv.data_ptr() == w.data_ptr() and float(kv[0, 0, 0]) == 1.5
    kv.zero_()
    assert float(w[0, 0]) == 0.0

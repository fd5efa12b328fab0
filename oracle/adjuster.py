"""CPU oracle of the adjuster -- TEST INFRASTRUCTURE ONLY.

Only the test-suite may import this module.  It restates, in plain Python and in the order the
page gives them, the rules of Rimuru, section "The adjuster: when to evict an expert, and which
one?":

1. How many.  The scheduler reports R_b, the expert pages it is short of this round, and F_b is
   the number of free expert pages.  R_b > 0: evict ceil((R_b + 1) / 3) experts.  Otherwise
   F_b < 2: evict 1.  Otherwise F_b > 9: add min(5, floor((F_b - 9) / 3)).  Otherwise nothing.
2. Which.  An offline ranking orders every layer's experts by routing probability, and a layer
   keeps the top slice of its ranking.  To grow, each layer that has an uncached expert
   nominates the next one in its ranking; the nominees with the highest probability are added.
   To shrink, each layer nominates the last expert it keeps; the nominees with the lowest
   probability are evicted; a layer that already offloads expert_offload_limit experts does not
   nominate.
3. Pages.  An expert is three pages (W1, W3, W2).  An added expert's pages are reserved when the
   decision is made.  An evicted expert keeps its pages until the forward pass that is running
   ends; only then do they return to the pool.

Readings where the page is silent (each listed with its reason in the design notes):
ranking ties go to the lower expert id; one nominee per layer per round, so a round changes at
most one expert per layer; ties between nominees go to the lower layer; reservations take the
lowest free page ids; pages lent out (KV cache) count as neither free nor an expert's; when
fewer layers nominate than the count asks for, the round takes what there is.
"""
from __future__ import annotations

import math


class AdjusterOracle:
    def __init__(self, probs, cached, offload_limit, num_pages, max_changes=None):
        self.probs = [[float(p) for p in row] for row in probs]
        self.L = len(self.probs)
        self.E = len(self.probs[0])
        self.limit = int(offload_limit)
        self.num_pages = int(num_pages)
        # ranking[l] = experts of layer l, most probable first (ties: lower id first).
        self.ranking = [sorted(range(self.E), key=lambda e, row=row: (-row[e], e))
                        for row in self.probs]
        self.kept = [int(c) for c in cached]
        # owner[page] = ("expert", l, e, j) | ("lent",) | None (free)
        self.owner = [None] * self.num_pages
        page = 0
        for l in range(self.L):
            for r in range(self.kept[l]):
                e = self.ranking[l][r]
                for j in range(3):
                    self.owner[page] = ("expert", l, e, j)
                    page += 1
        self.pending = []  # experts evicted this round, pages not yet released

    # -- state -----------------------------------------------------------------------------
    def free_pages(self):
        return sum(1 for o in self.owner if o is None)

    def pages_of(self, l, e):
        pg = [-1, -1, -1]
        for p, o in enumerate(self.owner):
            if o is not None and o[0] == "expert" and o[1] == l and o[2] == e:
                pg[o[3]] = p
        return pg

    def page_table(self, l):
        return [self.pages_of(l, e) for e in range(self.E)]

    # -- rule 1: how many ------------------------------------------------------------------
    @staticmethod
    def counts(R_b, F_b):
        """(experts to evict, experts to add) for one round."""
        if R_b > 0:
            return math.ceil((R_b + 1) / 3), 0
        if F_b < 2:
            return 1, 0
        if F_b > 9:
            return 0, min(5, (F_b - 9) // 3)
        return 0, 0

    # -- one round -------------------------------------------------------------------------
    def decide(self, R_b, max_changes=None):
        assert not self.pending, "end_forward first"
        if max_changes is None:
            max_changes = self.L
        n_evict, n_add = self.counts(R_b, self.free_pages())
        changes = []
        if n_evict:
            # rule 2, shrink: one nominee per layer -- the last expert it keeps
            nominees = []
            for l in range(self.L):
                if self.kept[l] == 0 or self.E - self.kept[l] >= self.limit:
                    continue
                e = self.ranking[l][self.kept[l] - 1]
                nominees.append((self.probs[l][e], l, e))
            nominees.sort(key=lambda t: (t[0], t[1]))  # lowest probability first
            for p, l, e in nominees[:min(n_evict, max_changes)]:
                changes.append([-1, l, e] + self.pages_of(l, e))
                self.kept[l] -= 1
                self.pending.append((l, e))  # rule 3: pages stay until the pass ends
        elif n_add:
            # rule 2, grow: one nominee per layer -- its next uncached expert
            nominees = []
            for l in range(self.L):
                if self.kept[l] == self.E:
                    continue
                e = self.ranking[l][self.kept[l]]
                nominees.append((self.probs[l][e], l, e))
            nominees.sort(key=lambda t: (-t[0], t[1]))  # highest probability first
            for p, l, e in nominees[:min(n_add, max_changes)]:
                free = [q for q, o in enumerate(self.owner) if o is None]
                if len(free) < 3:
                    break
                for j in range(3):  # rule 3: reserve the pages now
                    self.owner[free[j]] = ("expert", l, e, j)
                changes.append([1, l, e] + free[:3])
                self.kept[l] += 1
        return changes

    def end_forward(self):
        for l, e in self.pending:
            for p, o in enumerate(self.owner):
                if o is not None and o[0] == "expert" and o[1] == l and o[2] == e:
                    self.owner[p] = None
        self.pending = []

    # -- KV cache pages of the unified pool ------------------------------------------------
    def lend(self, n):
        free = [q for q, o in enumerate(self.owner) if o is None]
        assert len(free) >= n
        for q in free[:n]:
            self.owner[q] = ("lent",)
        return free[:n]

    def give_back(self, pages):
        for q in pages:
            assert self.owner[q] == ("lent",)
            self.owner[q] = None

"""CPU oracle of the three-tier page allocator -- TEST INFRASTRUCTURE ONLY.

Only the test-suite may import this module.  Plain Python restating Rimuru, section "One pool
for data whose sizes differ by orders of magnitude":

* sizes: the huge page is the least common multiple of the expert page and the SSM page (the
  expert page alone without SSM state); middle pages are expert and SSM pages; small pages are
  KV cache and convolution-state pages.
* allocation splits downward on demand: a small page comes from a free small page that is
  already split off, else from a free expert page split into small pages, else from a huge page
  split into expert pages (never a huge page cut straight into small pages); pages of one
  request are taken from the same split page where possible, so that they are freed together.
* reclamation merges upward: when every small page of a split expert page is free it is an
  expert page again; when every page under a huge page is free the huge page returns.

Readings where the section is silent (listed with reasons in the design notes): a split page
holds small pages of one kind and a huge page middle pages of one kind; small page sizes divide
the expert page; ties go to the lowest byte offset; "already split" small pages are taken
first from split pages holding the same request's pages, then from any split page.
"""
from __future__ import annotations

import math

EXPERT, SSM, KV, CONV = 0, 1, 2, 3


class TiersOracle:
    def __init__(self, pool_bytes, expert_page, ssm_page=0, kv_page=0, conv_page=0):
        assert (kv_page == 0 or expert_page % kv_page == 0) and (conv_page == 0 or expert_page % conv_page == 0)
        self.size = {EXPERT: expert_page, SSM: ssm_page, KV: kv_page, CONV: conv_page}
        self.huge = math.lcm(expert_page, ssm_page) if ssm_page else expert_page
        # every huge page: None (whole and free) or {"kind": EXPERT|SSM, "pages": {offset: state}}
        # where a middle page's state is "free", "live" or a list of small-page owners (split;
        # None for a free slot)
        self.pages = [None] * (pool_bytes // self.huge)

    # -- middle pages ------------------------------------------------------------------------
    def _free_middle(self, kind):
        found = []
        for h, hp in enumerate(self.pages):
            if hp is not None and hp["kind"] == kind:
                found += [off for off, st in hp["pages"].items() if st == "free"]
        return sorted(found)

    def _take_middle(self, kind):
        free = self._free_middle(kind)
        if not free:
            whole = [h for h, hp in enumerate(self.pages) if hp is None]
            if not whole:
                return None
            h = whole[0]
            step = self.size[kind]
            self.pages[h] = {"kind": kind,
                             "pages": {h * self.huge + i * step: "free" for i in range(self.huge // step)}}
            free = self._free_middle(kind)
        off = free[0]
        self._huge_of(off)["pages"][off] = "live"
        return off

    def _huge_of(self, off):
        return self.pages[off // self.huge]

    def _give_middle(self, off):
        hp = self._huge_of(off)
        hp["pages"][off] = "free"
        if all(st == "free" for st in hp["pages"].values()):
            self.pages[off // self.huge] = None          # the huge page is whole again

    # -- the calls ---------------------------------------------------------------------------
    def alloc(self, kind, owner=0):
        if kind in (EXPERT, SSM):
            return self._take_middle(kind)
        step = self.size[kind]
        split = []   # (offset of the split page, its owners list)
        for hp in self.pages:
            if hp is not None and hp["kind"] == EXPERT:
                for off, st in sorted(hp["pages"].items()):
                    if isinstance(st, dict) and st["kind"] == kind and None in st["owners"]:
                        split.append((off, st))
        same = [(off, st) for off, st in split if owner in st["owners"]]
        pick = same[0] if same else (split[0] if split else None)
        if pick is None:
            e = self._take_middle(EXPERT)
            if e is None:
                return None
            st = {"kind": kind, "owners": [None] * (self.size[EXPERT] // step)}
            self._huge_of(e)["pages"][e] = st
            pick = (e, st)
        off, st = pick
        slot = st["owners"].index(None)
        st["owners"][slot] = owner
        return off + slot * step

    def free(self, kind, off):
        if kind in (EXPERT, SSM):
            hp = self._huge_of(off)
            assert hp is not None and hp["kind"] == kind and hp["pages"].get(off) == "live"
            self._give_middle(off)
            return
        e = off - off % self.size[EXPERT]
        st = self._huge_of(e)["pages"][e]
        slot = (off - e) // self.size[kind]
        assert isinstance(st, dict) and st["kind"] == kind and st["owners"][slot] is not None
        st["owners"][slot] = None
        if all(o is None for o in st["owners"]):
            self._huge_of(e)["pages"][e] = "live"         # an expert page again ...
            self._give_middle(e)                          # ... and back among the free ones

    def stats(self):
        c = [self.huge, 0, 0, 0, 0, 0, 0, 0]
        for hp in self.pages:
            if hp is None:
                c[1] += 1
                continue
            for st in hp["pages"].values():
                if st == "free":
                    c[2 + hp["kind"]] += 1
                elif st == "live":
                    c[4 + hp["kind"]] += 1
                else:
                    c[6] += 1
                    c[7] += st["owners"].count(None)
        return c

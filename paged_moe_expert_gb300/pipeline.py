"""Multi-layer decode executor with double-buffered expert prefetch.

Rimuru (paper-daily.com/en), "Expert weights are scattered across pages. How does the kernel read
them?": two loading buffers alternate -- while one supplies this layer's experts, the other
receives the experts prefetched for the next layer, and the roles swap at the next layer; the
buffer holds at most expert_offload_limit experts.  "The adjuster...": copies finish before the
page table points at them, and a location is reused only after the forward that reads it ends.
FluxMoE (awesome-system-papers, "核心方法") states the same two hazards as RAW (compute after the
copy) and WAR (copy after the last reader), ordered by events between a loading stream and the
compute stream.

`DecodeStack` runs L layers of one MoE shape.  Layer l keeps its resident experts in pool pages
(cycling over a few pre-placed pool layouts, one per step, to mimic pages moving between steps);
its offloaded experts live in pinned host memory (or, with the compressed backend, as
exponent-Huffman blobs in device memory that libpmoe's decoder expands) and are brought into load
buffer l % 2 on a side stream one layer ahead of compute:

    iteration l:  copy stream: wait free[(l+1)%2]  -> copy layer l+1's experts -> record ready[(l+1)%2]
                  compute:     wait ready[l%2]      -> forward layer l            -> record free[l%2]

`ElasticDecodeStack` puts all layers on ONE page pool shared with the KV cache and lets the
adjuster (libpmoe's native `pmoe_adjuster_*`) decide each round which experts stay ("The
adjuster..."): KV pages are lent out of the free pages first, a remaining shortfall R_b makes the
adjuster evict, surplus free pages make it add; added experts are copied into their reserved
pages on a fill stream and a layer's page table points at them only after that copy; evicted
experts keep their pages until the round's forward pass has ended.  `KVPages` gives KV cache pages
finer than an expert page ("One pool for data whose sizes differ by orders of magnitude"): the
three-tier allocator carves them out of expert pages the adjuster lends, and
`ElasticDecodeStack.round_requests` runs a round with KV pages per request.

Only host bookkeeping lives here (which experts, which slots, which events); every copy is one
cudaMemcpyAsync or decode launch issued by libpmoe and every step of the layer runs in its kernels.
"""
from __future__ import annotations

import numpy as np
import torch

import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300.adjuster import Adjuster
from paged_moe_expert_gb300 import synthetic as syn


def routed_experts(logits: np.ndarray, k: int) -> np.ndarray:
    """Experts some token routes to (top-k on the logits, ties to the lower id) -- the set the
    prefetch must bring in; host-side bookkeeping for the copy list."""
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    return np.unique(order)


class DecodeStack:
    """backend "host": offloaded experts live in pinned host memory and are copied in;
    "compressed": they live in device memory as exponent-Huffman blobs (FluxMoE's compressed GPU
    backend) and are decoded into the load buffer on the copy stream instead."""

    def __init__(self, cfg, weights, n_layers: int, n_offload: int, layouts: int = 4,
                 device="cuda", seed: int = 0, backend: str = "host"):
        E, S, f, d = cfg.E, cfg.S, cfg.f, cfg.d
        self.cfg, self.L, self.n_off, self.layouts = cfg, n_layers, n_offload, layouts
        self.device = device
        rng = np.random.default_rng(seed)
        page = f * d
        src = pl.contiguous_weights(cfg, weights, device)     # expert e: pages 3e..3e+2
        self.slots = max(1, n_offload)
        self.desc = pm.make_desc(d, f, E, cfg.k, cfg.renormalize, S, self.slots)
        self.bufs = pl.new_load_buffers(self.slots, f, d, device)
        P = 3 * (E + S)
        self.offloaded = []          # per layer: sorted array of offloaded routed experts
        self.plans = []              # [layer][layout]
        self.tables = []             # [layer][layout] page_table (device)
        self.pools = []
        for l in range(n_layers):
            off = np.sort(rng.permutation(E)[:n_offload]).astype(np.int64)
            self.offloaded.append(off)
            row_plans, row_tables = [], []
            for j in range(layouts):
                perm = rng.permutation(P).astype(np.int32)
                pt = np.full((E + S, 3), -1, np.int32)
                pool_t = pl.new_pool(P, f, d, device)
                nxt = 0
                for e in range(E + S):
                    if e < E and e in set(off.tolist()):
                        continue
                    for m in range(3):
                        p = int(perm[nxt]); nxt += 1
                        pt[e, m] = p
                        pool_t[p * page:(p + 1) * page].copy_(src[(3 * e + m) * page:(3 * e + m + 1) * page])
                self.pools.append(pool_t)
                row_plans.append(pm.Plan(self.desc, pool_t, P, self.bufs))
                row_tables.append(torch.from_numpy(pt).to(device))
            self.plans.append(row_plans)
            self.tables.append(row_tables)
        del src
        # pinned host copies of every routed expert (W1 | W3 | W2), shared by all layers
        if backend not in ("host", "compressed"):
            raise ValueError("backend must be 'host' or 'compressed'")
        self.backend = backend
        self.host = None
        if backend == "host":
            self.host = [torch.from_numpy(pl.pack_expert(weights, e, E, f).view(np.int16)).pin_memory()
                         for e in range(E)]
        self.blobs = None
        if backend == "compressed":
            from paged_moe_expert_gb300 import expcodec
            self.blobs = [[torch.from_numpy(expcodec.encode(m)).to(device)
                           for m in pl.expert_matrices(weights, e, E, f)] for e in range(E)]
            self.compressed_bytes = sum(b.numel() for row in self.blobs for b in row)
        self.copy_stream = torch.cuda.Stream(device=device)
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [torch.cuda.Event() for _ in range(2)]
        # copy-in of experts a prediction missed: device-readable addresses of the pinned host
        # copies, and per layer the list of what the last step copied in
        self.host_table = pm.device_pointers(self.host) if self.host is not None else None
        self.missed = [torch.zeros(1 + 2 * E, dtype=torch.int32, device=device) for _ in range(n_layers)]

    # -- bookkeeping --------------------------------------------------------------------------
    def schedule(self, logits_np):
        """For one step (logits_np[l] = [T, E] of layer l): which offloaded experts each layer
        needs, their slots, and the buf_slot table (device) that points them at buffer l % 2."""
        E = self.cfg.E
        sched = []
        for l in range(self.L):
            need = np.intersect1d(routed_experts(logits_np[l], self.cfg.k), self.offloaded[l])
            bs = np.full(E, -1, np.int32)
            slots = np.arange(len(need), dtype=np.int32)
            bs[need] = (l % 2) * self.slots + slots
            sched.append((need, slots, torch.from_numpy(bs).to(self.device)))
        return sched

    def schedule_predicted(self, predicted):
        """For one step from a prediction (predicted[l] = experts expected at layer l, e.g. the
        previous step's routing) instead of the actual routing: the predicted offloaded experts are
        prefetched into buffer l % 2, every other offloaded expert is marked absent (-2), and the
        copy-in step before the layer brings in whatever the actual routing adds (Rimuru, "The
        pipeline...": predicted experts join the prefetch queue, actual routing decides)."""
        E = self.cfg.E
        sched = []
        for l in range(self.L):
            need = np.intersect1d(np.asarray(predicted[l], dtype=np.int64), self.offloaded[l])[:self.slots]
            bs = np.full(E, -1, np.int32)
            bs[self.offloaded[l]] = -2
            slots = np.arange(len(need), dtype=np.int32)
            bs[need] = (l % 2) * self.slots + slots
            sched.append((need, slots, torch.from_numpy(bs).to(self.device)))
        return sched

    def prefetch(self, l, sched_l):
        need, slots, _ = sched_l
        b = l % 2
        if self.backend == "host":
            pm.prefetch_async(self.plans[l][0], b, [self.host[int(e)] for e in need], slots,
                              self.copy_stream, buf_free=self.free[b], copy_done=self.ready[b])
            return
        from paged_moe_expert_gb300 import expcodec
        page = self.cfg.f * self.cfg.d
        if self.free[b].cuda_event != 0:
            self.copy_stream.wait_event(self.free[b])          # WAR: the buffer's last reader
        src, dst = [], []
        for e, s_ in zip(need, slots):
            for j in range(3):
                src.append(self.blobs[int(e)][j])
                dst.append(self.bufs[b][(3 * int(s_) + j) * page:(3 * int(s_) + j + 1) * page])
        for i in range(0, len(src), 128):
            expcodec.decode_async(src[i:i + 128], page, dst[i:i + 128], stream=self.copy_stream)
        self.ready[b].record(self.copy_stream)                 # RAW: compute waits for it

    # -- one step -----------------------------------------------------------------------------
    def step(self, x0, logits_dev, sched, step_idx, acts, ws, first_prefetched=False,
             copy_in=False, stall_events=None):
        """Run all layers on x0 ([T, d] bf16); layer l reads logits_dev[l].  The copy for layer 0
        is issued here unless the previous step already issued it (first_prefetched).  With
        copy_in (a schedule from schedule_predicted), each layer first copies in the routed
        experts the prediction missed, on the compute stream; stall_events[l] = (before, after)
        bracket that step.  Returns the last layer's output tensor (one of `acts`)."""
        cur = torch.cuda.current_stream()
        j = step_idx % self.layouts
        if not first_prefetched:
            self.prefetch(0, sched[0])
        x = x0
        for l in range(self.L):
            if l + 1 < self.L:
                self.prefetch(l + 1, sched[l + 1])          # overlaps layer l's compute
            cur.wait_event(self.ready[l % 2])                # RAW
            if copy_in:
                if stall_events is not None:
                    stall_events[l][0].record(cur)
                pm.copy_in_missing(self.plans[l][j], logits_dev[l], sched[l][2], l % 2,
                                   self.host_table, self.missed[l], stream=cur)
                if stall_events is not None:
                    stall_events[l][1].record(cur)
            out = acts[l % 2]
            self.plans[l][j].forward(x, logits_dev[l], self.tables[l][j], sched[l][2], out=out,
                                     workspace=ws)
            self.free[l % 2].record(cur)                     # WAR
            x = out
        return x


def kv_round(held: int, need: int, free: int):
    """One round of KV cache pages in the unified pool: (pages to take from the free pages,
    pages to give back, R_b = pages still missing).  The scheduler's KV allocation comes before
    the adjuster, which sees the free pages left after it and the shortfall."""
    if need <= held:
        return 0, held - need, 0
    take = min(free, need - held)
    return take, 0, need - held - take


class KVPages:
    """KV cache pages of the unified pool (Rimuru, "One pool for data whose sizes differ by orders
    of magnitude"): small pages carved by the three-tier allocator out of expert pages that the
    adjuster lends, one request's pages kept on the same expert pages where possible; an expert
    page whose KV pages are all free goes straight back to the adjuster.  Offsets are bytes from
    the start of the adjuster's pages."""

    def __init__(self, adj: Adjuster, expert_pages: int, page_bytes: int, kv_page_bytes: int):
        from paged_moe_expert_gb300 import tiers
        self._tiers = tiers
        self.t = tiers.Tiers(expert_pages * page_bytes, page_bytes, 0, kv_page_bytes, 0)
        # every page starts on the expert side: held by the tiers as a live expert page until the
        # adjuster lends it
        for p in range(expert_pages):
            if self.t.alloc(tiers.EXPERT) != p * page_bytes:
                raise RuntimeError("unexpected page order")
        self.adj, self.page, self.kv = adj, page_bytes, kv_page_bytes
        self.per_page = page_bytes // kv_page_bytes
        self.req = {}                  # request -> its KV page offsets

    def allocate(self, rid: int, n: int) -> int:
        """n more KV pages for request rid; returns how many could not be placed."""
        T = self._tiers
        got = self.req.setdefault(int(rid), [])
        for i in range(n):
            off = self.t.alloc(T.KV, int(rid))
            if off is None and self.adj.free_pages() > 0:
                p = int(self.adj.lend(1)[0])            # one more expert page turns to KV
                self.t.free(T.EXPERT, p * self.page)
                off = self.t.alloc(T.KV, int(rid))
            if off is None:
                return n - i
            got.append(off)
        return 0

    def release(self, rid: int):
        T = self._tiers
        for off in self.req.pop(int(rid), []):
            self.t.free(T.KV, off)
        c = self.t.stats()
        for _ in range(c[1] + c[2]):                   # whole free pages back to the adjuster
            off = self.t.alloc(T.EXPERT)
            self.adj.give_back([off // self.page])

    def live(self):
        return {r: list(v) for r, v in self.req.items()}


class ElasticDecodeStack:
    """L layers of one MoE shape over one page pool: pages [0, 3*S*L) hold the layers' shared
    chunks (always resident), pages base + [0, expert_pages) are the adjuster's, shared between
    routed experts and lent KV cache pages.  All layers carry the same weights (one synthetic
    set, pinned on the host once).  probs[l][e] is the offline routing probability the ranking
    comes from; cached[l] experts of layer l start resident."""

    def __init__(self, cfg, weights, n_layers: int, probs, cached, offload_limit: int,
                 expert_pages: int, device="cuda", backend: str = "host"):
        E, S, f, d = cfg.E, cfg.S, cfg.f, cfg.d
        self.cfg, self.L, self.device = cfg, n_layers, device
        self.base = 3 * S * n_layers
        num_pages = self.base + expert_pages
        self.pool = pl.new_pool(num_pages, f, d, device)
        # a layer offloads at most offload_limit experts, so each load buffer needs that many slots
        self.slots = max(1, int(offload_limit))
        self.desc = pm.make_desc(d, f, E, cfg.k, cfg.renormalize, S, self.slots)
        self.bufs = pl.new_load_buffers(self.slots, f, d, device)
        self.plan = pm.Plan(self.desc, self.pool, num_pages, self.bufs)
        self.adj = Adjuster(probs, cached, offload_limit, expert_pages)
        if (E - self.adj.cached() > self.slots).any():
            raise ValueError("a layer starts with more offloaded experts than offload_limit")
        self.host = [torch.from_numpy(pl.pack_expert(weights, e, E, f).view(np.int16)).pin_memory()
                     for e in range(E + S)]
        # "compressed": the routed experts' pages also live in device memory as exponent-Huffman
        # blobs, and both the streamed experts and the experts the adjuster adds are decoded from
        # them instead of copied from the host
        if backend not in ("host", "compressed"):
            raise ValueError("backend must be 'host' or 'compressed'")
        self.backend = backend
        self.blobs = None
        if backend == "compressed":
            from paged_moe_expert_gb300 import expcodec
            self.blobs = [[torch.from_numpy(expcodec.encode(m)).to(device)
                           for m in pl.expert_matrices(weights, e, E, f)] for e in range(E)]
        self.copy_stream = torch.cuda.Stream(device=device)
        self.fill_stream = torch.cuda.Stream(device=device)
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [torch.cuda.Event() for _ in range(2)]
        self.fill_done = [torch.cuda.Event() for _ in range(n_layers)]
        self.fwd_done = torch.cuda.Event()
        self.kv = []                                  # pages lent to the KV cache
        self.filling = [False] * n_layers
        self.filled_experts = 0
        # initial placement: shared chunks and the cached experts, straight into their pages
        hs, pg = [], []
        for l in range(n_layers):
            for s_ in range(S):
                hs.append(self.host[E + s_])
                pg.append([3 * (l * S + s_) + j for j in range(3)])
            pt = self.adj.page_table(l)
            for e in np.nonzero(pt[:, 0] >= 0)[0]:
                hs.append(self.host[int(e)])
                pg.append((pt[e] + self.base).tolist())
        pm.fill_pages_async(self.plan, hs, pg, self.fill_stream)
        self.fill_stream.synchronize()
        self.tables = [torch.empty((E + S, 3), dtype=torch.int32, device=device)
                       for _ in range(n_layers)]
        self.table_host = [torch.empty((E + S, 3), dtype=torch.int32).pin_memory()
                           for _ in range(n_layers)]
        self.uploaded = [None] * n_layers
        self.upload_done = [torch.cuda.Event() for _ in range(n_layers)]
        for l in range(n_layers):
            self.tables[l].copy_(torch.from_numpy(self.table_np(l)))
            self.uploaded[l] = self.table_np(l)

    # -- bookkeeping --------------------------------------------------------------------------
    def table_np(self, l):
        """Layer l's page_table [E+S][3] as the kernels must see it now."""
        E, S = self.cfg.E, self.cfg.S
        pt = self.adj.page_table(l)
        out = np.full((E + S, 3), -1, np.int32)
        has = pt[:, 0] >= 0
        out[:E][has] = pt[has] + self.base
        for s_ in range(S):
            out[E + s_] = [3 * (l * S + s_) + j for j in range(3)]
        return out

    def round(self, kv_need: int):
        """The round before a step, KV counted in whole expert pages: KV pages first, then the
        adjuster on what is left.  Returns (change records, R_b)."""
        take, back, short = kv_round(len(self.kv), int(kv_need), self.adj.free_pages())
        if back:
            self.adj.give_back(self.kv[-back:])
            del self.kv[-back:]
        if take:
            self.kv += self.adj.lend(take).tolist()
        changes = self.adj.decide(short)
        self._fill_adds(changes)
        return changes, short

    def round_requests(self, kv: "KVPages", arrivals, departures):
        """The round before a step with KV pages per request: finished requests give their pages
        back, then new ones ({request: KV pages}) are placed; the expert pages still missing are
        R_b for the adjuster, and the requests that did not fit are returned to be retried."""
        for rid in departures:
            kv.release(rid)
        waiting, short_kv = {}, 0
        for rid, n in arrivals.items():
            miss = kv.allocate(rid, n)
            if miss:
                waiting[rid] = miss
                short_kv += miss
        short = -(-short_kv // kv.per_page)                  # in expert pages
        changes = self.adj.decide(short)
        self._fill_adds(changes)
        return changes, short, waiting

    def _fill_adds(self, changes):
        """Added experts start copying into their reserved pages at once, after the previous
        forward pass (whose evictions may have freed those pages)."""
        self.filling = [False] * self.L
        adds = changes[changes[:, 0] == 1]
        for l in np.unique(adds[:, 1]) if len(adds) else []:
            mine = adds[adds[:, 1] == l]
            pages = (mine[:, 3:6] + self.base).tolist()
            if self.backend == "host":
                pm.fill_pages_async(self.plan, [self.host[int(e)] for e in mine[:, 2]], pages,
                                    self.fill_stream, after=self.fwd_done,
                                    copy_done=self.fill_done[int(l)])
            else:
                from paged_moe_expert_gb300 import expcodec
                page = self.cfg.f * self.cfg.d
                if self.fwd_done.cuda_event != 0:
                    self.fill_stream.wait_event(self.fwd_done)   # the pages' last reader
                src = [self.blobs[int(e)][j] for e in mine[:, 2] for j in range(3)]
                dst = [self.pool[p * page:(p + 1) * page] for row in pages for p in row]
                for i in range(0, len(src), 128):
                    expcodec.decode_async(src[i:i + 128], page, dst[i:i + 128], stream=self.fill_stream)
                self.fill_done[int(l)].record(self.fill_stream)
            self.filling[int(l)] = True
            self.filled_experts += len(mine)

    def resident(self, l):
        return self.adj.page_table(l)[:, 0] >= 0

    def schedule(self, logits_np):
        """Per layer: the routed experts without pages this round, their slots in buffer l % 2
        and the buf_slot table (device)."""
        E = self.cfg.E
        sched = []
        for l in range(self.L):
            off = np.nonzero(~self.resident(l))[0]
            need = np.intersect1d(routed_experts(logits_np[l], self.cfg.k), off)
            bs = np.full(E, -1, np.int32)
            slots = np.arange(len(need), dtype=np.int32)
            bs[need] = (l % 2) * self.slots + slots
            sched.append((need, slots, torch.from_numpy(bs).to(self.device)))
        return sched

    def prefetch(self, l, sched_l):
        need, slots, _ = sched_l
        b = l % 2
        if self.backend == "host":
            pm.prefetch_async(self.plan, b, [self.host[int(e)] for e in need], slots,
                              self.copy_stream, buf_free=self.free[b], copy_done=self.ready[b])
            return
        from paged_moe_expert_gb300 import expcodec
        page = self.cfg.f * self.cfg.d
        if self.free[b].cuda_event != 0:
            self.copy_stream.wait_event(self.free[b])
        src = [self.blobs[int(e)][j] for e in need for j in range(3)]
        dst = [self.bufs[b][(3 * int(s_) + j) * page:(3 * int(s_) + j + 1) * page]
               for s_ in slots for j in range(3)]
        for i in range(0, len(src), 128):
            expcodec.decode_async(src[i:i + 128], page, dst[i:i + 128], stream=self.copy_stream)
        self.ready[b].record(self.copy_stream)

    # -- one step -----------------------------------------------------------------------------
    def step(self, x0, logits_dev, sched, acts, ws):
        """All layers on x0 with this round's placement; ends the round's forward pass (the
        adjuster releases evicted experts' pages, to be reused after `fwd_done`)."""
        cur = torch.cuda.current_stream()
        self.prefetch(0, sched[0])
        x = x0
        for l in range(self.L):
            if l + 1 < self.L:
                self.prefetch(l + 1, sched[l + 1])
            if self.filling[l]:
                cur.wait_event(self.fill_done[l])           # copy before the table points there
            t = self.table_np(l)
            if not np.array_equal(t, self.uploaded[l]):
                self.upload_done[l].synchronize()           # the staging copy is free again
                self.table_host[l].numpy()[:] = t
                self.tables[l].copy_(self.table_host[l], non_blocking=True)
                self.upload_done[l].record(cur)
                self.uploaded[l] = t
            cur.wait_event(self.ready[l % 2])
            out = acts[l % 2]
            self.plan.forward(x, logits_dev[l], self.tables[l], sched[l][2], out=out, workspace=ws)
            self.free[l % 2].record(cur)
            x = out
        self.fwd_done.record(cur)
        self.adj.end_forward()
        return x

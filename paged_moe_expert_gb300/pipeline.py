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
its offloaded experts live in pinned host memory and are copied into load buffer l % 2 on a side
stream one layer ahead of compute:

    iteration l:  copy stream: wait free[(l+1)%2]  -> copy layer l+1's experts -> record ready[(l+1)%2]
                  compute:     wait ready[l%2]      -> forward layer l            -> record free[l%2]

Only host bookkeeping lives here (which experts, which slots, which events); every copy is one
cudaMemcpyAsync issued by libpmoe and every step of the layer runs in its kernels.
"""
from __future__ import annotations

import numpy as np
import torch

import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300 import synthetic as syn


def routed_experts(logits: np.ndarray, k: int) -> np.ndarray:
    """Experts some token routes to (top-k on the logits, ties to the lower id) -- the set the
    prefetch must bring in; host-side bookkeeping for the copy list."""
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    return np.unique(order)


class DecodeStack:
    def __init__(self, cfg, weights, n_layers: int, n_offload: int, layouts: int = 4,
                 device="cuda", seed: int = 0):
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
        self.host = [torch.from_numpy(pl.pack_expert(weights, e, E, f).view(np.int16)).pin_memory()
                     for e in range(E)]
        self.copy_stream = torch.cuda.Stream(device=device)
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [torch.cuda.Event() for _ in range(2)]

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

    def prefetch(self, l, sched_l):
        need, slots, _ = sched_l
        b = l % 2
        pm.prefetch_async(self.plans[l][0], b, [self.host[int(e)] for e in need], slots,
                          self.copy_stream, buf_free=self.free[b], copy_done=self.ready[b])

    # -- one step -----------------------------------------------------------------------------
    def step(self, x0, logits_dev, sched, step_idx, acts, ws, first_prefetched=False):
        """Run all layers on x0 ([T, d] bf16); layer l reads logits_dev[l].  The copy for layer 0
        is issued here unless the previous step already issued it (first_prefetched).  Returns
        the last layer's output tensor (one of `acts`)."""
        cur = torch.cuda.current_stream()
        j = step_idx % self.layouts
        if not first_prefetched:
            self.prefetch(0, sched[0])
        x = x0
        for l in range(self.L):
            if l + 1 < self.L:
                self.prefetch(l + 1, sched[l + 1])          # overlaps layer l's compute
            cur.wait_event(self.ready[l % 2])                # RAW
            out = acts[l % 2]
            self.plans[l][j].forward(x, logits_dev[l], self.tables[l][j], sched[l][2], out=out,
                                     workspace=ws)
            self.free[l % 2].record(cur)                     # WAR
            x = out
        return x

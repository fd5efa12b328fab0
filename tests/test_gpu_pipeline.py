"""Multi-layer decode with the double-buffered prefetch (paged_moe_expert_gb300.pipeline): a stack
whose offloaded experts stream from pinned host memory through the two alternating load buffers,
one layer ahead of compute, must give bit-identical outputs to the same stack with every expert
resident in its pool, over several steps and pool layouts; and the chain matches the oracle."""
import numpy as np
import pytest
import torch

import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import pipeline
from paged_moe_expert_gb300 import synthetic as syn

from helpers import assert_close, oracle_layer, out_bits

pytestmark = pytest.mark.gpu


def run(stack, hidden, logits_steps, T):
    ws = pm.alloc_workspace(stack.desc, T)
    acts = [torch.empty_like(hidden) for _ in range(2)]
    outs = []
    for s, lg in enumerate(logits_steps):
        sched = stack.schedule(lg)
        lg_dev = [torch.from_numpy(x).cuda() for x in lg]
        y = stack.step(hidden, lg_dev, sched, s, acts, ws)
        torch.cuda.synchronize()
        outs.append(out_bits(y).copy())
    return outs


@pytest.mark.parametrize("T", [3, 40])
def test_prefetched_stack_equals_resident_stack(T):
    cfg = syn.custom_config("stack", d=256, f=256, E=8, k=2, S=1, n_buffered=0)
    w = syn.make_weights(cfg)
    L, steps = 4, 3
    rng = np.random.default_rng(T)
    hidden_np = syn.to_bf16_bits(rng.standard_normal((T, cfg.d)).astype(np.float32))
    hidden = torch.from_numpy(hidden_np.view(np.int16)).view(torch.bfloat16).cuda()
    logits = [[syn.bf16_bits_to_f32(syn.to_bf16_bits(rng.standard_normal((T, cfg.E)).astype(np.float32)))
               for _ in range(L)] for _ in range(steps)]
    offl = pipeline.DecodeStack(cfg, w, L, n_offload=4, layouts=2, seed=1)
    res = pipeline.DecodeStack(cfg, w, L, n_offload=0, layouts=1, seed=2)
    a = run(offl, hidden, logits, T)
    b = run(res, hidden, logits, T)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # the chain against the oracle (step 0): layer by layer with the GPU's own rounding of h
    ref = hidden_np
    orc = oracle_layer(cfg, w)
    for l in range(L):
        ref = orc.forward(ref, logits[0][l])["out_bf16"]
    assert_close(a[0], ref, "4-layer chain")


@pytest.mark.parametrize("T", [3, 40])
def test_compressed_backend_stack_equals_resident_stack(T):
    """Offloaded experts decoded from exponent-Huffman blobs in device memory into the load
    buffers, one layer ahead of compute, give the resident stack's outputs bit for bit."""
    cfg = syn.custom_config("stackc", d=256, f=256, E=8, k=2, S=1, n_buffered=0)
    w = syn.make_weights(cfg)
    L, steps = 4, 3
    rng = np.random.default_rng(50 + T)
    hidden_np = syn.to_bf16_bits(rng.standard_normal((T, cfg.d)).astype(np.float32))
    hidden = torch.from_numpy(hidden_np.view(np.int16)).view(torch.bfloat16).cuda()
    logits = [[syn.bf16_bits_to_f32(syn.to_bf16_bits(rng.standard_normal((T, cfg.E)).astype(np.float32)))
               for _ in range(L)] for _ in range(steps)]
    comp = pipeline.DecodeStack(cfg, w, L, n_offload=5, layouts=2, seed=4, backend="compressed")
    res = pipeline.DecodeStack(cfg, w, L, n_offload=0, layouts=1, seed=2)
    a = run(comp, hidden, logits, T)
    b = run(res, hidden, logits, T)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert comp.compressed_bytes < 8 * 3 * cfg.f * cfg.d * 2


def test_schedule_points_needed_experts_at_alternating_buffers():
    cfg = syn.custom_config("sched", d=128, f=128, E=8, k=2, S=0, n_buffered=0)
    w = syn.make_weights(cfg)
    st = pipeline.DecodeStack(cfg, w, 3, n_offload=5, layouts=1, seed=3)
    lg = [np.random.default_rng(l).standard_normal((6, 8)).astype(np.float32) for l in range(3)]
    sched = st.schedule(lg)
    for l, (need, slots, bs) in enumerate(sched):
        routed = pipeline.routed_experts(lg[l], 2)
        assert set(need.tolist()) == set(routed.tolist()) & set(st.offloaded[l].tolist())
        bs = bs.cpu().numpy()
        assert (bs[need] // st.slots == l % 2).all()
        assert sorted((bs[need] % st.slots).tolist()) == list(range(len(need)))
        assert (bs[np.setdiff1d(np.arange(8), need)] == -1).all()


@pytest.mark.parametrize("backend", ["host", "compressed"])
def test_elastic_stack_follows_the_adjuster_and_equals_resident_stack(backend):
    """One pool for all layers and the KV cache; a KV demand trace makes the adjuster evict and
    add experts between steps.  Every step's output equals the all-resident stack's, and after
    every step each layer's table points at pages that hold exactly its resident experts."""
    from paged_moe_expert_gb300 import pool as pl
    cfg = syn.custom_config("elastic", d=256, f=256, E=8, k=2, S=1, n_buffered=0)
    w = syn.make_weights(cfg)
    L, T = 4, 24
    rng = np.random.default_rng(7)
    probs = rng.dirichlet(np.full(cfg.E, 0.5), size=L).astype(np.float32)
    cached = [6, 5, 7, 8]
    stack = pipeline.ElasticDecodeStack(cfg, w, L, probs, cached, offload_limit=4,
                                        expert_pages=3 * sum(cached) + 6, backend=backend)
    res = pipeline.DecodeStack(cfg, w, L, n_offload=0, layouts=1, seed=2)
    kv_trace = [0, 9, 30, 30, 0, 0, 12, 40, 0, 0]
    hidden_np = syn.to_bf16_bits(rng.standard_normal((T, cfg.d)).astype(np.float32))
    hidden = torch.from_numpy(hidden_np.view(np.int16)).view(torch.bfloat16).cuda()
    ws = pm.alloc_workspace(stack.desc, T)
    acts = [torch.empty_like(hidden) for _ in range(2)]
    kinds = set()
    for s, need in enumerate(kv_trace):
        lg = [syn.bf16_bits_to_f32(syn.to_bf16_bits(rng.standard_normal((T, cfg.E)).astype(np.float32)))
              for _ in range(L)]
        changes, short = stack.round(need)
        kinds |= set(changes[:, 0].tolist())
        sched = stack.schedule(lg)
        lg_dev = [torch.from_numpy(x).cuda() for x in lg]
        y = stack.step(hidden, lg_dev, sched, acts, ws)
        torch.cuda.synchronize()
        want = run(res, hidden, [lg], T)[0]
        assert np.array_equal(out_bits(y), want), "step %d" % s
        for l in range(L):
            t = stack.tables[l].cpu().numpy()
            assert np.array_equal(t, stack.uploaded[l])
            for e in range(cfg.E + cfg.S):
                if t[e, 0] < 0:
                    continue
                got = pl.read_expert(stack.pool, stack.bufs, t, np.full(cfg.E, -1), e, cfg.f,
                                     cfg.d, stack.slots)
                for g, m in zip(got, pl.expert_matrices(w, e, cfg.E, cfg.f)):
                    assert np.array_equal(g, m), (s, l, e)
    assert kinds == {1, -1}, "the trace must make the adjuster both add and evict"
    assert stack.filled_experts > 0


def test_elastic_stack_with_kv_pages_keeps_kv_and_outputs_intact():
    """KV cache pages carved from lent expert pages (the unified pool) hold what was written to
    them through the memory view while the adjuster evicts and adds experts and the stack runs;
    the outputs stay equal to the all-resident stack's."""
    from paged_moe_expert_gb300 import tiers as tr
    cfg = syn.custom_config("elastic_kv", d=256, f=256, E=8, k=2, S=1, n_buffered=0)
    w = syn.make_weights(cfg)
    L, T = 4, 24
    rng = np.random.default_rng(11)
    probs = rng.dirichlet(np.full(cfg.E, 0.5), size=L).astype(np.float32)
    cached = [6, 5, 7, 8]
    expert_pages = 3 * sum(cached) + 6
    stack = pipeline.ElasticDecodeStack(cfg, w, L, probs, cached, offload_limit=4,
                                        expert_pages=expert_pages)
    page_bytes = cfg.f * cfg.d * 2
    kvb = page_bytes // 8
    kv = pipeline.KVPages(stack.adj, expert_pages, page_bytes, kvb)
    res = pipeline.DecodeStack(cfg, w, L, n_offload=0, layouts=1, seed=2)
    base = stack.base * page_bytes
    hidden_np = syn.to_bf16_bits(rng.standard_normal((T, cfg.d)).astype(np.float32))
    hidden = torch.from_numpy(hidden_np.view(np.int16)).view(torch.bfloat16).cuda()
    ws = pm.alloc_workspace(stack.desc, T)
    acts = [torch.empty_like(hidden) for _ in range(2)]
    sig, active, waiting, nxt, kinds = {}, set(), {}, 0, set()

    def view(o):
        return tr.page_view(stack.pool, base + o, kvb, torch.int16, (kvb // 2,))

    for s_ in range(10):
        departures = [r for r in sorted(active) if rng.random() < 0.35]
        live = kv.live()
        for r in departures:
            active.discard(r)
            for o in live.get(r, []):
                sig.pop(o, None)
        arrivals = dict(waiting)
        for _ in range(int(rng.integers(1, 4))):
            arrivals[nxt] = int(rng.integers(4, 40))
            nxt += 1
        changes, short, waiting = stack.round_requests(kv, arrivals, departures)
        kinds |= set(changes[:, 0].tolist())
        for r, offs in kv.live().items():
            active.add(r)
            for o in offs:
                if o not in sig:
                    sig[o] = (r % 30000) + 1
                    view(o).fill_(sig[o])
        lg = [syn.bf16_bits_to_f32(syn.to_bf16_bits(rng.standard_normal((T, cfg.E)).astype(np.float32)))
              for _ in range(L)]
        sched = stack.schedule(lg)
        y = stack.step(hidden, [torch.from_numpy(x).cuda() for x in lg], sched, acts, ws)
        torch.cuda.synchronize()
        assert np.array_equal(out_bits(y), run(res, hidden, [lg], T)[0]), "step %d" % s_
        for o, v in sig.items():
            t = view(o)
            assert int(t.min()) == v and int(t.max()) == v, (s_, o)
    assert -1 in kinds, "the KV demand must make the adjuster evict"

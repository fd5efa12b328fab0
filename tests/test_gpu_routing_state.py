"""The routing and sort state that the layer forward itself computes, read back from its workspace
after a moe_paged_forward call, against the oracle.

The kernels that route and sort inside a forward call differ by token count and layer shape: the
fused decode kernel routes in every CTA (T <= 32, or 16 for layers of more than 128 experts), the
one-CTA prep routes and sorts small batches with light routing, and above that the routing kernel
runs before the one-CTA or the multi-CTA sort.  Whichever ran, its routing ids, sorted pair list,
block map, inverse map and padded count must equal the oracle's bit for bit, its weights agree to
the expf-vs-libm tolerance, and the structures derived from the sort (the valid rows of each block,
the CTA-pair work units with their page locations, the fused kernel's active slots) must follow
from the oracle's sort exactly.  The comparison rests on the pages' statement that the paged kernel
runs on identical inputs and routing to the contiguous one (Rimuru, paper-daily.com/en, "Expert
weights are scattered across pages. How does the kernel read them?").

The pools hold zeros: the routing and sort state does not depend on the weights, and skipping
the weight generation keeps the full-size shapes quick."""
import numpy as np
import pytest
import torch

import oracle
import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

_LAYERS = {}


def layer(name):
    """Plan over a zero pool and zero load buffers, with the config's placement tables."""
    if name not in _LAYERS:
        _LAYERS.clear()
        torch.cuda.empty_cache()
        cfg = syn.CONFIGS[name]
        plc = syn.make_placement(cfg)
        pool = torch.zeros(cfg.num_pages * cfg.f * cfg.d, dtype=torch.bfloat16, device="cuda")
        bufs = tuple(torch.zeros(cfg.slots_per_buffer * 3 * cfg.f * cfg.d, dtype=torch.bfloat16,
                                 device="cuda") for _ in range(2))
        desc = pm.make_desc(cfg.d, cfg.f, cfg.E, cfg.k, cfg.renormalize, cfg.S, cfg.slots_per_buffer)
        plan = pm.Plan(desc, pool, cfg.num_pages, bufs)
        buf_slot = np.where(plc.buffered, plc.slot_of, -1).astype(np.int32)   # buffer 0
        _LAYERS[name] = dict(cfg=cfg, plc=plc, pool=pool, bufs=bufs, desc=desc, plan=plan,
                             page_table=torch.from_numpy(plc.page_table.copy()).cuda(),
                             buf_slot=torch.from_numpy(buf_slot).cuda(), buf_slot_np=buf_slot)
    return _LAYERS[name]


def tied_logits(T, E, seed):
    """Small integers: most tokens have ties among their top-k candidates."""
    rng = np.random.default_rng(seed)
    return rng.integers(-2, 3, size=(T, E)).astype(np.float32)


def expected_units(block_expert, E, page_table, buf_slot, slots_per_buffer):
    """The CTA-pair work units that follow from a sort: per expert in ascending order, its blocks
    two at a time, then its odd last block, with the expert's W1 and W3 locations packed as
    map << 29 | page (map 0 = pool page, 1 + b = page 3s + j of load buffer b)."""
    def loc(e, j):
        bs = int(buf_slot[e]) if e < E else -1
        if bs >= 0:
            b, s = divmod(bs, slots_per_buffer)
            return ((1 + b) << 29) | (3 * s + j)
        return int(page_table[e, j])
    units = []
    b = 0
    nblk = len(block_expert)
    while b < nblk:
        e = int(block_expert[b])
        nb = 1
        while b + nb < nblk and block_expert[b + nb] == e:
            nb += 1
        for j in range(nb // 2):
            units.append(((b + 2 * j) << 1, e, loc(e, 0), loc(e, 1)))
        if nb % 2:
            units.append((((b + nb - 1) << 1) | 1, e, loc(e, 0), loc(e, 1)))
        b += nb
    return np.array(units, np.int32).reshape(-1, 4)


def run_and_check(name, T, path=pm.PATH_AUTO, logits=None, want_path=None):
    Ly = layer(name)
    cfg, plan = Ly["cfg"], Ly["plan"]
    hidden_np, lg = syn.make_tokens(cfg, T)
    if logits is not None:
        lg = logits
    hidden = torch.from_numpy(hidden_np.view(np.int16)).view(torch.bfloat16).cuda()
    ws = pm.alloc_workspace(Ly["desc"], T)
    ws.fill_(0xA5)   # stale bytes: nothing below may pass by reading what was there before
    plan.set_path(path)
    plan.forward(hidden, torch.from_numpy(lg).cuda(), Ly["page_table"], Ly["buf_slot"], workspace=ws)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    st = plan.routing_state(ws, T)
    if want_path is not None:
        assert st["path"] == want_path
    rids, rw = oracle.route(lg, cfg.k, cfg.renormalize)
    assert np.array_equal(st["ids"], rids), "routing ids differ"
    np.testing.assert_allclose(st["weights"].astype(np.float64), rw, rtol=3e-5, atol=1e-7)
    E, S = cfg.E, cfg.S
    if st["path"] in (pm.PATH_FUSED, pm.PATH_SLICE):
        want = np.concatenate([E + np.arange(S), np.unique(rids)]).astype(np.int32)
        assert np.array_equal(st["active"], want), "active slots differ"
        return st
    bm = st["block_m"]
    ref = oracle.align(rids, E, S, bm)
    assert int(st["meta"][0]) == ref["n_padded"]
    assert np.array_equal(st["sorted_ids"], ref["sorted_ids"]), "sorted pair list differs"
    assert np.array_equal(st["block_expert"], ref["block_expert"]), "block map differs"
    assert np.array_equal(st["inv"], ref["inv"]), "inverse map differs"
    NP = T * (cfg.k + S)
    if "block_rows" in st:
        rows = (ref["sorted_ids"].reshape(-1, bm) != NP).sum(axis=1).astype(np.int32)
        assert np.array_equal(st["block_rows"], rows), "valid rows per block differ"
    if "units" in st:
        want = expected_units(ref["block_expert"], E, Ly["plc"].page_table, Ly["buf_slot_np"],
                              cfg.slots_per_buffer)
        assert np.array_equal(st["units"], want), "CTA-pair work units differ"
        assert int(st["meta"][2]) == int((want[:, 0] & 1).sum())
    return st


TOKENS = [1, 3, 16, 32, 33, 100, 128, 129, 4096]


@pytest.mark.parametrize("T", TOKENS)
@pytest.mark.parametrize("name", ["tiny", "qwen15", "mixtral", "qwen3next"])
def test_forward_routing_state_matches_oracle(name, T):
    """The automatic path of every layer shape at token counts on both sides of each kernel
    boundary (fused / one-CTA prep / routing + one-CTA sort / routing + multi-CTA sort)."""
    run_and_check(name, T)


def test_forward_routing_state_mixtral_8192():
    st = run_and_check("mixtral", 8192, want_path=pm.PATH_TC2)
    assert len(st["units"]) > 0


@pytest.mark.parametrize("name,T,path", [
    ("tiny", 3, pm.PATH_STREAM),        # one-CTA prep, 4-row blocks
    ("tiny", 16, pm.PATH_TC_DECODE),    # one-CTA prep, 16-row blocks
    ("tiny", 100, pm.PATH_TC),          # one-CTA prep, 128-row blocks with valid-row counts
    ("tiny", 100, pm.PATH_TC2),         # one-CTA prep writing CTA-pair units
    ("tiny", 129, pm.PATH_TC2),         # routing kernel + one-CTA sort writing units
    ("tiny", 4096, pm.PATH_TC2),        # routing kernel + multi-CTA sort writing units
    ("qwen15", 16, pm.PATH_STREAM),     # prep with shared chunks
    ("qwen15", 4096, pm.PATH_TC),       # multi-CTA sort with valid-row counts
    ("qwen3next", 1, pm.PATH_TC_DECODE),   # prep with 512 experts (16 logits per lane)
    ("qwen3next", 3, pm.PATH_TC_DECODE),   # routing kernel + one-CTA sort, 512 experts
    ("qwen3next", 64, pm.PATH_TC_DECODE),  # heavy routing: routing kernel + one-CTA sort
    ("qwen3next", 16, pm.PATH_FUSED),
    ("mixtral", 32, pm.PATH_FUSED),
    ("tiny", 3, pm.PATH_SLICE),
    ("qwen15", 8, pm.PATH_SLICE),
    ("qwen15", 16, pm.PATH_SLICE),
    ("qwen3next", 1, pm.PATH_SLICE),
    ("qwen3next", 8, pm.PATH_SLICE),
    ("mixtral", 2048, pm.PATH_TC2),
])
def test_forced_path_routing_state_matches_oracle(name, T, path):
    run_and_check(name, T, path=path, want_path=path)


@pytest.mark.parametrize("T", [1, 16, 33, 129, 4096])
def test_tied_logits_at_512_experts(T):
    """Integer logits over 512 experts: nearly every token's top-10 cuts through a tie, which
    must go to the lower expert id in every routing kernel."""
    cfg = syn.CONFIGS["qwen3next"]
    run_and_check("qwen3next", T, logits=tied_logits(T, cfg.E, 40 + T))


@pytest.mark.parametrize("T", [1, 32, 100, 4096])
def test_tied_logits_few_experts(T):
    cfg = syn.CONFIGS["qwen15"]
    run_and_check("qwen15", T, logits=tied_logits(T, cfg.E, 50 + T))


def test_routing_view_refuses_another_token_count():
    Ly = layer("tiny")
    run_and_check("tiny", 16)
    ws = pm.alloc_workspace(Ly["desc"], 16)
    with pytest.raises(pm.PmoeError) as ei:
        Ly["plan"].routing_state(ws, 15)
    assert ei.value.status == pm._lib.ERR_INVALID_ARG


@pytest.mark.parametrize("T", [1, 2, 5, 8, 16])
@pytest.mark.parametrize("name", ["qwen15", "qwen3next"])
def test_tied_logits_on_the_column_slice_path(name, T):
    """The column-slice kernel's own routing (every CTA routes all tokens) on integer logits,
    where nearly every token's top-k cuts through a tie: the experts chosen must be the oracle's
    (ties to the lower id) bit for bit."""
    cfg = syn.CONFIGS[name]
    run_and_check(name, T, path=pm.PATH_SLICE, logits=tied_logits(T, cfg.E, 70 + T), want_path=pm.PATH_SLICE)

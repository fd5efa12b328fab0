"""GPU parity: every step of the CUDA path, called through the C ABI, against the oracle on the
same seeded inputs.  Integer outputs (routing ids, sorted ids, block map, inverse map, padded
count) must be bit-exact; the layer output must meet the bf16 tolerance in helpers.py; outputs
must be bit-identical wherever the weights live (Rimuru, paper-daily.com/en, "Expert weights
are scattered across pages...": the address rule only relocates rows)."""
import numpy as np
import pytest
import torch

import oracle
import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300 import synthetic as syn

from helpers import assert_close, oracle_layer, out_bits, setup_layer

pytestmark = pytest.mark.gpu


# --------------------------------------------------------------------------------------------
# routing and sort + pad
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k,renorm,ties", [(1, 8, 2, True, False), (37, 60, 4, False, False),
                                                (4096, 512, 10, True, False), (300, 16, 5, True, True),
                                                (129, 512, 10, False, True), (64, 1024, 16, True, False),
                                                (5, 3, 3, False, True), (8192, 8, 2, True, False)])
def test_route_bit_exact(T, E, k, renorm, ties):
    rng = np.random.default_rng(T * 7 + E)
    if ties:
        lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        lg = syn.bf16_bits_to_f32(syn.to_bf16_bits(rng.standard_normal((T, E)).astype(np.float32)))
    ids, w = pm.route(torch.from_numpy(lg).cuda(), k, renorm)
    torch.cuda.synchronize()
    rids, rw = oracle.route(lg, k, renorm)
    assert np.array_equal(ids.cpu().numpy(), rids)
    np.testing.assert_allclose(w.cpu().numpy().astype(np.float64), rw, rtol=3e-5, atol=1e-7)


@pytest.mark.parametrize("multi", [False, True], ids=["one_cta", "multi_cta"])
@pytest.mark.parametrize("T,E,k,S,BM", [(16, 8, 2, 0, 16), (37, 60, 4, 4, 16), (4096, 512, 10, 1, 128),
                                         (4096, 60, 4, 4, 128), (8192, 8, 2, 0, 128), (1, 60, 4, 4, 1),
                                         (0, 8, 2, 1, 16), (33, 3, 3, 2, 4), (1000, 1000, 16, 24, 64),
                                         (30000, 512, 10, 1, 128), (2049, 7, 1, 0, 32), (8192, 8, 2, 0, 256)])
def test_align_bit_exact(T, E, k, S, BM, multi):
    rng = np.random.default_rng(T + 3 * E)
    if T > 5000:   # skewed: a few experts take most pairs
        pop = np.exp(-1.1 * np.log(np.arange(1, E + 1)))
        ids = np.array([rng.choice(E, size=k, replace=False, p=pop / pop.sum()) for _ in range(T)],
                       np.int32).reshape(T, k)
    else:
        ids = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32).reshape(T, k)
    s, b, inv, npad = pm.align(torch.from_numpy(ids).cuda(), E, S, BM, multi_cta=multi)
    torch.cuda.synchronize()
    ref = oracle.align(ids, E, S, BM)
    n = int(npad.item())
    assert n == ref["n_padded"]
    assert np.array_equal(s[:n].cpu().numpy(), ref["sorted_ids"])
    assert np.array_equal(b[:n // BM].cpu().numpy(), ref["block_expert"])
    if T:
        assert np.array_equal(inv.cpu().numpy(), ref["inv"])


# --------------------------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------------------------

SMALL = [
    syn.CONFIGS["tiny"],
    syn.custom_config("ragged", d=192, f=256, E=5, k=3, S=2, renormalize=False, n_buffered=2),
    syn.custom_config("one_expert", d=64, f=128, E=1, k=1, S=0, n_buffered=0, slots_per_buffer=1),
    syn.custom_config("wide_k", d=320, f=384, E=16, k=16, S=1, n_buffered=5),
]


PATHS = [pm.PATH_STREAM, pm.PATH_TC, pm.PATH_TC_DECODE, pm.PATH_TC2, pm.PATH_FUSED, pm.PATH_SLICE]
PATH_IDS = ["stream", "tc", "tc_decode", "tc2", "fused", "slice"]
FUSED_MAX_T = 32
SLICE_MAX_T = 16
DECODE_PATHS = (pm.PATH_FUSED, pm.PATH_SLICE)   # no sort: active slots instead


def serves(path, T):
    return not ((path == pm.PATH_FUSED and T > FUSED_MAX_T) or (path == pm.PATH_SLICE and T > SLICE_MAX_T))


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("T", [1, 3, 16, 17, 32, 37, 128, 300])
def test_forward_matches_oracle(cfg, T, path):
    if not serves(path, T):
        pytest.skip("the decode kernels take at most 32 (fused) or 16 (column-slice) tokens")
    if path != pm.PATH_FUSED and T in (17, 32):
        pytest.skip("token counts that only change the fused kernel's tile width")
    L = setup_layer(cfg, T)
    L.plan.set_path(path)
    out = L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)
    torch.cuda.synchronize()
    assert L.plan.device_error() == 0
    assert L.plan.last_run()[0] == path
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np, L.logits_np)
    assert_close(out_bits(out), ref["out_bf16"], "%s T=%d" % (cfg.name, T))


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
def test_output_independent_of_placement(path):
    cfg = syn.custom_config("inv", d=256, f=256, E=12, k=3, S=1, n_buffered=4, slots_per_buffer=6,
                            num_pages=60)
    w = syn.make_weights(cfg)
    T = 13 if path == pm.PATH_SLICE else 29   # every path serves it
    outs = []
    for pseed, bidx, nb in [(1, 0, 4), (2, 0, 4), (3, 1, 4), (4, 1, 6), (5, 0, 0)]:
        L = setup_layer(cfg, T, placement_seed=pseed, buffer_index=bidx, n_buffered=nb, weights=w)
        L.plan.set_path(path)
        outs.append(out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)))
        assert L.plan.device_error() == 0
    # contiguous twin, same inputs and routing
    cw = pl.contiguous_weights(cfg, w)
    cplan = pm.Plan(L.desc, cw, 3 * (cfg.E + cfg.S))
    cplan.set_path(path)
    outs.append(out_bits(cplan.contig_forward(L.hidden, L.logits)))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    ref = oracle_layer(cfg, w).forward(L.hidden_np, L.logits_np)
    assert_close(outs[0], ref["out_bf16"])


@pytest.mark.parametrize("T", [16, 4])   # the fused and the column-slice decode kernels
def test_bad_page_sets_device_error(T):
    cfg = syn.CONFIGS["tiny"]
    L = setup_layer(cfg, T)
    pt = L.page_table.clone()
    ids, _ = oracle.route(L.logits_np, cfg.k, cfg.renormalize)
    e = int(next(x for x in ids.reshape(-1) if not L.placement.buffered[x]))
    pt[e, 1] = cfg.num_pages          # one past the end
    L.plan.forward(L.hidden, L.logits, pt, L.buf_slot)
    assert L.plan.device_error() == pm._lib.ERR_PAGE_OOB
    assert L.plan.device_error() == 0   # cleared by the previous read
    bs = L.buf_slot.clone()
    bs[e] = 2 * cfg.slots_per_buffer    # past both buffers
    L.plan.forward(L.hidden, L.logits, L.page_table, bs)
    assert L.plan.device_error() == pm._lib.ERR_SLOT_OOB


def test_invalid_arguments_rejected():
    cfg = syn.CONFIGS["tiny"]
    L = setup_layer(cfg, 4)
    with pytest.raises(pm.PmoeError) as ei:
        L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot,
                       workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == pm._lib.ERR_WORKSPACE
    with pytest.raises(pm.PmoeError):
        pm.Plan(pm.make_desc(100, 128, 8, 2, True), L.pool, 32)   # d not a multiple of 64


def test_auto_path_by_token_count():
    cfg = syn.CONFIGS["tiny"]
    # up to 16 tokens the column-slice kernel (tiny: one column tile per CTA at most), up to 32 the
    # fused decode kernel; then by T*k/E (tiny: E=8, k=2 -> T/4): small-batch kernels up to T=96,
    # single-CTA blocks below T=256, pairs from T=256
    for T, want in [(1, pm.PATH_SLICE), (8, pm.PATH_SLICE), (16, pm.PATH_SLICE), (17, pm.PATH_FUSED),
                    (32, pm.PATH_FUSED),
                    (33, pm.PATH_TC_DECODE), (96, pm.PATH_TC_DECODE), (97, pm.PATH_TC),
                    (255, pm.PATH_TC), (256, pm.PATH_TC2), (4096, pm.PATH_TC2)]:
        L = setup_layer(cfg, T)
        L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)
        assert L.plan.last_run()[0] == want


def test_auto_path_small_batch_token_cap():
    """Many experts: T*k/E stays small far past 320 tokens, but from 321 tokens the automatic path
    takes 128-token blocks (layers of more than 128 experts never take CTA pairs)."""
    cfg = syn.custom_config("e256", d=256, f=128, E=256, k=2)
    for T, want in [(320, pm.PATH_TC_DECODE), (321, pm.PATH_TC)]:
        L = setup_layer(cfg, T)
        L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)
        assert L.plan.last_run()[0] == want


@pytest.mark.parametrize("T", [16, 300])
def test_paths_agree(T):
    cfg = syn.custom_config("agree", d=256, f=256, E=6, k=2, S=1, n_buffered=2)
    L = setup_layer(cfg, T)
    outs = []
    for path in PATHS:
        if not serves(path, T):
            continue
        L.plan.set_path(path)
        outs.append(out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)))
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np, L.logits_np)
    for o in outs:
        assert_close(o, ref["out_bf16"])


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
def test_forward_replays_from_a_cuda_graph(path):
    cfg = syn.custom_config("graph", d=256, f=256, E=6, k=2, S=1, n_buffered=2)
    T = {pm.PATH_FUSED: 24, pm.PATH_SLICE: 6}.get(path, 40)
    L = setup_layer(cfg, T)
    L.plan.set_path(path)
    ws = pm.alloc_workspace(L.desc, T)
    out = torch.empty_like(L.hidden)
    run = lambda: L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot, out=out, workspace=ws)  # noqa: E731
    run()
    torch.cuda.synchronize()
    eager = out_bits(out)
    out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(out), eager)


def test_fused_rejects_more_than_32_tokens():
    cfg = syn.CONFIGS["tiny"]
    L = setup_layer(cfg, 33)
    L.plan.set_path(pm.PATH_FUSED)
    with pytest.raises(pm.PmoeError) as ei:
        L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)
    assert ei.value.status == pm._lib.ERR_UNSUPPORTED


def test_fused_back_to_back_calls_reuse_the_grid_barrier():
    """Many fused calls in a row on one stream (each passes three grid barriers through the plan's
    words) stay bit-identical, with no error raised."""
    cfg = syn.custom_config("repeat", d=256, f=384, E=16, k=4, S=2, n_buffered=3)
    L = setup_layer(cfg, 9)
    L.plan.set_path(pm.PATH_FUSED)
    ws = pm.alloc_workspace(L.desc, 9)
    outs = [torch.empty_like(L.hidden) for _ in range(20)]
    for o in outs:
        L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot, out=o, workspace=ws)
    torch.cuda.synchronize()
    assert L.plan.device_error() == 0
    first = out_bits(outs[0])
    for o in outs[1:]:
        assert np.array_equal(out_bits(o), first)
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np, L.logits_np)
    assert_close(first, ref["out_bf16"])


def test_fused_calls_with_changing_token_counts_share_one_plan():
    """One plan serves fused calls of different token counts in turn (1, 16, 5, 1, 32, 1): the
    grid barrier's per-CTA words stay in step across them, no call times out, and each output
    matches the oracle."""
    cfg = syn.custom_config("mixT", d=256, f=384, E=16, k=4, S=2, n_buffered=3)
    L = setup_layer(cfg, 32)
    L.plan.set_path(pm.PATH_FUSED)
    orc = oracle_layer(cfg, L.w)
    ws = pm.alloc_workspace(L.desc, 32)
    for T in (1, 16, 5, 1, 32, 1):
        h, lg = syn.make_tokens(cfg, T)
        out = L.plan.forward(pl._bf16(h).cuda(), torch.from_numpy(lg).cuda(), L.page_table,
                             L.buf_slot, workspace=ws)
        torch.cuda.synchronize()
        assert L.plan.device_error() == 0, "T=%d" % T
        assert_close(out_bits(out), orc.forward(h, lg)["out_bf16"], "T=%d" % T)


def test_pair_path_back_to_back_calls_are_identical():
    """Many CTA-pair calls in a row on one workspace, with more tiles than CTA pairs and odd
    blocks (M=128 units), stay bit-identical and match the oracle."""
    cfg = syn.custom_config("pairs", d=256, f=384, E=12, k=3, S=2, n_buffered=3)
    T = 700
    L = setup_layer(cfg, T)
    L.plan.set_path(pm.PATH_TC2)
    ws = pm.alloc_workspace(L.desc, T)
    outs = [torch.empty_like(L.hidden) for _ in range(8)]
    for o in outs:
        L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot, out=o, workspace=ws)
    torch.cuda.synchronize()
    assert L.plan.device_error() == 0
    assert L.plan.last_run()[0] == pm.PATH_TC2
    first = out_bits(outs[0])
    for o in outs[1:]:
        assert np.array_equal(out_bits(o), first)
    rows = np.arange(0, T, 37)
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np[rows], L.logits_np[rows])
    assert_close(first[rows], ref["out_bf16"])


def test_pair_path_with_experts_larger_than_l2_share():
    """Experts whose gate/up and down matrices each exceed a quarter of L2 switch the CTA-pair
    GEMMs to the expert-major tile order (N tile by N tile, the expert's units innermost).  Its
    output matches the oracle, is bit-identical to the contiguous twin, and the routing state is
    unchanged by the order."""
    cfg = syn.custom_config("bigexp", d=2048, f=8704, E=4, k=2, S=0, n_buffered=1, slots_per_buffer=1)
    T = 1500
    L = setup_layer(cfg, T)
    L.plan.set_path(pm.PATH_TC2)
    ws = pm.alloc_workspace(L.desc, T)
    out = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot, workspace=ws))
    assert L.plan.device_error() == 0
    st = L.plan.routing_state(ws, T)
    rids, _ = oracle.route(L.logits_np, cfg.k, cfg.renormalize)
    assert np.array_equal(st["ids"], rids)
    cw = pl.contiguous_weights(cfg, L.w)
    cplan = pm.Plan(L.desc, cw, 3 * (cfg.E + cfg.S))
    cplan.set_path(pm.PATH_TC2)
    assert np.array_equal(out, out_bits(cplan.contig_forward(L.hidden, L.logits)))
    rows = np.unique(np.concatenate([[0, T - 1], np.random.default_rng(3).choice(T, 46, replace=False)]))
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np[rows], L.logits_np[rows])
    assert_close(out[rows], ref["out_bf16"], "expert-major order")


MAXCFG = syn.custom_config("maxsizes", d=64, f=128, E=976, k=16, S=48, n_buffered=40,
                           slots_per_buffer=40)


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("T", [1, 16, 300])
def test_forward_at_maximum_sizes(T, path):
    """E + S = 1024 experts (the most the library takes), k = 16, k + S = 64 pairs per token:
    routing with 32 logits per lane, the widest sort and every kernel family against the oracle,
    with the routing state of the call read back bit-exact."""
    if not serves(path, T):
        pytest.skip("the decode kernels take at most 32 (fused) or 16 (column-slice) tokens")
    cfg = MAXCFG
    L = setup_layer(cfg, T)
    L.plan.set_path(path)
    ws = pm.alloc_workspace(L.desc, T)
    out = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot, workspace=ws))
    assert L.plan.device_error() == 0
    st = L.plan.routing_state(ws, T)
    rids, rw = oracle.route(L.logits_np, cfg.k, cfg.renormalize)
    assert np.array_equal(st["ids"], rids)
    np.testing.assert_allclose(st["weights"], rw, rtol=3e-5, atol=1e-7)
    if st["path"] not in DECODE_PATHS:
        ref_al = oracle.align(rids, cfg.E, cfg.S, st["block_m"])
        assert np.array_equal(st["sorted_ids"], ref_al["sorted_ids"])
        assert np.array_equal(st["inv"], ref_al["inv"])
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np, L.logits_np)
    assert_close(out, ref["out_bf16"], "max sizes T=%d" % T)


def test_empty_batch_writes_nothing():
    cfg = syn.CONFIGS["tiny"]
    L = setup_layer(cfg, 4)
    out = torch.full((0, cfg.d), 1.0, dtype=torch.bfloat16, device="cuda")
    res = L.plan.forward(L.hidden[:0], L.logits[:0], L.page_table, L.buf_slot, out=out,
                         workspace=pm.alloc_workspace(L.desc, 4))
    torch.cuda.synchronize()
    assert res.shape == (0, cfg.d)
    assert L.plan.device_error() == 0


def test_slice_rejects_more_than_16_tokens():
    cfg = syn.CONFIGS["tiny"]
    L = setup_layer(cfg, 17)
    L.plan.set_path(pm.PATH_SLICE)
    with pytest.raises(pm.PmoeError) as ei:
        L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)
    assert ei.value.status == pm._lib.ERR_UNSUPPORTED


def test_slice_and_fused_calls_share_one_plan():
    """Column-slice and fused calls of different token counts in turn on one plan and one
    workspace: both kernels step the plan's grid-barrier words the same way, so no call waits
    out its barrier, every output matches the oracle, and repeated calls are bit-identical."""
    cfg = syn.custom_config("mixS", d=256, f=384, E=16, k=4, S=2, n_buffered=3)
    L = setup_layer(cfg, 32)
    orc = oracle_layer(cfg, L.w)
    ws = pm.alloc_workspace(L.desc, 32)
    seen = {}
    for T, path in [(1, pm.PATH_SLICE), (16, pm.PATH_FUSED), (5, pm.PATH_SLICE), (8, pm.PATH_SLICE),
                    (32, pm.PATH_FUSED), (16, pm.PATH_SLICE), (1, pm.PATH_SLICE), (11, pm.PATH_SLICE),
                    (5, pm.PATH_SLICE), (1, pm.PATH_FUSED)]:
        h, lg = syn.make_tokens(cfg, T)
        L.plan.set_path(path)
        out = out_bits(L.plan.forward(pl._bf16(h).cuda(), torch.from_numpy(lg).cuda(), L.page_table,
                                      L.buf_slot, workspace=ws))
        assert L.plan.device_error() == 0, "T=%d path=%d" % (T, path)
        assert L.plan.last_run()[0] == path
        assert_close(out, orc.forward(h, lg)["out_bf16"], "T=%d path=%d" % (T, path))
        if (T, path) in seen:
            assert np.array_equal(out, seen[(T, path)])
        seen[(T, path)] = out


@pytest.mark.parametrize("name,T", [("qwen15", 1), ("qwen15", 4), ("qwen15", 8), ("qwen15", 16),
                                    ("qwen3next", 1), ("qwen3next", 8), ("qwen3next", 12), ("qwen3next", 16),
                                    ("mixtral", 1), ("mixtral", 4)])
def test_slice_tile_counts_per_cta(name, T):
    """The column-slice kernel on the measured layer shapes, from one tile per working CTA
    (Qwen3-Next-shaped, one token: 88 tiles on 88 CTAs) to twelve (Mixtral-shaped, 4 tokens),
    with shared-chunk tiles streamed before routing on the Qwen shapes, against the oracle on
    every token."""
    cfg = syn.CONFIGS[name]
    L = setup_layer(cfg, T, weights=_weights(name))
    L.plan.set_path(pm.PATH_SLICE)
    ws = pm.alloc_workspace(L.desc, T)
    out = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot, workspace=ws))
    assert L.plan.device_error() == 0
    assert L.plan.last_run()[0] == pm.PATH_SLICE
    st = L.plan.routing_state(ws, T)
    rids, rw = oracle.route(L.logits_np, cfg.k, cfg.renormalize)
    assert np.array_equal(st["ids"], rids)
    assert np.array_equal(st["active"], np.concatenate([cfg.E + np.arange(cfg.S), np.unique(rids)]))
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np, L.logits_np)
    s = assert_close(out, ref["out_bf16"], "%s T=%d" % (name, T))
    # h reaches the down projection rounded to bf16 as the definition has it (the routing weight
    # rides on a high/low pair): the error stays at the level of the fp32-y paths, well inside
    # what rounding w * h itself to bf16 would give
    assert s["mean_rel"] <= 1e-3, s


_WCACHE = {}


def _weights(name):
    if name not in _WCACHE:
        _WCACHE.clear()
        _WCACHE[name] = syn.make_weights(syn.CONFIGS[name])
    return _WCACHE[name]


def spread_logits(T, E, k, seed):
    """Logits under which token t prefers experts t*k .. t*k+k-1 (mod E): the tokens spread over
    the most experts, so the column-slice kernel's CTAs get the most column tiles."""
    lg = np.random.default_rng(seed).normal(size=(T, E)).astype(np.float32)
    for t in range(T):
        for j in range(k):
            lg[t, (t * k + j) % E] += 20.0
    return lg


@pytest.mark.parametrize("name,T", [("qwen15", 16), ("qwen15", 9), ("qwen3next", 16), ("mixtral", 2)])
def test_slice_spread_routing(name, T):
    """The column-slice kernel with the most active experts a token count allows (Qwen1.5-shaped
    16 tokens: 64 experts, 10 column tiles per CTA; Qwen3-Next-shaped 16 tokens: 161 experts;
    9 tokens: a routing warp with one token beside warps with two), against the oracle on every
    token, and the automatic path picks it for these layers at these token counts."""
    cfg = syn.CONFIGS[name]
    L = setup_layer(cfg, T, weights=_weights(name))
    lg = spread_logits(T, cfg.E, cfg.k, 90 + T)
    ws = pm.alloc_workspace(L.desc, T)
    out = out_bits(L.plan.forward(L.hidden, torch.from_numpy(lg).cuda(), L.page_table, L.buf_slot,
                                  workspace=ws))
    assert L.plan.device_error() == 0
    assert L.plan.last_run()[0] == pm.PATH_SLICE
    st = L.plan.routing_state(ws, T)
    rids, _ = oracle.route(lg, cfg.k, cfg.renormalize)
    assert np.array_equal(st["ids"], rids)
    assert len(st["active"]) == cfg.S + len(np.unique(rids)) == cfg.S + min(cfg.E, T * cfg.k)
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np, lg)
    s = assert_close(out, ref["out_bf16"], "%s T=%d spread" % (name, T))
    assert s["mean_rel"] <= 1e-3, s

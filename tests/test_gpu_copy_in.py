"""Copy-in of routed experts that were not prefetched (pmoe_copy_in_missing), through the C ABI.

Rimuru (paper-daily.com/en, "The pipeline: what happens in one scheduling round"): the manager
prefetches the experts it predicts a layer will need, but the layer's actual routing decides, and
an expert the routing picks that is neither cached nor prefetched is copied in before the layer
computes.  Here a prediction is injected on the host (wrong on purpose); the copy-in step must
bring exactly the missed experts (routed, offloaded, not prefetched) into the free slots of the
current load buffer in ascending order, and the layer's output must then equal the all-resident
layer's bit for bit, with no device error.  Failures are made on the host (too few slots, an
expert without a host copy) and must come back as error codes."""
import numpy as np
import pytest
import torch

import oracle
import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import pipeline
from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300 import synthetic as syn

from helpers import assert_close, oracle_layer, out_bits, setup_layer

pytestmark = pytest.mark.gpu


def absent_layer(cfg, T, prefetched_slots, seed=0):
    """A layer whose buffered experts are absent (buffer contents erased), except the ones in
    prefetched_slots {expert: slot}, whose bytes are copied into load buffer 0 at that slot."""
    L = setup_layer(cfg, T, seed=seed)
    pl.nan_fill(L.bufs[0])
    pl.nan_fill(L.bufs[1])
    bs = np.full(cfg.E, -1, np.int32)
    offl = np.flatnonzero(L.placement.buffered)
    bs[offl] = -2
    page = 3 * cfg.f * cfg.d
    for e, s in prefetched_slots.items():
        assert L.placement.buffered[e]
        L.bufs[0][s * page:(s + 1) * page].copy_(pl._bf16(pl.pack_expert(L.w, e, cfg.E, cfg.f)))
        bs[e] = s
    L.buf_slot = torch.from_numpy(bs).cuda()
    L.offloaded = offl
    L.host = [torch.from_numpy(pl.pack_expert(L.w, e, cfg.E, cfg.f).view(np.int16)).pin_memory()
              for e in range(cfg.E)]
    return L


def expected_copy_in(cfg, logits, buffered, bs):
    ids, _ = oracle.route(logits, cfg.k, cfg.renormalize)
    routed = np.unique(ids)
    absent = [int(e) for e in routed if buffered[e] and bs[e] == -2]
    used = set(int(x) for x in bs if x >= 0)
    free = [s for s in range(cfg.slots_per_buffer) if s not in used]
    return absent, free


CFG = syn.custom_config("copyin", d=256, f=256, E=12, k=3, S=1, n_buffered=7, slots_per_buffer=8)


@pytest.mark.parametrize("T", [1, 5, 40, 300])
def test_copy_in_fills_free_slots_in_order_and_matches_resident(T):
    cfg = CFG
    probe = setup_layer(cfg, T)
    offl = np.flatnonzero(probe.placement.buffered)
    pre = {int(offl[0]): 1, int(offl[3]): 4}        # prediction: two experts, slots 1 and 4
    L = absent_layer(cfg, T, pre)
    bs0 = L.buf_slot.cpu().numpy()
    absent, free = expected_copy_in(cfg, L.logits_np, L.placement.buffered, bs0)
    table = pm.device_pointers(L.host)
    missed = torch.full((1 + 2 * cfg.E,), -7, dtype=torch.int32, device="cuda")
    pm.copy_in_missing(L.plan, L.logits, L.buf_slot, 0, table, missed)
    torch.cuda.synchronize()
    assert L.plan.device_error() == 0
    m = missed.cpu().numpy()
    n = len(absent)
    assert m[0] == n
    assert m[1:1 + n].tolist() == absent
    assert m[1 + cfg.E:1 + cfg.E + n].tolist() == free[:n]
    bs1 = L.buf_slot.cpu().numpy()
    want = bs0.copy()
    want[absent] = free[:n]
    assert np.array_equal(bs1, want)
    page = 3 * cfg.f * cfg.d
    for e, s in zip(absent, free):
        got = L.bufs[0][s * page:(s + 1) * page].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, pl.pack_expert(L.w, e, cfg.E, cfg.f))
    # the layer now runs on the copied experts: bit-identical to every expert in the pool
    out = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot))
    assert L.plan.device_error() == 0
    cw = pl.contiguous_weights(cfg, L.w)
    cplan = pm.Plan(L.desc, cw, 3 * (cfg.E + cfg.S))
    assert np.array_equal(out, out_bits(cplan.contig_forward(L.hidden, L.logits)))
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np, L.logits_np)
    assert_close(out, ref["out_bf16"], "copy-in T=%d" % T)


def test_copy_in_with_nothing_absent_copies_nothing():
    cfg = CFG
    L = absent_layer(cfg, 4, {})
    L.buf_slot = torch.full((cfg.E,), -1, dtype=torch.int32, device="cuda")   # no expert absent
    missed = torch.full((1 + 2 * cfg.E,), -7, dtype=torch.int32, device="cuda")
    before = L.buf_slot.clone()
    pm.copy_in_missing(L.plan, L.logits, L.buf_slot, 0, pm.device_pointers(L.host), missed)
    torch.cuda.synchronize()
    assert int(missed[0].item()) == 0
    assert torch.equal(before, L.buf_slot)
    assert L.plan.device_error() == 0


def test_copy_in_reports_running_out_of_slots():
    cfg = syn.custom_config("fewslots", d=256, f=256, E=12, k=3, S=0, n_buffered=7, slots_per_buffer=7)
    T = 40
    L = absent_layer(cfg, T, {})
    # the same memory through a plan whose load buffers have two slots each
    plan2 = pm.Plan(pm.make_desc(cfg.d, cfg.f, cfg.E, cfg.k, cfg.renormalize, cfg.S, 2), L.pool,
                    cfg.num_pages, L.bufs)
    absent, _ = expected_copy_in(cfg, L.logits_np, L.placement.buffered, L.buf_slot.cpu().numpy())
    assert len(absent) > 2
    missed = torch.zeros(1 + 2 * cfg.E, dtype=torch.int32, device="cuda")
    pm.copy_in_missing(plan2, L.logits, L.buf_slot, 0, pm.device_pointers(L.host), missed)
    torch.cuda.synchronize()
    assert plan2.device_error() == pm._lib.ERR_SLOT_OOB
    m = missed.cpu().numpy()
    assert m[0] == 2 and m[1:3].tolist() == absent[:2] and m[1 + cfg.E:3 + cfg.E].tolist() == [0, 1]
    bs = L.buf_slot.cpu().numpy()
    assert bs[absent[:2]].tolist() == [0, 1]
    assert (bs[absent[2:]] == -2).all()


def test_copy_in_reports_an_expert_without_host_copy():
    cfg = CFG
    L = absent_layer(cfg, 20, {})
    absent, _ = expected_copy_in(cfg, L.logits_np, L.placement.buffered, L.buf_slot.cpu().numpy())
    host = list(L.host)
    host[absent[0]] = None
    missed = torch.zeros(1 + 2 * cfg.E, dtype=torch.int32, device="cuda")
    pm.copy_in_missing(L.plan, L.logits, L.buf_slot, 0, pm.device_pointers(host), missed)
    torch.cuda.synchronize()
    assert L.plan.device_error() == pm._lib.ERR_INVALID_ARG
    assert int(missed[0].item()) == len(absent) - 1
    assert int(L.buf_slot[absent[0]].item()) == -2


def test_device_pointers_refuse_misaligned_memory():
    pinned = torch.zeros(64, dtype=torch.int16).pin_memory()
    assert int(pm.device_pointers([pinned, None]).cpu()[1]) == 0
    with pytest.raises(pm.PmoeError):
        pm.device_pointers([pinned[1:]])    # 2 bytes past a 16-byte boundary


def _routed(lg, k):
    ids, _ = oracle.route(lg, k, True)
    return np.unique(ids)


@pytest.mark.parametrize("T", [3, 40])
@pytest.mark.parametrize("kind", ["empty", "wrong", "previous_step"])
def test_stack_driven_by_a_prediction_equals_resident_stack(T, kind):
    """A 4-layer decode stack prefetches from a prediction instead of the actual routing; each
    layer copies in what the prediction missed.  Every step equals the all-resident stack bit for
    bit, no plan raises a device error, and each layer copied in exactly the routed offloaded
    experts that were not predicted."""
    cfg = syn.custom_config("pstack", d=256, f=256, E=8, k=2, S=1, n_buffered=0)
    w = syn.make_weights(cfg)
    L, steps = 4, 3
    rng = np.random.default_rng(11 + T)
    hidden_np = syn.to_bf16_bits(rng.standard_normal((T, cfg.d)).astype(np.float32))
    hidden = torch.from_numpy(hidden_np.view(np.int16)).view(torch.bfloat16).cuda()
    logits = [[syn.bf16_bits_to_f32(syn.to_bf16_bits(rng.standard_normal((T, cfg.E)).astype(np.float32)))
               for _ in range(L)] for _ in range(steps)]
    pred_stack = pipeline.DecodeStack(cfg, w, L, n_offload=4, layouts=2, seed=1)
    res = pipeline.DecodeStack(cfg, w, L, n_offload=0, layouts=1, seed=2)
    ws = pm.alloc_workspace(pred_stack.desc, T)
    acts = [torch.empty_like(hidden) for _ in range(2)]
    acts_r = [torch.empty_like(hidden) for _ in range(2)]
    prev = [np.arange(cfg.E) for _ in range(L)]
    for s, lg in enumerate(logits):
        if kind == "empty":
            pred = [np.array([], np.int64) for _ in range(L)]
        elif kind == "wrong":
            pred = [np.setdiff1d(np.arange(cfg.E), _routed(lg[l], cfg.k)) for l in range(L)]
        else:
            pred = prev
        sched = pred_stack.schedule_predicted(pred)
        lg_dev = [torch.from_numpy(x).cuda() for x in lg]
        y = out_bits(pred_stack.step(hidden, lg_dev, sched, s, acts, ws, copy_in=True)).copy()
        yr = out_bits(res.step(hidden, lg_dev, res.schedule(lg), s, acts_r, ws)).copy()
        torch.cuda.synchronize()
        assert np.array_equal(y, yr), "step %d" % s
        for l in range(L):
            for p in pred_stack.plans[l]:
                assert p.device_error() == 0
            want = np.setdiff1d(np.intersect1d(_routed(lg[l], cfg.k), pred_stack.offloaded[l]),
                                np.asarray(pred[l]))
            m = pred_stack.missed[l].cpu().numpy()
            assert m[1:1 + m[0]].tolist() == want.tolist(), "step %d layer %d" % (s, l)
        prev = [_routed(lg[l], cfg.k) for l in range(L)]

"""The double-buffered load-buffer swap, through the C ABI (Rimuru, paper-daily.com/en, "Expert
weights are scattered across pages...": two loading buffers alternate, one feeds this layer while
the other receives the next layer's experts; "The adjuster...": finish copying before the table
points at the new location, finish computing before a location is reused).

Load buffers start NaN-filled, so a forward that read a slot before its copy landed, or after a
later copy overwrote it, would produce NaN or a different output."""
import numpy as np
import pytest
import torch

import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300 import synthetic as syn

from helpers import assert_close, oracle_layer, out_bits, setup_layer

pytestmark = pytest.mark.gpu


def _host_experts(cfg, w, experts):
    return [torch.from_numpy(pl.pack_expert(w, e, cfg.E, cfg.f).view(np.int16)).pin_memory()
            for e in experts]


def test_prefetched_buffer_gives_identical_output():
    cfg = syn.CONFIGS["qwen15"]
    L = setup_layer(cfg, 64)                      # buffered experts placed in buffer 0
    ref = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot))
    buffered = np.flatnonzero(L.placement.buffered)
    slots = L.placement.slot_of[buffered]
    copy = torch.cuda.Stream()
    done = torch.cuda.Event()
    pm.prefetch_async(L.plan, 1, _host_experts(cfg, L.w, buffered), slots, copy, copy_done=done)
    cur = torch.cuda.current_stream()
    cur.wait_event(done)                          # RAW: compute after the copy
    bs1 = L.buf_slot.clone()
    bs1[torch.from_numpy(buffered).cuda()] += cfg.slots_per_buffer   # now buffer 1
    got = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, bs1))
    assert L.plan.device_error() == 0
    assert np.array_equal(got, ref)


def test_compute_waits_for_a_slow_copy():
    # A large copy on a side stream; the compute stream waits only on copy_done.  If the wait
    # were missing the forward would read NaN-filled slots.
    cfg = syn.CONFIGS["mixtral"]
    w = syn.make_weights(cfg)
    L = setup_layer(cfg, 32, weights=w, n_buffered=2)
    ref = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot))
    buffered = np.flatnonzero(L.placement.buffered)
    host = _host_experts(cfg, w, buffered)        # 2 x 352 MB
    copy = torch.cuda.Stream()
    done = torch.cuda.Event()
    torch.cuda.synchronize()
    pm.prefetch_async(L.plan, 1, host, L.placement.slot_of[buffered], copy, copy_done=done)
    torch.cuda.current_stream().wait_event(done)
    bs1 = L.buf_slot.clone()
    bs1[torch.from_numpy(buffered).cuda()] += cfg.slots_per_buffer
    got = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, bs1))
    assert np.array_equal(got, ref)


def test_buffer_reuse_waits_for_its_last_reader():
    # WAR: layer A reads buffer 0; the next prefetch into buffer 0 must wait for buf_free,
    # recorded after layer A's forward, or A would read the new experts.
    cfg = syn.custom_config("war", d=1024, f=1024, E=8, k=2, S=0, n_buffered=4, slots_per_buffer=4)
    wA = syn.make_weights(cfg, seed=1)
    wB = syn.make_weights(cfg, seed=2)
    L = setup_layer(cfg, 512, weights=wA)
    ref = oracle_layer(cfg, wA).forward(L.hidden_np, L.logits_np)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    torch.cuda._sleep(20_000_000)                 # keep the compute stream busy (bounded)
    outA = L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)
    free = torch.cuda.Event()
    free.record(cur)
    copy = torch.cuda.Stream()
    buffered = np.flatnonzero(L.placement.buffered)
    pm.prefetch_async(L.plan, 0, _host_experts(cfg, wB, buffered), L.placement.slot_of[buffered],
                      copy, buf_free=free, copy_done=torch.cuda.Event())
    torch.cuda.synchronize()
    assert_close(out_bits(outA), ref["out_bf16"], "layer A after the buffer was refilled")
    # and the refilled buffer now serves the other weights
    refB = oracle_layer(cfg, wB).forward(L.hidden_np, L.logits_np)
    outB = L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot)
    torch.cuda.synchronize()
    # experts still in the pool keep wA's weights, so compare only tokens whose experts are all buffered
    ids = refB["ids"]
    only_buf = np.all(L.placement.buffered[ids], axis=1)
    assert only_buf.sum() > 0
    assert_close(out_bits(outB)[only_buf], refB["out_bf16"][only_buf], "layer B")


def test_prefetch_argument_checks_and_wait_timeout():
    cfg = syn.CONFIGS["tiny"]
    L = setup_layer(cfg, 4)
    host = _host_experts(cfg, L.w, [0, 1, 2])
    s = torch.cuda.Stream()
    with pytest.raises(pm.PmoeError) as ei:        # 3 experts > expert_offload_limit (2)
        pm.prefetch_async(L.plan, 0, host, [0, 1, 0], s)
    assert ei.value.status == pm._lib.ERR_INVALID_ARG
    with pytest.raises(pm.PmoeError) as ei:
        pm.prefetch_async(L.plan, 0, host[:2], [0, 0], s)   # duplicate slot
    assert ei.value.status == pm._lib.ERR_INVALID_ARG
    with pytest.raises(pm.PmoeError) as ei:
        pm.prefetch_async(L.plan, 1, host[:1], [2], s)      # slot out of range
    assert ei.value.status == pm._lib.ERR_SLOT_OOB
    with pytest.raises(pm.PmoeError):
        pm.prefetch_async(L.plan, 2, host[:1], [0], s)      # no buffer 2
    # host-side wait with a timeout: pending work -> timeout, then completes
    ev = torch.cuda.Event()
    torch.cuda._sleep(200_000_000)                 # ~0.1 s of bounded device work
    ev.record()
    assert pm.wait_event(ev, 1) is False
    assert pm.wait_event(ev, 10_000) is True

"""The allocation-free forward entry point (moe_paged_forward_noalloc), through the C ABI.

It serves callers that cannot allocate device memory when they run the layer (a plugin or an
embedded runtime held to a fixed device-memory budget, or a loop where cudaMalloc would stall on
in-flight work), so it keeps its intermediates in a fixed device array inside the library instead
of a caller workspace.  Its output must match the plan-based moe_paged_forward and the oracle
within the layer tolerance, on consecutive calls (the array keeps the previous call's contents);
calls after the first must not change the device's free memory; a bad page must reach the
caller's error word; an oversized call must be refused.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import synthetic as syn

from helpers import assert_close, oracle_layer, out_bits, setup_layer

pytestmark = pytest.mark.gpu


def _noalloc(L, err, out=None):
    return pm.forward_noalloc(L.desc, L.pool, L.cfg.num_pages, L.bufs, L.hidden, L.logits,
                              L.page_table, L.buf_slot, out=out, device_error=err)


@pytest.mark.parametrize("name,T1,T2", [("tiny", 16, 5), ("qwen15", 16, 1)])
def test_noalloc_matches_plan_forward_and_oracle_on_two_calls(name, T1, T2):
    cfg = syn.CONFIGS[name]
    w = syn.make_weights(cfg)
    for T in (T1, T2):
        L = setup_layer(cfg, T, weights=w)
        ref = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot))
        orc = oracle_layer(cfg, w).forward(L.hidden_np, L.logits_np)["out_bf16"]
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = out_bits(_noalloc(L, err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(got, ref, "%s T=%d vs plan" % (name, T))
        assert_close(got, orc, "%s T=%d vs oracle" % (name, T))
        got2 = out_bits(_noalloc(L, err))        # second call in a row on the same array
        assert int(err.item()) == 0
        assert_close(got2, orc, "%s T=%d (repeat) vs oracle" % (name, T))
        assert np.array_equal(got, got2)


def test_noalloc_calls_leave_free_device_memory_unchanged():
    cfg = syn.CONFIGS["tiny"]
    w = syn.make_weights(cfg)
    layers = [setup_layer(cfg, T, weights=w) for T in (16, 3)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.empty_like(L.hidden) for L in layers]
    for L, o in zip(layers, outs):     # first calls: kernel loading, the array's address
        _noalloc(L, err, o)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for L, o in zip(layers, outs):
            _noalloc(L, err, o)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(err.item()) == 0


def test_noalloc_reports_a_bad_page_in_the_callers_error_word():
    cfg = syn.CONFIGS["tiny"]
    L = setup_layer(cfg, 16)
    ids, _ = oracle.route(L.logits_np, cfg.k, cfg.renormalize)
    e = int(next(x for x in ids.reshape(-1) if not L.placement.buffered[x]))   # a routed pool expert
    L.page_table = L.page_table.clone()
    L.page_table[e, 2] = cfg.num_pages    # one past the end
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _noalloc(L, err)
    torch.cuda.synchronize()
    assert int(err.item()) == pm._lib.ERR_PAGE_OOB


def test_noalloc_refuses_sizes_beyond_its_scratch():
    cfg = syn.CONFIGS["qwen15"]
    L = setup_layer(cfg, 512, weights=syn.make_weights(cfg))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pm.PmoeError) as ei:
        _noalloc(L, err)
    assert ei.value.status == pm._lib.ERR_WORKSPACE
    assert "scratch" in str(ei.value)

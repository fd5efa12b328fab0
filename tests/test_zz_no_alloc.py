"""The allocation-free forward entry point (moe_paged_forward_noalloc), through the C ABI.

It serves callers that cannot allocate device memory when they run the layer, so it keeps its
intermediates in a fixed device array inside the library instead of a caller workspace.  Its
output must match the plan-based moe_paged_forward within the layer tolerance, on consecutive
calls (the array keeps the previous call's contents), and an oversized call must be refused.
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import synthetic as syn

from helpers import assert_close, out_bits, setup_layer

pytestmark = pytest.mark.gpu


def _noalloc(L, err=None):
    return pm.forward_noalloc(L.desc, L.pool, L.cfg.num_pages, L.bufs, L.hidden, L.logits,
                              L.page_table, L.buf_slot, device_error=err)


@pytest.mark.parametrize("name,T1,T2", [("tiny", 16, 5), ("qwen15", 16, 1)])
def test_noalloc_matches_plan_forward_on_two_calls(name, T1, T2):
    cfg = syn.CONFIGS[name]
    w = syn.make_weights(cfg)
    for T in (T1, T2):
        L = setup_layer(cfg, T, weights=w)
        ref = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = out_bits(_noalloc(L, err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(got, ref, "%s T=%d" % (name, T))
        got2 = out_bits(_noalloc(L))        # second call in a row, internal error word
        assert_close(got2, ref, "%s T=%d (repeat)" % (name, T))
        assert np.array_equal(got, got2)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    cfg = syn.CONFIGS["qwen15"]
    L = setup_layer(cfg, 512, weights=syn.make_weights(cfg))
    with pytest.raises(pm.PmoeError) as ei:
        _noalloc(L)
    assert ei.value.status == pm._lib.ERR_WORKSPACE

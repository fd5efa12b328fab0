"""Parity at the full sizes of the measured workloads, in the launch configuration bench.py
times: integer outputs (routing, sort + pad) compared whole and bit-exact; the layer output
compared on sampled tokens, for which the oracle runs one token at a time (each token's output
depends only on its own hidden row and logits).  Every config is checked on both kernel families
that serve it (weight streaming at decode sizes, tensor cores above)."""
import numpy as np
import pytest
import torch

import oracle
import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import synthetic as syn

from helpers import assert_close, oracle_layer, out_bits, setup_layer

pytestmark = pytest.mark.gpu

_W = {}


def weights(name):
    if name not in _W:
        _W.clear()
        _W[name] = syn.make_weights(syn.CONFIGS[name])
    return _W[name]


CASES = [("qwen15", 1), ("qwen15", 16), ("qwen15", 32), ("qwen15", 128), ("qwen15", 1024),
         ("qwen15", 4096), ("mixtral", 1), ("mixtral", 32), ("mixtral", 512), ("mixtral", 2048),
         ("qwen3next", 1), ("qwen3next", 16), ("qwen3next", 64), ("qwen3next", 256),
         ("qwen3next", 4096)]


@pytest.mark.parametrize("name,T", CASES)
@pytest.mark.parametrize("path", [pm.PATH_AUTO, pm.PATH_STREAM, pm.PATH_TC_DECODE, pm.PATH_TC, pm.PATH_TC2],
                         ids=["auto", "stream", "tc_decode", "tc", "tc2"])
def test_full_size_sampled(name, T, path):
    if path == pm.PATH_STREAM and T > 16:
        pytest.skip("the weight-streaming kernels serve decode sizes")
    if path == pm.PATH_TC_DECODE and T > 32:
        pytest.skip("covered by the automatic path above 32 tokens")
    if path in (pm.PATH_TC, pm.PATH_TC2) and T < 512:
        pytest.skip("the 128-token-block kernels serve prefill sizes")
    cfg = syn.CONFIGS[name]
    L = setup_layer(cfg, T, weights=weights(name))
    L.plan.set_path(path)
    out = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot))
    assert L.plan.device_error() == 0
    # routing and sort + pad, whole, bit-exact (block size of the path that ran)
    path = L.plan.last_run()[0]
    ids, w = pm.route(L.logits, cfg.k, cfg.renormalize)
    rids, rw = oracle.route(L.logits_np, cfg.k, cfg.renormalize)
    assert np.array_equal(ids.cpu().numpy(), rids)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=3e-5, atol=1e-7)
    p2 = 1 << max(0, (T - 1).bit_length())            # next power of two >= T
    bm = {pm.PATH_TC: 128, pm.PATH_TC2: 128, pm.PATH_TC_DECODE: min(128, max(16, p2)),
          pm.PATH_STREAM: min(16, p2), pm.PATH_FUSED: None}[path]
    if bm is not None:   # the fused decode kernel routes in place and needs no sort
        s, b, inv, npad = pm.align(ids, cfg.E, cfg.S, bm)
        ref_al = oracle.align(rids, cfg.E, cfg.S, bm)
        n = int(npad.item())
        assert n == ref_al["n_padded"]
        assert np.array_equal(s[:n].cpu().numpy(), ref_al["sorted_ids"])
        assert np.array_equal(inv.cpu().numpy(), ref_al["inv"])
    # sampled tokens through the oracle
    rng = np.random.default_rng(T)
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=min(T, 6), replace=False)]))
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np[rows], L.logits_np[rows])
    assert_close(out[rows], ref["out_bf16"], "%s T=%d" % (name, T))
    assert np.isfinite(syn.bf16_bits_to_f32(out)).all()

"""Parity at the full sizes of the measured workloads, in the launch configuration bench.py
times: the routing and sort + pad that the forward call itself computed, read back from its
workspace and compared whole and bit-exact; the layer output compared on sampled tokens, for
which the oracle runs one token at a time (each token's output depends only on its own hidden
row and logits).  Every config is checked on both kernel families that serve it (weight
streaming at decode sizes, tensor cores above)."""
import numpy as np
import pytest
import torch

import oracle
import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import synthetic as syn

from helpers import assert_close, oracle_layer, out_bits, setup_layer

pytestmark = pytest.mark.gpu

_W = {}
PATH_NAMES = {pm.PATH_STREAM: "stream", pm.PATH_TC: "tc", pm.PATH_TC_DECODE: "tc_decode",
              pm.PATH_TC2: "tc2", pm.PATH_FUSED: "fused", pm.PATH_SLICE: "slice"}


def weights(name):
    if name not in _W:
        _W.clear()
        _W[name] = syn.make_weights(syn.CONFIGS[name])
    return _W[name]


CASES = [("qwen15", 1), ("qwen15", 16), ("qwen15", 32), ("qwen15", 128), ("qwen15", 1024),
         ("qwen15", 4096), ("mixtral", 1), ("mixtral", 32), ("mixtral", 512), ("mixtral", 2048),
         ("mixtral", 8192), ("qwen3next", 1), ("qwen3next", 16), ("qwen3next", 64),
         ("qwen3next", 256), ("qwen3next", 4096)]


@pytest.mark.parametrize("name,T", CASES)
@pytest.mark.parametrize("path", [pm.PATH_AUTO, pm.PATH_STREAM, pm.PATH_TC_DECODE, pm.PATH_TC, pm.PATH_TC2,
                                  pm.PATH_SLICE],
                         ids=["auto", "stream", "tc_decode", "tc", "tc2", "slice"])
def test_full_size_sampled(name, T, path):
    if path == pm.PATH_STREAM and T > 16:
        pytest.skip("the weight-streaming kernels serve decode sizes")
    if path == pm.PATH_SLICE and T > 16:
        pytest.skip("the column-slice kernel takes at most 16 tokens")
    if path == pm.PATH_TC_DECODE and T > 32:
        pytest.skip("covered by the automatic path above 32 tokens")
    if path in (pm.PATH_TC, pm.PATH_TC2) and T < 512:
        pytest.skip("the 128-token-block kernels serve prefill sizes")
    cfg = syn.CONFIGS[name]
    L = setup_layer(cfg, T, weights=weights(name))
    L.plan.set_path(path)
    ws = pm.alloc_workspace(L.desc, T)
    out = out_bits(L.plan.forward(L.hidden, L.logits, L.page_table, L.buf_slot, workspace=ws))
    assert L.plan.device_error() == 0
    # the routing and sort + pad this very call computed, whole and bit-exact
    st = L.plan.routing_state(ws, T)
    rids, rw = oracle.route(L.logits_np, cfg.k, cfg.renormalize)
    assert np.array_equal(st["ids"], rids)
    np.testing.assert_allclose(st["weights"], rw, rtol=3e-5, atol=1e-7)
    if st["path"] in (pm.PATH_FUSED, pm.PATH_SLICE):
        assert np.array_equal(st["active"], np.concatenate([cfg.E + np.arange(cfg.S), np.unique(rids)]))
    else:
        ref_al = oracle.align(rids, cfg.E, cfg.S, st["block_m"])
        assert int(st["meta"][0]) == ref_al["n_padded"]
        assert np.array_equal(st["sorted_ids"], ref_al["sorted_ids"])
        assert np.array_equal(st["block_expert"], ref_al["block_expert"])
        assert np.array_equal(st["inv"], ref_al["inv"])
    # sampled tokens through the oracle (64 of them from 512 tokens on)
    rng = np.random.default_rng(T)
    n = 64 if T >= 512 else 6
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=min(T, n), replace=False)]))
    ref = oracle_layer(cfg, L.w).forward(L.hidden_np[rows], L.logits_np[rows])
    s = assert_close(out[rows], ref["out_bf16"], "%s T=%d" % (name, T))
    # the margin left inside the tolerance, per case (pytest -s shows it)
    print("\nERRSTAT %s T=%d path=%s tokens=%d max_err/max_ref=%.3e mean_rel=%.3e"
          % (name, T, PATH_NAMES[st["path"]], len(rows), s["max_err"] / s["max_ref"], s["mean_rel"]))
    assert np.isfinite(syn.bf16_bits_to_f32(out)).all()

"""Host-side logic without a GPU: the seeded generators, the placement of experts into pool
pages and load-buffer slots, and reading them back through the tables the kernels use."""
import numpy as np
import pytest
import torch

from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300 import synthetic as syn


def test_generators_are_seeded():
    cfg = syn.CONFIGS["tiny"]
    a = syn.make_weights(cfg, threads=1)
    b = syn.make_weights(cfg, threads=4)
    assert np.array_equal(a.W1, b.W1) and np.array_equal(a.W2, b.W2)
    h1, l1 = syn.make_tokens(cfg, 16)
    h2, l2 = syn.make_tokens(cfg, 16)
    assert np.array_equal(h1, h2) and np.array_equal(l1, l2)
    h3, _ = syn.make_tokens(cfg, 16, seed=5)
    assert not np.array_equal(h1, h3)
    # logits hold bf16 values
    assert np.array_equal(syn.bf16_bits_to_f32(syn.to_bf16_bits(l1)), l1)


def test_value_distributions():
    cfg = syn.CONFIGS["tiny"]
    w = syn.make_weights(cfg)
    x = syn.bf16_bits_to_f32(w.W1).astype(np.float64)
    assert abs(x.std() - 0.02) < 0.001 and abs(x.mean()) < 0.001
    h, _ = syn.make_tokens(cfg, 4096)
    hv = syn.bf16_bits_to_f32(h).astype(np.float64)
    assert abs(hv.std() - 1.0) < 0.01


def test_zipf_and_hot_biases():
    cfg = syn.CONFIGS["qwen3next"]
    _, lg = syn.make_tokens(cfg, 256)
    rank = syn._zipf_rank(cfg, cfg.config_id)
    top = int(np.argmin(rank))
    assert lg[:, top].mean() > lg.mean() + 1.0
    plc = syn.make_placement(cfg)
    assert plc.buffered.sum() == 128
    assert rank[plc.buffered].min() > rank[~plc.buffered].max()   # least popular are buffered
    m = syn.CONFIGS["mixtral"]
    _, lg = syn.make_tokens(m, 2048)
    assert lg[:, :2].mean() - lg[:, 2:].mean() == pytest.approx(1.0, abs=0.1)
    assert syn.make_placement(m).buffered.tolist() == [False] * 6 + [True] * 2


@pytest.mark.parametrize("name", ["tiny", "qwen15", "qwen3next"])
def test_placement_tables(name):
    cfg = syn.CONFIGS[name]
    plc = syn.make_placement(cfg)
    used = plc.page_table[plc.page_table >= 0]
    assert len(np.unique(used)) == len(used)                       # no page shared
    assert used.min() >= 0 and used.max() < cfg.num_pages
    assert (plc.page_table[cfg.E:] >= 0).all()                     # shared chunks in the pool
    assert (plc.page_table[:cfg.E][plc.buffered] == -1).all()
    slots = plc.slot_of[plc.buffered]
    assert sorted(slots.tolist()) == list(range(cfg.n_buffered))
    assert cfg.n_buffered <= cfg.slots_per_buffer


@pytest.mark.parametrize("bidx", [0, 1])
def test_place_and_read_back(bidx):
    cfg = syn.custom_config("rb", d=64, f=128, E=6, k=2, S=2, n_buffered=3, num_pages=40)
    w = syn.make_weights(cfg)
    plc = syn.make_placement(cfg, seed=9)
    pool = pl.new_pool(cfg.num_pages, cfg.f, cfg.d, "cpu")
    bufs = pl.new_load_buffers(cfg.slots_per_buffer, cfg.f, cfg.d, "cpu")
    pt, bs = pl.place(cfg, w, plc, pool, bufs, bidx)
    for e in range(cfg.E + cfg.S):
        got = pl.read_expert(pool, bufs, pt, bs, e, cfg.f, cfg.d, cfg.slots_per_buffer)
        want = pl.expert_matrices(w, e, cfg.E, cfg.f)
        for g, m in zip(got, want):
            assert np.array_equal(g, m)
    # unplaced pages stay NaN; buffered experts' slots follow buf_slot = b*S_buf + s
    free = sorted(set(range(cfg.num_pages)) - set(pt[pt >= 0].tolist()))
    page = cfg.f * cfg.d
    for p in free:
        assert torch.isnan(pool[p * page:(p + 1) * page].float()).all()
    assert ((bs[plc.buffered] // cfg.slots_per_buffer) == bidx).all()


def test_shared_chunk_pages_split_the_shared_expert():
    cfg = syn.custom_config("sh", d=64, f=128, E=2, k=1, S=3, n_buffered=0)
    w = syn.make_weights(cfg)
    for s in range(cfg.S):
        W1c, W3c, W2c = pl.expert_matrices(w, cfg.E + s, cfg.E, cfg.f)
        assert np.array_equal(W1c, w.W1s[s * 128:(s + 1) * 128])
        assert np.array_equal(W2c, w.W2s[:, s * 128:(s + 1) * 128])
    packed = pl.pack_expert(w, 1, cfg.E, cfg.f)
    assert packed.shape == (3 * cfg.f * cfg.d,)
    assert np.array_equal(packed[:cfg.f * cfg.d], w.W1[1].reshape(-1))

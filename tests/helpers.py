"""Shared set-up for the GPU tests: seeded layer inputs placed in a page pool, the oracle's
reference, and the output tolerance.

Tolerance (bf16 outputs from fp32 accumulation): max|err| <= 2e-2 * max|ref| and
sum|err| / sum|ref| <= 5e-3, where ref is the oracle's bf16 output."""
from __future__ import annotations

import types

import numpy as np
import torch

import oracle
import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300 import synthetic as syn

MAX_REL = 2e-2
MEAN_REL = 5e-3


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return syn.bf16_bits_to_f32(b).astype(np.float64)


def out_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def err_stats(got_bits, ref_bits):
    g, r = bits_to_f64(got_bits), bits_to_f64(ref_bits)
    err = np.abs(g - r)
    return {"max_err": float(err.max(initial=0.0)), "max_ref": float(np.abs(r).max(initial=0.0)),
            "mean_rel": float(err.sum() / max(np.abs(r).sum(), 1e-300)),
            "nonfinite": int((~np.isfinite(g)).sum())}


def assert_close(got_bits, ref_bits, what=""):
    s = err_stats(got_bits, ref_bits)
    assert s["nonfinite"] == 0, "%s: %d non-finite outputs" % (what, s["nonfinite"])
    assert s["max_err"] <= MAX_REL * s["max_ref"], "%s: %s" % (what, s)
    assert s["mean_rel"] <= MEAN_REL, "%s: %s" % (what, s)
    return s


def desc_of(cfg):
    return pm.make_desc(cfg.d, cfg.f, cfg.E, cfg.k, cfg.renormalize, cfg.S, cfg.slots_per_buffer)


def setup_layer(cfg, T, seed=None, placement_seed=None, buffer_index=0, n_buffered=None,
                weights=None, device="cuda"):
    """Weights (or the given ones), tokens, a placement, the pool and buffers filled, the
    tables on the device, and a plan."""
    w = weights if weights is not None else syn.make_weights(cfg)
    hidden, logits = syn.make_tokens(cfg, T, seed)
    plc = syn.make_placement(cfg, placement_seed, n_buffered=n_buffered)
    pool = pl.new_pool(cfg.num_pages, cfg.f, cfg.d, device)
    bufs = pl.new_load_buffers(cfg.slots_per_buffer, cfg.f, cfg.d, device)
    pt, bs = pl.place(cfg, w, plc, pool, bufs, buffer_index)
    desc = desc_of(cfg)
    plan = pm.Plan(desc, pool, cfg.num_pages, bufs)
    ns = types.SimpleNamespace(cfg=cfg, w=w, hidden_np=hidden, logits_np=logits, placement=plc,
                               pool=pool, bufs=bufs, desc=desc, plan=plan,
                               page_table=pt.to(device), buf_slot=bs.to(device))
    ns.hidden = pl._bf16(hidden).to(device)
    ns.logits = torch.from_numpy(logits).to(device)
    return ns


def oracle_layer(cfg, w):
    return oracle.Layer(w.W1, w.W3, w.W2, cfg.k, cfg.renormalize, W1s=w.W1s, W3s=w.W3s,
                        W2s=w.W2s, S=cfg.S)

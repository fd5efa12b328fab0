"""Seeded synthetic inputs for the paged fused-MoE layer (shared by the tests and the benchmark).

This module holds no step of the method's arithmetic: it only draws the layer's inputs (hidden
states, router logits, expert weights) and decides where each expert lives (pool pages or a
load-buffer slot), with the shapes and value distributions of the workloads the pages measure.
Random numbers are drawn with numpy's PCG64 from ``SeedSequence(seed)``; per-expert streams are
spawned so the result does not depend on how many threads draw them.

Recipe (one seed per (config, T): ``seed = 1000 * config_id + T``):
  * weights ~ N(0, 0.02), hidden ~ N(0, 1), logits ~ N(0, 1), each rounded to bf16 (RNE);
    logits are handed to the layer as fp32 holding bf16 values;
  * Mixtral-shaped: +1.0 on the logits of experts 0 and 1 (the two hot experts) before rounding;
  * Qwen3-Next-shaped: + bias_e = -1.1 * ln(rank_e), rank a seeded permutation of 1..E, so the
    routing prior follows Zipf(1.1); the least popular experts are the buffered ones;
  * pool: P = 3 * (E + S) pages (tiny: 32), placement = a seeded permutation of the pages;
    pages and slots that hold no expert are filled with bf16 NaN so a stray read shows up.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    config_id: int
    d: int                 # hidden size
    f: int                 # per-expert intermediate size (one page = f*d bf16)
    E: int                 # routed experts
    k: int                 # top-k
    S: int                 # shared-expert chunks of width f (shared intermediate = S*f)
    renormalize: bool
    tokens: tuple          # token counts the workload is measured at
    n_buffered: int        # experts served from a load buffer (the rest are pool-resident)
    slots_per_buffer: int  # expert_offload_limit
    num_pages: int         # pool pages P
    logit_bias: str        # "none" | "hot2" | "zipf1.1"

    @property
    def fs(self) -> int:
        return self.S * self.f


CONFIGS = {
    "tiny": LayerConfig("tiny", 0, d=256, f=128, E=8, k=2, S=0, renormalize=True,
                        tokens=(16,), n_buffered=2, slots_per_buffer=2, num_pages=32,
                        logit_bias="none"),
    "qwen15": LayerConfig("qwen15_moe_14b_shaped", 1, d=2048, f=1408, E=60, k=4, S=4,
                          renormalize=False, tokens=(1, 16, 128, 1024, 4096), n_buffered=15,
                          slots_per_buffer=15, num_pages=3 * (60 + 4), logit_bias="none"),
    "mixtral": LayerConfig("mixtral_8x7b_shaped", 2, d=4096, f=14336, E=8, k=2, S=0,
                           renormalize=True, tokens=(1, 32, 512, 2048, 8192), n_buffered=2,
                           slots_per_buffer=2, num_pages=3 * 8, logit_bias="hot2"),
    "qwen3next": LayerConfig("qwen3_next_80b_a3b_shaped", 3, d=2048, f=512, E=512, k=10, S=1,
                             renormalize=True, tokens=(1, 64, 256, 4096), n_buffered=128,
                             slots_per_buffer=128, num_pages=3 * (512 + 1),
                             logit_bias="zipf1.1"),
}


def custom_config(name="custom", d=256, f=128, E=8, k=2, S=0, renormalize=True, n_buffered=2,
                  slots_per_buffer=None, num_pages=None, logit_bias="none"):
    """A small layer of arbitrary shape (tests: ragged tiles, degenerate cases)."""
    if slots_per_buffer is None:
        slots_per_buffer = max(1, n_buffered)
    if num_pages is None:
        num_pages = 3 * (E + S)
    return LayerConfig(name, 99, d=d, f=f, E=E, k=k, S=S, renormalize=renormalize, tokens=(),
                       n_buffered=n_buffered, slots_per_buffer=slots_per_buffer,
                       num_pages=num_pages, logit_bias=logit_bias)


def seed_for(cfg: LayerConfig, T: int) -> int:
    return 1000 * cfg.config_id + int(T)


# ---------------------------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even.  Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, scale: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return to_bf16_bits(x)


def _zipf_rank(cfg: LayerConfig, seed: int) -> np.ndarray:
    """rank_e in 1..E (1 = most popular), a seeded permutation fixed per config."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    return rng.permutation(cfg.E) + 1


def make_tokens(cfg: LayerConfig, T: int, seed: int | None = None):
    """hidden [T,d] bf16 bits (uint16) and router logits [T,E] fp32 (bf16 values)."""
    if seed is None:
        seed = seed_for(cfg, T)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1])))
    hidden = _normal_bf16(rng, (T, cfg.d), 1.0)
    lg = rng.standard_normal(size=(T, cfg.E), dtype=np.float32)
    if cfg.logit_bias == "hot2":
        lg[:, :2] += np.float32(1.0)
    elif cfg.logit_bias == "zipf1.1":
        rank = _zipf_rank(cfg, cfg.config_id)
        lg += (-1.1 * np.log(rank.astype(np.float64))).astype(np.float32)[None, :]
    logits = bf16_bits_to_f32(to_bf16_bits(lg))
    return hidden, logits


@dataclasses.dataclass
class ExpertWeights:
    """Contiguous per-expert weights, bf16 bit patterns.  W1/W3 [E,f,d], W2 [E,d,f];
    shared W1s/W3s [S*f,d], W2s [d,S*f] (None when S == 0)."""
    W1: np.ndarray
    W3: np.ndarray
    W2: np.ndarray
    W1s: np.ndarray | None
    W3s: np.ndarray | None
    W2s: np.ndarray | None


def make_weights(cfg: LayerConfig, seed: int | None = None, threads: int | None = None) -> ExpertWeights:
    if seed is None:
        seed = 1000 * cfg.config_id
    E, f, d, S = cfg.E, cfg.f, cfg.d, cfg.S
    W1 = np.empty((E, f, d), np.uint16)
    W3 = np.empty((E, f, d), np.uint16)
    W2 = np.empty((E, d, f), np.uint16)
    children = np.random.SeedSequence([seed, 2]).spawn(E + 1)

    def one(e):
        rng = np.random.Generator(np.random.PCG64(children[e]))
        W1[e] = _normal_bf16(rng, (f, d), 0.02)
        W3[e] = _normal_bf16(rng, (f, d), 0.02)
        W2[e] = _normal_bf16(rng, (d, f), 0.02)

    threads = threads or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, range(E)))
    if S:
        rng = np.random.Generator(np.random.PCG64(children[E]))
        W1s = _normal_bf16(rng, (S * f, d), 0.02)
        W3s = _normal_bf16(rng, (S * f, d), 0.02)
        W2s = _normal_bf16(rng, (d, S * f), 0.02)
    else:
        W1s = W3s = W2s = None
    return ExpertWeights(W1, W3, W2, W1s, W3s, W2s)


@dataclasses.dataclass
class Placement:
    """Where each expert lives.  buffered[e] = True -> in a load buffer, slot buf_slot_of[e];
    otherwise page_of[e] = (page of W1, page of W3, page of W2) in the pool.  Shared chunks
    (rows E..E+S-1 of the page table) are always pool-resident."""
    page_table: np.ndarray     # [E+S, 3] int32, -1 for buffered experts
    slot_of: np.ndarray        # [E] int32: slot within its buffer, -1 when pool-resident
    num_pages: int
    buffered: np.ndarray       # [E] bool


def make_placement(cfg: LayerConfig, seed: int | None = None, n_buffered: int | None = None) -> Placement:
    if seed is None:
        seed = 1000 * cfg.config_id
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 3])))
    E, S, P = cfg.E, cfg.S, cfg.num_pages
    nb = cfg.n_buffered if n_buffered is None else n_buffered
    if cfg.logit_bias == "zipf1.1":
        rank = _zipf_rank(cfg, cfg.config_id)
        buffered_ids = np.argsort(-rank, kind="stable")[:nb]       # least popular
    elif cfg.logit_bias == "hot2":
        buffered_ids = np.arange(E - nb, E)                         # coldest = highest ids
    else:
        buffered_ids = rng.permutation(E)[:nb]
    buffered = np.zeros(E, bool)
    buffered[buffered_ids] = True
    n_resident = (E - nb) + S
    if 3 * n_resident > P:
        raise ValueError("pool of %d pages cannot hold %d resident experts" % (P, n_resident))
    perm = rng.permutation(P).astype(np.int32)
    page_table = np.full((E + S, 3), -1, np.int32)
    slot_of = np.full(E, -1, np.int32)
    nxt = 0
    for e in range(E + S):
        if e < E and buffered[e]:
            continue
        page_table[e] = perm[nxt:nxt + 3]
        nxt += 3
    slot = 0
    for e in range(E):
        if buffered[e]:
            slot_of[e] = slot
            slot += 1
    return Placement(page_table, slot_of, P, buffered)

"""Host-side page-pool bookkeeping: lay experts out in pool pages and load-buffer slots.

Rimuru (paper-daily.com/en, "One pool for data whose sizes differ by orders of magnitude") keeps
one contiguous byte range and reads it through views; an expert page holds one weight matrix
(f*d bf16), and an expert takes three of them (section "The adjuster": gate W1, up W3, down W2).
A load-buffer slot holds the same three matrices back to back.  This module only copies bytes
into those places and builds the tables the kernels read; it does no arithmetic on them.
"""
from __future__ import annotations

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0


def _bf16(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 (CPU, no copy of the values)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def nan_fill(t: torch.Tensor) -> torch.Tensor:
    t.view(torch.int16).fill_(BF16_NAN_BITS)
    return t


def new_pool(num_pages: int, f: int, d: int, device="cuda") -> torch.Tensor:
    """num_pages pages of f*d bf16, filled with NaN so an unplaced page never reads as data."""
    return nan_fill(torch.empty(num_pages * f * d, dtype=torch.bfloat16, device=device))


def new_load_buffers(slots: int, f: int, d: int, device="cuda"):
    if slots == 0:
        return (None, None)
    return tuple(nan_fill(torch.empty(slots * 3 * f * d, dtype=torch.bfloat16, device=device))
                 for _ in range(2))


def expert_matrices(w, e: int, E: int, f: int):
    """The three page-sized matrices of expert e (shared chunk s = expert E + s), as uint16:
    W1 [f,d], W3 [f,d], W2 [d,f]."""
    if e < E:
        return w.W1[e], w.W3[e], w.W2[e]
    s = e - E
    return (w.W1s[s * f:(s + 1) * f], w.W3s[s * f:(s + 1) * f],
            np.ascontiguousarray(w.W2s[:, s * f:(s + 1) * f]))


def pack_expert(w, e: int, E: int, f: int) -> np.ndarray:
    """W1 | W3 | W2 of one expert, back to back (the load-buffer slot layout)."""
    return np.concatenate([m.reshape(-1) for m in expert_matrices(w, e, E, f)])


def place(cfg, w, placement, pool: torch.Tensor, load_bufs, buffer_index: int = 0):
    """Copy every expert to where `placement` says and return (page_table, buf_slot) as int32
    CPU tensors.  Pool experts go to their three pages; buffered experts go to slot
    placement.slot_of[e] of load buffer `buffer_index` (buf_slot = b * S_buf + slot)."""
    E, S, f, d = cfg.E, cfg.S, cfg.f, cfg.d
    page = f * d
    for e in range(E + S):
        mats = expert_matrices(w, e, E, f)
        if e < E and placement.buffered[e]:
            s = int(placement.slot_of[e])
            dst = load_bufs[buffer_index]
            for j, m in enumerate(mats):
                dst[(3 * s + j) * page:(3 * s + j + 1) * page].copy_(_bf16(m.reshape(-1)))
        else:
            for j, m in enumerate(mats):
                p = int(placement.page_table[e, j])
                pool[p * page:(p + 1) * page].copy_(_bf16(m.reshape(-1)))
    page_table = torch.from_numpy(placement.page_table.copy())
    buf_slot = torch.from_numpy(np.where(placement.buffered,
                                         buffer_index * cfg.slots_per_buffer + placement.slot_of,
                                         -1).astype(np.int32))
    return page_table, buf_slot


def contiguous_weights(cfg, w, device="cuda") -> torch.Tensor:
    """Expert e's W1, W3, W2 as pages 3e, 3e+1, 3e+2 of one array (shared chunk s = expert
    E + s): the layout the contiguous twin of the forward reads with fixed addressing."""
    E, S, f, d = cfg.E, cfg.S, cfg.f, cfg.d
    out = torch.empty(3 * (E + S) * f * d, dtype=torch.bfloat16, device=device)
    page = f * d
    for e in range(E + S):
        for j, m in enumerate(expert_matrices(w, e, E, f)):
            out[(3 * e + j) * page:(3 * e + j + 1) * page].copy_(_bf16(m.reshape(-1)))
    return out


def read_expert(pool: torch.Tensor, load_bufs, page_table, buf_slot, e: int, f: int, d: int,
                slots_per_buffer: int):
    """Inverse of `place` for one expert (host check of the tables): its three matrices as
    uint16 numpy arrays, fetched through the table exactly as the kernels address them."""
    page = f * d
    bs = int(buf_slot[e]) if e < len(buf_slot) else -1
    mats = []
    for j in range(3):
        if bs >= 0:
            b, s = divmod(bs, slots_per_buffer)
            src = load_bufs[b][(3 * s + j) * page:(3 * s + j + 1) * page]
        else:
            p = int(page_table[e, j])
            src = pool[p * page:(p + 1) * page]
        mats.append(src.cpu().view(torch.int16).numpy().view(np.uint16))
    return mats[0].reshape(f, d), mats[1].reshape(f, d), mats[2].reshape(d, f)

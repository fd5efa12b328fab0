"""Python binding of libpmoe's three-tier page allocator (host only; marshalling only), and the
memory views that read one pool with each tier's page size.

Rimuru, section "One pool for data whose sizes differ by orders of magnitude": the pool is one
contiguous byte range; experts, the KV cache, SSM states and convolution states each read it
through a view with their own page size and shape (no copy), and pages move between tiers by
splitting downward and merging upward.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib

EXPERT, SSM, KV, CONV = 0, 1, 2, 3


class Tiers:
    def __init__(self, pool_bytes: int, expert_page: int, ssm_page: int = 0, kv_page: int = 0,
                 conv_page: int = 0):
        self._lib = _lib.load()
        h = ctypes.c_void_p()
        _lib.check(self._lib.pmoe_tiers_create(int(pool_bytes), int(expert_page), int(ssm_page),
                                               int(kv_page), int(conv_page), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            self._lib.pmoe_tiers_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        self.close()

    def alloc(self, kind: int, owner: int = 0):
        """Byte offset of a new page of `kind`, or None when the pool has no room."""
        off = ctypes.c_int64()
        _lib.check(self._lib.pmoe_tiers_alloc(self._h, int(kind), int(owner), ctypes.byref(off)))
        return None if off.value < 0 else off.value

    def free(self, kind: int, offset: int):
        _lib.check(self._lib.pmoe_tiers_free(self._h, int(kind), int(offset)))

    def stats(self):
        """[huge page bytes, free huge, free expert, free SSM, live expert, live SSM, split expert
        pages, free small pages]."""
        c = np.zeros(8, dtype=np.int64)
        _lib.check(self._lib.pmoe_tiers_stats(self._h, c.ctypes.data))
        return c.tolist()


def page_view(pool: torch.Tensor, offset: int, nbytes: int, dtype: torch.dtype, shape) -> torch.Tensor:
    """The page at byte `offset` of the pool as a tensor of `dtype` and `shape`, sharing the
    pool's memory (the section's memory view: .view(dtype) and .view(shape), no copy)."""
    raw = pool.view(torch.uint8)
    return raw[offset:offset + nbytes].view(dtype).view(shape)


def expert_page_index(offset: int, expert_page: int) -> int:
    """The kernels' page number of an expert page at byte `offset` of the pool."""
    if offset % expert_page:
        raise ValueError("not an expert page boundary")
    return offset // expert_page

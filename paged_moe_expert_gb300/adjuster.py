"""Python binding of libpmoe's adjuster (host only; marshalling only).

The adjuster (Rimuru, section "The adjuster: when to evict an expert, and which one?") decides
after each scheduling round whether the expert cache grows, shrinks or stays, which experts
move and which pages of the shared pool they take or release.  The rules run in libpmoe's
native code; this class converts numpy arrays to pointers and raises on a bad status.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib

ADD, EVICT = 1, -1


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


class Adjuster:
    """Per-layer expert cache over one page pool.

    probs: [n_layers, n_experts] routing probabilities of the offline ranking; cached:
    [n_layers] experts each layer keeps at the start (its top-ranked ones, on pages 0, 1, 2, ...
    layer by layer); offload_limit: layers offloading that many experts are left out of
    shrinking; num_pages: the pool's size in expert pages.
    """

    def __init__(self, probs, cached, offload_limit: int, num_pages: int):
        self._lib = _lib.load()
        probs = np.ascontiguousarray(probs, dtype=np.float32)
        if probs.ndim != 2:
            raise ValueError("probs must be [n_layers, n_experts]")
        self.n_layers, self.n_experts = probs.shape
        cached = _i32(cached)
        if cached.shape != (self.n_layers,):
            raise ValueError("cached must be [n_layers]")
        h = ctypes.c_void_p()
        _lib.check(self._lib.pmoe_adjuster_create(
            self.n_layers, self.n_experts, probs.ctypes.data, int(offload_limit),
            cached.ctypes.data, int(num_pages), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pmoe_adjuster_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def decide(self, short_pages: int, max_changes: int | None = None) -> np.ndarray:
        """One round with R_b = short_pages: returns int32 [n, 6] records
        (+1 add / -1 evict, layer, expert, page of W1, page of W3, page of W2)."""
        if max_changes is None:
            max_changes = self.n_layers
        out = np.zeros((max(int(max_changes), 1), 6), dtype=np.int32)
        n = ctypes.c_int32()
        _lib.check(self._lib.pmoe_adjuster_decide(self._h, int(short_pages), int(max_changes),
                                                  out.ctypes.data, ctypes.byref(n)))
        return out[:n.value].copy()

    def end_forward(self):
        _lib.check(self._lib.pmoe_adjuster_end_forward(self._h))

    def lend(self, n: int) -> np.ndarray:
        pages = np.zeros(max(int(n), 1), dtype=np.int32)
        _lib.check(self._lib.pmoe_adjuster_lend(self._h, int(n), pages.ctypes.data))
        return pages[:int(n)].copy()

    def give_back(self, pages):
        pages = _i32(pages).reshape(-1)
        _lib.check(self._lib.pmoe_adjuster_give_back(self._h, pages.size, pages.ctypes.data))

    def free_pages(self) -> int:
        f = ctypes.c_int64()
        _lib.check(self._lib.pmoe_adjuster_state(self._h, ctypes.byref(f), None))
        return f.value

    def cached(self) -> np.ndarray:
        f = ctypes.c_int64()
        c = np.zeros(self.n_layers, dtype=np.int32)
        _lib.check(self._lib.pmoe_adjuster_state(self._h, ctypes.byref(f), c.ctypes.data))
        return c

    def page_table(self, layer: int) -> np.ndarray:
        t = np.zeros((self.n_experts, 3), dtype=np.int32)
        _lib.check(self._lib.pmoe_adjuster_page_table(self._h, int(layer), t.ctypes.data))
        return t

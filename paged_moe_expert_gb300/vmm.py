"""Python binding of libpmoe's remapped contiguous view (host calls; marshalling only).

FluxMoE (awesome-system-papers, section "核心方法", PagedTensor) reads scattered expert weights
with an unmodified contiguous kernel by mapping physical blocks under stable virtual addresses
(CUDA driver virtual memory management) before the kernel runs.  `VmmView` holds one physical
block per expert page and two address ranges over them: `blocks` (block i at page i, for the
page-table forward) and `view` (virtual pages mapped on request, for the contiguous forward).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib


def granularity(device: int = 0) -> int:
    g = ctypes.c_size_t()
    _lib.check(_lib.load().pmoe_vmm_granularity(int(device), ctypes.byref(g)))
    return g.value


class DevicePointer:
    """A device address with the `data_ptr()` the plan and copy calls read."""

    def __init__(self, ptr: int):
        self.ptr = int(ptr)

    def data_ptr(self) -> int:
        return self.ptr


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64).reshape(-1))


class VmmView:
    def __init__(self, block_bytes: int, n_blocks: int, n_virtual: int, device: int = 0):
        self._lib = _lib.load()
        h = ctypes.c_void_p()
        _lib.check(self._lib.pmoe_vmm_create(int(device), int(block_bytes), int(n_blocks),
                                             int(n_virtual), ctypes.byref(h)))
        self._h = h
        self.block_bytes, self.n_blocks, self.n_virtual = int(block_bytes), int(n_blocks), int(n_virtual)
        b, v = ctypes.c_void_p(), ctypes.c_void_p()
        _lib.check(self._lib.pmoe_vmm_pointers(h, ctypes.byref(b), ctypes.byref(v)))
        self.blocks = DevicePointer(b.value)
        self.view = DevicePointer(v.value)

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            _lib.check(self._lib.pmoe_vmm_destroy(self._h))
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def map(self, virt, blocks):
        v, b = _i64(virt), _i64(blocks)
        if v.size != b.size:
            raise ValueError("virt and blocks differ in length")
        _lib.check(self._lib.pmoe_vmm_map(self._h, v.size, v.ctypes.data, b.ctypes.data))

    def unmap(self, virt, readers_done=None, timeout_ms: int = 2000):
        v = _i64(virt)
        ev = None
        if readers_done is not None and readers_done.cuda_event != 0:
            ev = ctypes.c_void_p(readers_done.cuda_event)
        _lib.check(self._lib.pmoe_vmm_unmap(self._h, v.size, v.ctypes.data, ev, int(timeout_ms)))

    def lookup(self) -> np.ndarray:
        out = np.empty(self.n_virtual, dtype=np.int64)
        _lib.check(self._lib.pmoe_vmm_lookup(self._h, out.ctypes.data))
        return out


def expert_view_pages(E: int, S: int) -> np.ndarray:
    """Virtual page of every expert matrix in the contiguous layout: expert e (shared chunk s is
    expert E + s), matrix j (W1, W3, W2) at page 3e + j."""
    return np.arange(3 * (E + S), dtype=np.int64).reshape(E + S, 3)


def map_experts(vmm: VmmView, page_table) -> None:
    """Map the view so that expert e's matrix j (virtual page 3e + j) reads the block the page
    table names for it: the remapped twin of a paged placement, same physical bytes."""
    pt = np.asarray(page_table, dtype=np.int64)
    vmm.map(expert_view_pages(pt.shape[0], 0).reshape(-1)[:pt.size], pt.reshape(-1))

"""Paged fused-MoE layer forward for GB300 (sm_103a) -- Python binding of libpmoe.

The layer (Rimuru, paper-daily.com/en, "Expert weights are scattered across pages. How does the
kernel read them?") reads each expert's gate (W1), up (W3) and down (W2) projection from pages
of a shared pool, or from a slot of one of two alternating load buffers, through a per-expert
page table -- never from a contiguous copy.  Every step runs in libpmoe's CUDA kernels; this
module only converts torch tensors to pointers and sizes and raises on a bad status.  PyTorch
supplies device memory, streams and events.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib
from .adjuster import Adjuster
from ._lib import (PATH_AUTO, PATH_FUSED, PATH_SLICE, PATH_STREAM, PATH_TC, PATH_TC2, PATH_TC_DECODE, LayerDesc,
                   PmoeError)

__all__ = ["Adjuster", "LayerDesc", "Plan", "PmoeError", "workspace_size", "route", "align",
           "prefetch_async", "fill_pages_async", "wait_event", "copy_in_missing", "device_pointers", "PATH_AUTO", "PATH_STREAM", "PATH_TC", "PATH_TC_DECODE", "PATH_TC2", "PATH_FUSED", "PATH_SLICE",
           "make_desc"]


def make_desc(d, f, num_experts, top_k, renormalize, num_shared_chunks=0, slots_per_buffer=0):
    return LayerDesc(int(d), int(f), int(num_experts), int(top_k), int(bool(renormalize)),
                     int(num_shared_chunks), int(slots_per_buffer))


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _event(e, stream=None):
    """cudaEvent_t of a torch.cuda.Event; torch creates the event on its first record, so an
    event never recorded is recorded once here (on `stream`) to bring it into existence."""
    if e is None:
        return None
    if e.cuda_event == 0:
        e.record(stream if stream is not None else torch.cuda.current_stream())
    return ctypes.c_void_p(e.cuda_event)


def workspace_size(desc: LayerDesc, max_tokens: int) -> int:
    return int(_lib.load().pmoe_workspace_size(ctypes.byref(desc), int(max_tokens)))


def alloc_workspace(desc: LayerDesc, max_tokens: int, device="cuda") -> torch.Tensor:
    n = workspace_size(desc, max_tokens)
    if n == 0:
        raise PmoeError(_lib.ERR_INVALID_ARG, "bad descriptor or token count")
    return torch.empty(n, dtype=torch.uint8, device=device)


class Plan:
    """Owns a libpmoe plan over a page pool (bf16, num_pages * f * d elements) and up to two
    load buffers (bf16, slots_per_buffer * 3 * f * d elements each)."""

    def __init__(self, desc: LayerDesc, pool: torch.Tensor, num_pages: int,
                 load_bufs=(None, None)):
        self.desc = desc
        self._keep = (pool,) + tuple(load_bufs)   # the tensors must outlive the plan
        h = ctypes.c_void_p()
        b0, b1 = load_bufs
        _lib.check(_lib.load().pmoe_plan_create(ctypes.byref(desc), _ptr(pool), int(num_pages),
                                                _ptr(b0), _ptr(b1), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            _lib.check(_lib.load().pmoe_plan_destroy(self._h))
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_path(self, path: int):
        _lib.check(_lib.load().pmoe_plan_set_path(self._h, int(path)))

    def forward(self, hidden, logits, page_table, buf_slot, out=None, workspace=None,
                stream=None):
        T = hidden.shape[0]
        if out is None:
            out = torch.empty_like(hidden)
        if workspace is None:
            workspace = alloc_workspace(self.desc, T, hidden.device)
        _lib.check(_lib.load().moe_paged_forward(
            self._h, _ptr(hidden), int(T), _ptr(logits), int(self.desc.top_k), _ptr(page_table),
            _ptr(buf_slot), _ptr(out), _ptr(workspace), int(workspace.numel()), _stream(stream)))
        return out

    def contig_forward(self, hidden, logits, out=None, workspace=None, stream=None):
        T = hidden.shape[0]
        if out is None:
            out = torch.empty_like(hidden)
        if workspace is None:
            workspace = alloc_workspace(self.desc, T, hidden.device)
        _lib.check(_lib.load().moe_contig_forward(
            self._h, _ptr(hidden), int(T), _ptr(logits), int(self.desc.top_k), _ptr(out),
            _ptr(workspace), int(workspace.numel()), _stream(stream)))
        return out

    def last_run(self):
        """(path, profiled steps, kernel launches) of the last forward call."""
        p, n, k = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        _lib.check(_lib.load().pmoe_plan_last_run(self._h, ctypes.byref(p), ctypes.byref(n),
                                                  ctypes.byref(k)))
        return int(p.value), int(n.value), int(k.value)

    def routing_state(self, workspace: torch.Tensor, T: int) -> dict:
        """The routing and sort state the last forward call (T tokens, this workspace) left in the
        workspace, copied to host numpy arrays (pmoe_plan_routing_view gives the offsets).  Keys:
        path, block_m, ids [T,k], weights [T,k], meta [16], and when the call's path writes them
        sorted_ids [n_padded], block_expert, inv, block_rows, units [n,4], active."""
        v = _lib.RoutingView()
        _lib.check(_lib.load().pmoe_plan_routing_view(self._h, int(T), ctypes.byref(v)))
        torch.cuda.synchronize(workspace.device)
        ws = workspace.cpu().numpy()
        k, S, E = self.desc.top_k, self.desc.num_shared_chunks, self.desc.num_experts

        def arr(off, n, dt=np.int32):
            return ws[off:off + 4 * n].view(dt).copy()

        meta = arr(v.meta, 16)
        out = {"path": int(v.path), "block_m": int(v.block_m), "meta": meta,
               "ids": arr(v.ids, T * k).reshape(T, k), "weights": arr(v.weights, T * k, np.float32).reshape(T, k)}
        if v.sorted_ids >= 0:
            npad = int(meta[0])
            out["sorted_ids"] = arr(v.sorted_ids, npad)
            out["block_expert"] = arr(v.block_expert, npad // v.block_m)
            out["inv"] = arr(v.inv, T * (k + S))
        if v.block_rows >= 0:
            out["block_rows"] = arr(v.block_rows, int(meta[0]) // v.block_m)
        if v.units >= 0:
            out["units"] = arr(v.units, 4 * int(meta[1])).reshape(-1, 4)
        if v.active >= 0:
            out["active"] = arr(v.active, int(meta[3]))
        return out

    def set_profile_events(self, events):
        """Record events[i] before the forward's i-th kernel (and one after the last); pass
        None or [] to stop.  The events must stay alive while set."""
        events = list(events or [])
        arr = (ctypes.c_void_p * max(len(events), 1))(
            *[(_event(e).value if e is not None else None) for e in events])
        self._prof = events
        _lib.check(_lib.load().pmoe_plan_set_profile_events(self._h, arr, len(events)))

    def device_error(self, clear: bool = True, stream=None) -> int:
        code = ctypes.c_int32(0)
        _lib.check(_lib.load().pmoe_get_device_error(self._h, int(bool(clear)), ctypes.byref(code),
                                                     _stream(stream)))
        return int(code.value)


def forward_noalloc(desc: LayerDesc, pool, num_pages, load_bufs, hidden, logits, page_table,
                    buf_slot, out=None, device_error=None, stream=None):
    """moe_paged_forward_noalloc: the layer forward with the library's fixed scratch instead of
    a plan and a workspace (no device allocation in the call; decode-size token counts)."""
    if out is None:
        out = torch.empty_like(hidden)
    b0, b1 = load_bufs
    _lib.check(_lib.load().moe_paged_forward_noalloc(
        ctypes.byref(desc), _ptr(pool), int(num_pages), _ptr(b0), _ptr(b1), _ptr(hidden),
        int(hidden.shape[0]), _ptr(logits), int(desc.top_k), _ptr(page_table), _ptr(buf_slot),
        _ptr(out), _ptr(device_error), _stream(stream)))
    return out


def route(logits: torch.Tensor, top_k: int, renormalize: bool, stream=None):
    T, E = logits.shape
    ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _lib.check(_lib.load().pmoe_route(_ptr(logits), int(T), int(E), int(top_k),
                                      int(bool(renormalize)), _ptr(ids), _ptr(w), _stream(stream)))
    return ids, w


def align(ids: torch.Tensor, E: int, S: int, block_m: int, stream=None, multi_cta=False):
    T, k = ids.shape
    NP = T * (k + S)
    dev = ids.device
    sorted_ids = torch.empty(NP + (E + S) * (block_m - 1) + 1, dtype=torch.int32, device=dev)
    block_expert = torch.empty(NP // block_m + E + S + 1, dtype=torch.int32, device=dev)
    inv = torch.empty(max(NP, 1), dtype=torch.int32, device=dev)
    npad = torch.zeros(1, dtype=torch.int32, device=dev)
    scratch = None
    if multi_cta:
        scratch = torch.empty(int(_lib.load().pmoe_align_scratch_size()), dtype=torch.uint8, device=dev)
    _lib.check(_lib.load().pmoe_align(_ptr(ids), int(T), int(k), int(E), int(S), int(block_m),
                                      _ptr(sorted_ids), _ptr(block_expert), _ptr(inv), _ptr(npad),
                                      _ptr(scratch), _stream(stream)))
    return sorted_ids, block_expert, inv[:NP], npad


def prefetch_async(plan: Plan, buf: int, host_experts, slots, copy_stream, buf_free=None,
                   copy_done=None):
    """Copy experts (pinned host tensors of 3*f*d bf16: W1|W3|W2) into slots of load buffer
    `buf` on `copy_stream`, after `buf_free` and before `copy_done` (torch.cuda.Event or None)."""
    n = len(host_experts)
    ptrs = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in host_experts])
    sl = (ctypes.c_int32 * max(n, 1))(*[int(s) for s in slots])
    # an event that was never recorded has nothing to wait for
    free = _event(buf_free) if (buf_free is not None and buf_free.cuda_event != 0) else None
    _lib.check(_lib.load().pmoe_prefetch_async(plan._h, int(buf), int(n), ptrs, sl,
                                               _stream(copy_stream), free,
                                               _event(copy_done, copy_stream)))


def fill_pages_async(plan: Plan, host_experts, pages, copy_stream, after=None, copy_done=None):
    """Copy experts (pinned host tensors of 3*f*d bf16: W1|W3|W2) into pool pages
    (pages[i] = the three pages of expert i) on `copy_stream`, after `after` and before
    `copy_done` (torch.cuda.Event or None)."""
    n = len(host_experts)
    ptrs = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in host_experts])
    flat = [int(p) for row in pages for p in row]
    if len(flat) != 3 * n:
        raise ValueError("pages must hold three pages per expert")
    pg = (ctypes.c_int32 * max(3 * n, 1))(*flat)
    wait = _event(after) if (after is not None and after.cuda_event != 0) else None
    _lib.check(_lib.load().pmoe_fill_pages_async(plan._h, int(n), ptrs, pg, _stream(copy_stream),
                                                 wait, _event(copy_done, copy_stream)))


def device_pointers(host_tensors) -> torch.Tensor:
    """Device-readable addresses of pinned host tensors (None stays 0), as an int64 tensor on
    the current device: the host_experts table of copy_in_missing."""
    n = len(host_tensors)
    src = (ctypes.c_void_p * max(n, 1))(*[(t.data_ptr() if t is not None else None) for t in host_tensors])
    dst = (ctypes.c_void_p * max(n, 1))()
    _lib.check(_lib.load().pmoe_device_pointers(int(n), src, dst))
    return torch.tensor([int(p or 0) for p in dst[:n]], dtype=torch.int64, device="cuda")


def copy_in_missing(plan: Plan, logits, buf_slot, buf: int, host_table, missed, stream=None):
    """Bring the routed experts marked absent (buf_slot == -2) into free slots of load buffer
    `buf` on `stream` (pmoe_copy_in_missing); buf_slot (device int32 [E]) is updated in place and
    missed (device int32 [1 + 2E]) lists what was copied."""
    _lib.check(_lib.load().pmoe_copy_in_missing(plan._h, _ptr(logits), int(logits.shape[0]),
                                                _ptr(buf_slot), int(buf), _ptr(host_table),
                                                _ptr(missed), _stream(stream)))


def wait_event(event, timeout_ms: int) -> bool:
    """True when `event` completed within timeout_ms, False on timeout (host polling)."""
    if event.cuda_event == 0:
        return True   # never recorded: nothing pending
    st = _lib.load().pmoe_wait_event(ctypes.c_void_p(event.cuda_event), int(timeout_ms))
    if st == _lib.ERR_TIMEOUT:
        return False
    _lib.check(st)
    return True

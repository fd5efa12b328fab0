"""ctypes declarations for libpmoe.so (include/pmoe.h).  Marshalling only.

The library must have been built (``paged_moe_expert_gb300.build.build()``); a missing library
is an error, never a reason to compute anything elsewhere.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
SZ = ctypes.c_size_t

STATUS = {0: "PMOE_OK", 1: "PMOE_ERR_INVALID_ARG", 2: "PMOE_ERR_PAGE_OOB", 3: "PMOE_ERR_SLOT_OOB",
          4: "PMOE_ERR_UNSUPPORTED", 5: "PMOE_ERR_CUDA", 6: "PMOE_ERR_TIMEOUT",
          7: "PMOE_ERR_WORKSPACE"}
OK, ERR_INVALID_ARG, ERR_PAGE_OOB, ERR_SLOT_OOB, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, \
    ERR_WORKSPACE = range(8)
PATH_AUTO, PATH_STREAM, PATH_TC, PATH_TC_DECODE, PATH_TC2, PATH_FUSED, PATH_SLICE = 0, 1, 2, 3, 4, 5, 6


class LayerDesc(ctypes.Structure):
    _fields_ = [("d", I32), ("f", I32), ("num_experts", I32), ("top_k", I32),
                ("renormalize", I32), ("num_shared_chunks", I32), ("slots_per_buffer", I32)]


class RoutingView(ctypes.Structure):
    _fields_ = [("path", I32), ("tokens", I32), ("block_m", I32), ("top_k", I32), ("ids", I64),
                ("weights", I64), ("sorted_ids", I64), ("block_expert", I64), ("inv", I64),
                ("meta", I64), ("block_rows", I64), ("units", I64), ("active", I64)]


# name -> (restype, argtypes); mirrors include/pmoe.h
SIGNATURES = {
    "pmoe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pmoe_last_error": (ctypes.c_char_p, []),
    "pmoe_plan_create": (ctypes.c_int, [ctypes.POINTER(LayerDesc), P, I64, P, P, ctypes.POINTER(P)]),
    "pmoe_plan_destroy": (ctypes.c_int, [P]),
    "pmoe_plan_set_path": (ctypes.c_int, [P, I32]),
    "pmoe_plan_last_run": (ctypes.c_int, [P, ctypes.POINTER(I32), ctypes.POINTER(I32),
                                          ctypes.POINTER(I32)]),
    "pmoe_plan_set_profile_events": (ctypes.c_int, [P, ctypes.POINTER(P), I32]),
    "pmoe_workspace_size": (SZ, [ctypes.POINTER(LayerDesc), I32]),
    "moe_paged_forward": (ctypes.c_int, [P, P, I32, P, I32, P, P, P, P, SZ, P]),
    "moe_contig_forward": (ctypes.c_int, [P, P, I32, P, I32, P, P, SZ, P]),
    "pmoe_plan_routing_view": (ctypes.c_int, [P, I32, ctypes.POINTER(RoutingView)]),
    "moe_paged_forward_noalloc": (ctypes.c_int, [ctypes.POINTER(LayerDesc), P, I64, P, P, P, I32, P,
                                                  I32, P, P, P, P, P]),
    "pmoe_prefetch_async": (ctypes.c_int, [P, I32, I32, ctypes.POINTER(P), ctypes.POINTER(I32), P, P, P]),
    "pmoe_fill_pages_async": (ctypes.c_int, [P, I32, ctypes.POINTER(P), P, P, P, P]),
    "pmoe_wait_event": (ctypes.c_int, [P, I32]),
    "pmoe_copy_in_missing": (ctypes.c_int, [P, P, I32, P, I32, P, P, P]),
    "pmoe_device_pointers": (ctypes.c_int, [I32, ctypes.POINTER(P), ctypes.POINTER(P)]),
    "pmoe_get_device_error": (ctypes.c_int, [P, I32, ctypes.POINTER(I32), P]),
    "pmoe_route": (ctypes.c_int, [P, I32, I32, I32, I32, P, P, P]),
    "pmoe_align": (ctypes.c_int, [P, I32, I32, I32, I32, I32, P, P, P, P, P, P]),
    "pmoe_align_scratch_size": (SZ, []),
    "pmoe_vmm_granularity": (ctypes.c_int, [I32, ctypes.POINTER(SZ)]),
    "pmoe_vmm_create": (ctypes.c_int, [I32, SZ, I64, I64, ctypes.POINTER(P)]),
    "pmoe_vmm_destroy": (ctypes.c_int, [P]),
    "pmoe_vmm_pointers": (ctypes.c_int, [P, ctypes.POINTER(P), ctypes.POINTER(P)]),
    "pmoe_vmm_map": (ctypes.c_int, [P, I64, P, P]),
    "pmoe_vmm_unmap": (ctypes.c_int, [P, I64, P, P, I32]),
    "pmoe_vmm_lookup": (ctypes.c_int, [P, P]),
    "pmoe_exp_encode_bound": (SZ, [I64]),
    "pmoe_exp_encode": (ctypes.c_int, [P, I64, P, SZ, ctypes.POINTER(SZ)]),
    "pmoe_exp_decode_async": (ctypes.c_int, [I32, I64, ctypes.POINTER(P), P, ctypes.POINTER(P), P, P]),
    "pmoe_tiers_create": (ctypes.c_int, [I64, I64, I64, I64, I64, ctypes.POINTER(P)]),
    "pmoe_tiers_destroy": (ctypes.c_int, [P]),
    "pmoe_tiers_alloc": (ctypes.c_int, [P, I32, I64, ctypes.POINTER(I64)]),
    "pmoe_tiers_free": (ctypes.c_int, [P, I32, I64]),
    "pmoe_tiers_stats": (ctypes.c_int, [P, P]),
    "pmoe_adjuster_create": (ctypes.c_int, [I32, I32, P, I32, P, I64, ctypes.POINTER(P)]),
    "pmoe_adjuster_destroy": (ctypes.c_int, [P]),
    "pmoe_adjuster_decide": (ctypes.c_int, [P, I32, I32, P, ctypes.POINTER(I32)]),
    "pmoe_adjuster_end_forward": (ctypes.c_int, [P]),
    "pmoe_adjuster_lend": (ctypes.c_int, [P, I32, P]),
    "pmoe_adjuster_give_back": (ctypes.c_int, [P, I32, P]),
    "pmoe_adjuster_state": (ctypes.c_int, [P, ctypes.POINTER(I64), P]),
    "pmoe_adjuster_page_table": (ctypes.c_int, [P, I32, P]),
}

_lock = threading.Lock()
_lib = None


class PmoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), msg))
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load():
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError("libpmoe.so is not built (%s); run "
                                   "`python -m paged_moe_expert_gb300.build`" % path)
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def check(status: int):
    if status != OK:
        lib = load()
        raise PmoeError(status, lib.pmoe_last_error().decode(errors="replace"))

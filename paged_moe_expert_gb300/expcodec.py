"""Python binding of libpmoe's exponent-only Huffman codec for bf16 expert pages (marshalling only).

FluxMoE (awesome-system-papers, section "核心方法"): sign and mantissa stay as they are, the
exponent is Huffman-coded; the host encodes once, the GPU decodes before the weights are read
(here: into a load-buffer slot or pool page, one thread per 256 values).
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib


def encode(values) -> np.ndarray:
    """bf16 bit patterns (any shape) -> the compressed blob as uint8."""
    v = np.ascontiguousarray(values, dtype=np.uint16).reshape(-1)
    lib = _lib.load()
    cap = lib.pmoe_exp_encode_bound(v.size)
    out = np.empty(cap, dtype=np.uint8)
    nb = ctypes.c_size_t()
    _lib.check(lib.pmoe_exp_encode(v.ctypes.data if v.size else None, v.size, out.ctypes.data, cap,
                                   ctypes.byref(nb)))
    return out[:nb.value].copy()


def decode_async(blobs, n: int, dsts, device_error=None, stream=None):
    """Decode device blobs (uint8 tensors) of n values each into device tensors (n bf16 each),
    at most 128 per call, on `stream`."""
    k = len(blobs)
    if k != len(dsts):
        raise ValueError("one destination per blob")
    src = (ctypes.c_void_p * max(k, 1))(*[b.data_ptr() for b in blobs])
    nbytes = np.asarray([b.numel() * b.element_size() for b in blobs] or [0], dtype=np.int64)
    dst = (ctypes.c_void_p * max(k, 1))(*[d.data_ptr() for d in dsts])
    if stream is None:
        stream = torch.cuda.current_stream()
    _lib.check(_lib.load().pmoe_exp_decode_async(
        k, int(n), src, nbytes.ctypes.data, dst,
        None if device_error is None else ctypes.c_void_p(device_error.data_ptr()),
        ctypes.c_void_p(stream.cuda_stream)))

"""CPU oracle for the paged fused-MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference legs of
``bench.py`` may import this package.  The product library never does, and shares no code with
it: the arithmetic lives in ``pmoe_oracle.c`` (plain C, IEEE fp64), this module only marshals
numpy arrays into it through ctypes and compiles it on first use with the host C compiler.

Source of the semantics: Rimuru (paper-daily.com/en), section "Expert weights are scattered
across pages. How does the kernel read them?" -- the paged kernel computes the ordinary MoE
layer, only reading expert rows through the page rule addr_e(n,t) = B_P + p_e(n)*f*d +
(n mod f)*d + t; section "The adjuster" -- an expert is three pages: gate W1, up W3, down W2.
Every function below therefore works on contiguous per-expert arrays and never sees a page.

Pins (all in ``tests/test_oracle.py``): the bf16 rounding against binary32 rounding and hand
tie cases; routing and align against brute-force ``sorted``; the FFN against hand-computed
two-expert values (``tests/golden/two_expert.json``), the textbook SwiGLU MLP (E=1, k=1) and
the dense-mixture closed form (k=E); the per-token loop against the grouped-by-expert loop.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pmoe_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle_pmoe.so")
# A pre-built copy to load instead (used only by the mutation test, which plants mistakes in a
# copy of the C source and checks that the pins catch them).
_OVERRIDE = os.environ.get("PMOE_ORACLE_LIB")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable flags: no -march)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Layer(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("renormalize", ctypes.c_int32), ("S", ctypes.c_int32),
                ("W1", ctypes.c_void_p), ("W3", ctypes.c_void_p), ("W2", ctypes.c_void_p),
                ("W1s", ctypes.c_void_p), ("W3s", ctypes.c_void_p), ("W2s", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_OVERRIDE if _OVERRIDE else build())
            P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            lib.orc_bf16_to_f64_vec.argtypes = [P, P, I64]
            lib.orc_f64_to_bf16_vec.argtypes = [P, P, I64]
            lib.orc_route.argtypes = [I, I, I, I, P, P, P]
            lib.orc_align.argtypes = [I, I, I, I, I, P, ctypes.c_int32, P, P, P, P]
            lib.orc_expert_ffn.argtypes = [I, I, P, P, P, P, I, P]
            lib.orc_expert_ffn.restype = None
            lib.orc_forward.argtypes = [ctypes.POINTER(_Layer), I, P, P, I, I, P, P, P, P]
            lib.orc_forward_grouped.argtypes = [ctypes.POINTER(_Layer), I, I, P, P, I, P, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------------------------
# bf16
# ---------------------------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().orc_bf16_to_f64_vec(_p(b), _p(out), b.size)
    return out


def f64_to_bf16(x) -> np.ndarray:
    a = _c(x, np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().orc_f64_to_bf16_vec(_p(a), _p(out), a.size)
    return out


# ---------------------------------------------------------------------------------------------
# steps
# ---------------------------------------------------------------------------------------------

def route(logits, k: int, renormalize: bool):
    """logits [T,E] fp32 -> (ids [T,k] int32, w [T,k] fp64)."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    rc = _load().orc_route(T, E, k, int(bool(renormalize)), _p(lg), _p(ids), _p(w))
    if rc:
        raise ValueError("orc_route: bad sizes (T=%d E=%d k=%d)" % (T, E, k))
    return ids, w


def align(ids, E: int, S: int, BM: int):
    """ids [T,k] -> dict(sorted_ids, block_expert, inv, n_padded).  Shared pairs follow the
    routed ones (pair T*k + s*T + t goes to expert E+s); pad entries hold T*(k+S)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    NP = T * (k + S)
    cap = NP + (E + S) * BM
    sorted_ids = np.empty(cap, np.int32)
    block_expert = np.empty(cap // BM + 1, np.int32)
    inv = np.empty(NP, np.int32)
    npad = np.zeros(1, np.int32)
    rc = _load().orc_align(T, k, E, S, BM, _p(ids), cap, _p(sorted_ids), _p(block_expert),
                           _p(inv), _p(npad))
    if rc:
        raise ValueError("orc_align failed (rc=%d)" % rc)
    n = int(npad[0])
    return {"sorted_ids": sorted_ids[:n].copy(), "block_expert": block_expert[: n // BM].copy(),
            "inv": inv, "n_padded": n}


def expert_ffn(W1, W3, W2, x, round_h: bool = True) -> np.ndarray:
    """One expert on one token: W1,W3 [f,d], W2 [d,f], x [d] (bf16 bits) -> y [d] fp64."""
    W1, W3, W2, x = (_c(a, np.uint16) for a in (W1, W3, W2, x))
    f, d = W1.shape
    assert W3.shape == (f, d) and W2.shape == (d, f) and x.shape == (d,)
    y = np.empty(d, np.float64)
    _load().orc_expert_ffn(d, f, _p(W1), _p(W3), _p(W2), _p(x), int(bool(round_h)), _p(y))
    return y


class Layer:
    """Contiguous per-expert weights (bf16 bit patterns as uint16).

    W1, W3: [E, f, d]; W2: [E, d, f]; shared (optional): W1s, W3s [S*f, d], W2s [d, S*f]."""

    def __init__(self, W1, W3, W2, top_k, renormalize, W1s=None, W3s=None, W2s=None, S=0):
        self.W1, self.W3, self.W2 = (_c(a, np.uint16) for a in (W1, W3, W2))
        self.E, self.f, self.d = self.W1.shape
        assert self.W3.shape == self.W1.shape and self.W2.shape == (self.E, self.d, self.f)
        self.k, self.renormalize, self.S = int(top_k), bool(renormalize), int(S)
        if self.S:
            self.W1s, self.W3s, self.W2s = (_c(a, np.uint16) for a in (W1s, W3s, W2s))
            fs = self.S * self.f
            assert self.W1s.shape == (fs, self.d) and self.W2s.shape == (self.d, fs)
        else:
            self.W1s = self.W3s = self.W2s = None

    def _struct(self):
        return _Layer(self.d, self.f, self.E, self.k, int(self.renormalize), self.S,
                      _p(self.W1), _p(self.W3), _p(self.W2), _p(self.W1s), _p(self.W3s),
                      _p(self.W2s))

    def forward(self, hidden, logits, round_h=True, nthreads=None):
        """hidden [T,d] bf16 bits, logits [T,E] fp32 -> dict(out_bf16 [T,d] uint16,
        out_f64 [T,d] (the sum before the output rounding), ids [T,k], w [T,k])."""
        hidden = _c(hidden, np.uint16)
        logits = _c(logits, np.float32)
        T = hidden.shape[0]
        assert hidden.shape == (T, self.d) and logits.shape == (T, self.E)
        out_f64 = np.empty((T, self.d), np.float64)
        out_bf16 = np.empty((T, self.d), np.uint16)
        ids = np.empty((T, self.k), np.int32)
        w = np.empty((T, self.k), np.float64)
        if nthreads is None:
            nthreads = os.cpu_count() or 1
        st = self._struct()
        rc = _load().orc_forward(ctypes.byref(st), T, _p(hidden), _p(logits), int(bool(round_h)),
                                 int(nthreads), _p(out_f64), _p(out_bf16), _p(ids), _p(w))
        if rc:
            raise ValueError("orc_forward failed")
        return {"out_bf16": out_bf16, "out_f64": out_f64, "ids": ids, "w": w}

    def forward_grouped(self, hidden, logits, BM=4, round_h=True):
        hidden = _c(hidden, np.uint16)
        logits = _c(logits, np.float32)
        T = hidden.shape[0]
        out_f64 = np.empty((T, self.d), np.float64)
        out_bf16 = np.empty((T, self.d), np.uint16)
        st = self._struct()
        rc = _load().orc_forward_grouped(ctypes.byref(st), T, BM, _p(hidden), _p(logits),
                                         int(bool(round_h)), _p(out_f64), _p(out_bf16))
        if rc:
            raise ValueError("orc_forward_grouped failed")
        return {"out_bf16": out_bf16, "out_f64": out_f64}

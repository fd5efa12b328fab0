"""CPU-only checks of the C-ABI library: it builds, loads, exports every function that
include/pmoe.h declares, and validates arguments on the host before touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "return")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("moe_paged_forward", "moe_contig_forward", "pmoe_prefetch_async",
                 "pmoe_plan_create", "pmoe_route", "pmoe_align", "pmoe_wait_event"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)
        assert n in _lib.SIGNATURES, "binding lacks %s" % n


def test_workspace_size_is_host_only_and_monotone(lib):
    d = pm.make_desc(2048, 1408, 60, 4, False, 4, 15)
    sizes = [pm.workspace_size(d, T) for T in (0, 1, 16, 128, 1024, 4096)]
    assert all(s > 0 for s in sizes)
    assert sizes == sorted(sizes)
    assert pm.workspace_size(pm.make_desc(2048, 1408, 60, 0, False), 16) == 0  # k = 0
    assert pm.workspace_size(d, -1) == 0


@pytest.mark.parametrize("shape", [(256, 128, 8, 2, 0), (2048, 1408, 60, 4, 4), (2048, 512, 512, 10, 1),
                                   (4096, 14336, 8, 2, 0)])
def test_workspace_size_covers_every_smaller_call(lib, shape):
    """pmoe_workspace_size(desc, n) is enough for any call of up to n tokens: the decode kernels'
    scratch exists only up to 16 and 32 tokens, so a call of that size can need more than a larger
    one, and the size for n must cover it."""
    d, f, E, k, S = shape
    desc = pm.make_desc(d, f, E, k, True, S, 4)
    own = {T: pm.workspace_size(desc, T) for T in range(0, 70)}
    for n in range(0, 70):
        need = max(own[T] for T in range(0, n + 1))
        assert pm.workspace_size(desc, n) >= need, (n, pm.workspace_size(desc, n), need)


def test_host_validation_statuses(lib):
    h = ctypes.c_void_p()
    bad = pm.make_desc(2048, 1408, 60, 61, False)          # k > E
    assert lib.pmoe_plan_create(ctypes.byref(bad), ctypes.c_void_p(256), 10, None, None,
                                ctypes.byref(h)) == _lib.ERR_INVALID_ARG
    odd = pm.make_desc(100, 128, 8, 2, True)               # d % 64 != 0
    assert lib.pmoe_plan_create(ctypes.byref(odd), ctypes.c_void_p(256), 10, None, None,
                                ctypes.byref(h)) == _lib.ERR_UNSUPPORTED
    assert lib.moe_paged_forward(None, None, 1, None, 2, None, None, None, None, 0, None) == \
        _lib.ERR_INVALID_ARG
    assert lib.pmoe_prefetch_async(None, 0, 1, None, None, None, None, None) == _lib.ERR_INVALID_ARG
    assert lib.pmoe_route(None, 4, 0, 1, 0, None, None, None) == _lib.ERR_INVALID_ARG
    assert lib.pmoe_align(None, 4, 2, 8, 0, 3, None, None, None, None, None, None) == _lib.ERR_INVALID_ARG
    assert lib.pmoe_wait_event(None, 10) == _lib.ERR_INVALID_ARG
    assert lib.pmoe_plan_set_path(None, 0) == _lib.ERR_INVALID_ARG
    assert lib.pmoe_plan_destroy(None) == _lib.OK
    assert lib.pmoe_status_string(_lib.ERR_PAGE_OOB) == b"page index out of range"
    assert b"k" in lib.pmoe_last_error() or lib.pmoe_last_error() != b""


def test_noalloc_refuses_bad_arguments_before_any_device_work(lib):
    """The allocation-free forward checks its arguments on the host first: these calls pass
    made-up device addresses and must return before touching a GPU."""
    fn = lib.moe_paged_forward_noalloc
    A = ctypes.c_void_p(0x100000)   # 16-byte aligned stand-ins, never dereferenced

    def call(desc, T=4, buf0=A, buf1=A, err=A, top_k=None):
        k = desc.top_k if top_k is None else top_k
        return fn(ctypes.byref(desc), A, 32, buf0, buf1, A, T, A, k, A, A, A, err, None)

    tiny = pm.make_desc(256, 128, 8, 2, True, 0, 2)
    assert call(pm.make_desc(256, 128, 8, 9, True, 0, 2)) == _lib.ERR_INVALID_ARG       # k > E
    assert call(pm.make_desc(100, 128, 8, 2, True, 0, 2)) == _lib.ERR_UNSUPPORTED       # d % 64
    assert call(pm.make_desc(32768, 128, 8, 2, True, 0, 2)) == _lib.ERR_UNSUPPORTED     # d too large
    assert call(tiny, buf0=ctypes.c_void_p(0x100008)) == _lib.ERR_INVALID_ARG           # misaligned buffer
    assert b"aligned" in lib.pmoe_last_error()
    assert call(tiny, buf1=ctypes.c_void_p(0x100004)) == _lib.ERR_INVALID_ARG
    assert call(tiny, err=None) == _lib.ERR_INVALID_ARG                                 # no error word
    assert b"device_error" in lib.pmoe_last_error()
    assert call(tiny, top_k=1) == _lib.ERR_INVALID_ARG
    q15 = pm.make_desc(2048, 1408, 60, 4, False, 4, 15)
    assert call(q15, T=512) == _lib.ERR_WORKSPACE                                       # beyond the scratch
    assert b"scratch" in lib.pmoe_last_error()
    assert call(tiny, T=0) == _lib.OK                                                   # nothing to do


def test_routing_view_needs_a_forward_call(lib):
    v = _lib.RoutingView()
    assert lib.pmoe_plan_routing_view(None, 1, ctypes.byref(v)) == _lib.ERR_INVALID_ARG

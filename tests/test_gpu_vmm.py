"""The remapped contiguous view (FluxMoE's PagedTensor, awesome-system-papers, "核心方法"): the
contiguous forward reading a virtual range whose pages are mapped onto scattered physical blocks
must give bit-identical outputs to the page-table forward over the same blocks and to the
contiguous forward over an ordinary allocation; remapping a virtual page moves what the
contiguous kernel reads; the mapping calls reject what would break the view's invariants."""
import numpy as np
import pytest
import torch

import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import _lib
from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300 import synthetic as syn
from paged_moe_expert_gb300 import vmm as vm

from helpers import assert_close, oracle_layer, out_bits

pytestmark = pytest.mark.gpu


def setup(cfg, w, extra_blocks=5, seed=0):
    """Blocks in a random order: page_table[e][j] = block of expert e's matrix j; the view maps
    virtual page 3e+j onto it."""
    E, S, f, d = cfg.E, cfg.S, cfg.f, cfg.d
    n_pages = 3 * (E + S)
    vmm = vm.VmmView(f * d * 2, n_pages + extra_blocks, n_pages)
    rng = np.random.default_rng(seed)
    pt = rng.permutation(n_pages + extra_blocks)[:n_pages].astype(np.int32).reshape(E + S, 3)
    desc = pm.make_desc(d, f, E, cfg.k, cfg.renormalize, S, 1)
    plan_blocks = pm.Plan(desc, vmm.blocks, vmm.n_blocks)
    host = [torch.from_numpy(pl.pack_expert(w, e, E, f).view(np.int16)).pin_memory() for e in range(E + S)]
    s = torch.cuda.Stream()
    pm.fill_pages_async(plan_blocks, host, pt.tolist(), s)
    s.synchronize()
    vm.map_experts(vmm, pt)
    assert (vmm.lookup() >= 0).all()          # every page the kernel can read is mapped
    plan_view = pm.Plan(desc, vmm.view, n_pages)
    return vmm, pt, plan_blocks, plan_view, host, desc


@pytest.mark.parametrize("T", [5, 300])
def test_remapped_view_equals_page_table_and_contiguous(T):
    if 1024 * 1024 * 2 % vm.granularity() != 0:
        pytest.skip("2 MiB pages are not a multiple of this device's VMM granularity")
    cfg = syn.custom_config("vmm", d=1024, f=1024, E=8, k=2, S=1, n_buffered=0)
    w = syn.make_weights(cfg)
    vmm, pt, plan_blocks, plan_view, host, desc = setup(cfg, w)
    h, lg = syn.make_tokens(cfg, T)
    hd, ld = pl._bf16(h).cuda(), torch.from_numpy(lg).cuda()
    ptd = torch.from_numpy(pt).cuda()
    bs = torch.full((cfg.E,), -1, dtype=torch.int32, device="cuda")
    a = plan_blocks.forward(hd, ld, ptd, bs)
    b = plan_view.contig_forward(hd, ld)
    cw = pl.contiguous_weights(cfg, w)
    c = pm.Plan(desc, cw, 3 * (cfg.E + cfg.S)).contig_forward(hd, ld)
    torch.cuda.synchronize()
    assert plan_blocks.device_error() == 0
    assert np.array_equal(out_bits(a), out_bits(b))
    assert np.array_equal(out_bits(a), out_bits(c))
    assert_close(out_bits(b), oracle_layer(cfg, w).forward(h, lg)["out_bf16"], "remapped view")
    del plan_view, plan_blocks
    vmm.close()


def test_remapping_moves_what_the_contiguous_kernel_reads():
    if 1024 * 1024 * 2 % vm.granularity() != 0:
        pytest.skip("2 MiB pages are not a multiple of this device's VMM granularity")
    cfg = syn.custom_config("vmm2", d=1024, f=1024, E=8, k=2, S=0, n_buffered=0)
    w = syn.make_weights(cfg)
    vmm, pt, plan_blocks, plan_view, host, desc = setup(cfg, w, seed=3)
    h, lg = syn.make_tokens(cfg, 40)
    hd, ld = pl._bf16(h).cuda(), torch.from_numpy(lg).cuda()
    done = torch.cuda.Event()
    plan_view.contig_forward(hd, ld)
    done.record()
    # expert 0 now reads expert 1's blocks (each virtual page still maps exactly one block)
    vmm.unmap([0, 1, 2], readers_done=done)
    assert (vmm.lookup()[:3] == -1).all()
    vmm.map([0, 1, 2], pt[1])
    pt2 = pt.copy()
    pt2[0] = pt[1]
    bs = torch.full((cfg.E,), -1, dtype=torch.int32, device="cuda")
    want = plan_blocks.forward(hd, ld, torch.from_numpy(pt2).cuda(), bs)
    got = plan_view.contig_forward(hd, ld)
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(got), out_bits(want))
    del plan_view, plan_blocks
    vmm.close()


def test_mapping_calls_keep_the_invariants():
    g = vm.granularity()
    assert g > 0
    with pytest.raises(_lib.PmoeError, match="UNSUPPORTED"):
        vm.VmmView(g + 4096, 2, 2)                 # not a multiple of the granularity
    v = vm.VmmView(g, 3, 4)
    v.map([0, 1], [2, 2])                          # one block under two pages: allowed (aliases)
    with pytest.raises(_lib.PmoeError, match="already mapped"):
        v.map([1], [0])                            # a page maps at most one block
    with pytest.raises(_lib.PmoeError, match="listed twice"):
        v.map([2, 2], [0, 1])
    with pytest.raises(_lib.PmoeError, match="out of range"):
        v.map([4], [0])
    with pytest.raises(_lib.PmoeError, match="not mapped"):
        v.unmap([3])
    assert v.lookup().tolist() == [2, 2, -1, -1]
    v.unmap([0, 1])
    assert v.lookup().tolist() == [-1, -1, -1, -1]
    v.close()

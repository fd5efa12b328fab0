"""GPU decoder of the exponent-only Huffman codec (FluxMoE, awesome-system-papers, "核心方法"):
decoding gives back every bit pattern of the original pages (several per launch, ragged sizes,
special values), a blob whose header does not match is reported on the device word, and expert
pages decoded into a load buffer feed the layer forward with the same output as resident pages."""
import numpy as np
import pytest
import torch

import paged_moe_expert_gb300 as pm
from paged_moe_expert_gb300 import expcodec as nc
from paged_moe_expert_gb300 import pool as pl
from paged_moe_expert_gb300 import synthetic as syn

from helpers import out_bits

pytestmark = pytest.mark.gpu

SPECIALS = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x807F], dtype=np.uint16)


def bf16_normal(rng, n, scale):
    w = (rng.standard_normal(n) * scale).astype(np.float32).view(np.uint32)
    return ((w + 0x7FFF + ((w >> 16) & 1)) >> 16).astype(np.uint16)


def to_dev(a: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    assert t.data_ptr() % 16 == 0
    return t


@pytest.mark.parametrize("n", [1, 8, 255, 256, 1000, 65536, 65536 * 3 + 77, 1408 * 2048])
def test_decode_is_bit_exact(n):
    rng = np.random.default_rng(n)
    pages = []
    for i in range(3):
        if i == 2:
            v = rng.integers(0, 1 << 16, size=n, dtype=np.uint16)     # every exponent value
        else:
            v = bf16_normal(rng, n, [0.02, 1.0][i])
        v[: min(n, SPECIALS.size)] = SPECIALS[: min(n, SPECIALS.size)]
        pages.append(v)
    blobs = [to_dev(nc.encode(v)) for v in pages]
    out = [torch.full((n,), 0x5555, dtype=torch.int16, device="cuda") for _ in pages]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    nc.decode_async(blobs, n, out, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for v, o in zip(pages, out):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), v)


def test_mismatched_header_is_reported():
    rng = np.random.default_rng(1)
    good = bf16_normal(rng, 5000, 0.02)
    bad = bf16_normal(rng, 4000, 0.02)
    b_good = to_dev(nc.encode(good))
    b_bad = np.zeros(len(nc.encode(good)) + 64, dtype=np.uint8)
    enc = nc.encode(bad)
    b_bad[: enc.size] = enc                                  # a blob of 4000 values, sized like 5000
    out = [torch.zeros(5000, dtype=torch.int16, device="cuda") for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    nc.decode_async([b_good, to_dev(b_bad)], 5000, out, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1                               # PMOE_ERR_INVALID_ARG
    assert np.array_equal(out[0].cpu().numpy().view(np.uint16), good)
    assert not out[1].any()


def test_decoded_load_buffer_feeds_the_forward():
    cfg = syn.custom_config("codec", d=256, f=256, E=8, k=2, S=1, n_buffered=0)
    w = syn.make_weights(cfg)
    E, S, f, d = cfg.E, cfg.S, cfg.f, cfg.d
    slots = 4
    desc = pm.make_desc(d, f, E, cfg.k, cfg.renormalize, S, slots)
    bufs = pl.new_load_buffers(slots, f, d)
    # experts 0..3 compressed in device memory; the rest in pool pages
    pool = pl.new_pool(3 * (E + S), f, d)
    cw = pl.contiguous_weights(cfg, w)
    pool.copy_(cw)
    pt = torch.arange(3 * (E + S), dtype=torch.int32).reshape(E + S, 3).cuda()
    plan = pm.Plan(desc, pool, 3 * (E + S), bufs)
    page = f * d
    blobs, dsts = [], []
    for s_, e in enumerate(range(4)):
        for j, m in enumerate(pl.expert_matrices(w, e, E, f)):
            blobs.append(to_dev(nc.encode(m)))
            dsts.append(bufs[1][(3 * s_ + j) * page:(3 * s_ + j + 1) * page])
    nc.decode_async(blobs, page, dsts)
    bs = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    bs[:4] = slots + torch.arange(4, dtype=torch.int32, device="cuda")     # buffer 1, slots 0..3
    for T in (3, 100):
        h, lg = syn.make_tokens(cfg, T)
        hd, ld = pl._bf16(h).cuda(), torch.from_numpy(lg).cuda()
        a = plan.forward(hd, ld, pt, bs)
        b = plan.forward(hd, ld, pt, torch.full((E,), -1, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert plan.device_error() == 0
        assert np.array_equal(out_bits(a), out_bits(b))

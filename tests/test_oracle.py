"""Pins for the CPU oracle: every check here compares it with something other than itself --
binary32 rounding, hand-derived closed forms, numpy/scipy textbook formulas, brute force.

Sources: Rimuru (paper-daily.com/en), "Expert weights are scattered across pages. How does the
kernel read them?" (gate W1 / up W3 pages, first vs second half of the output columns) and
"The adjuster" (three pages per expert: W1, W3, W2).  Routing, sort/pad, SiLU-and-mul and the
weighted top-k combine are the ordinary MoE layer steps those sections leave unchanged.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_moe_expert_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(x):
    return syn.to_bf16_bits(np.asarray(x, np.float32))


def f64(b):
    return syn.bf16_bits_to_f32(b).astype(np.float64)


# --------------------------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------------------------

def test_bf16_matches_binary32_rounding():
    # For values exactly representable in binary32, one RNE step from fp64 must equal torch's
    # fp32 -> bf16 conversion (round to nearest even).
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        rng.standard_normal(2000) * 1e-39]).astype(np.float32)
    ours = oracle.f64_to_bf16(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("value,expect", [
    (1.0, 0x3F80), (-2.0, 0xC000), (1.0 + 2.0 ** -8, 0x3F80),          # tie -> even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),                                      # tie -> even (up)
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),                             # above the tie -> up
    (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000), (3 * 2.0 ** -134, 0x0002),  # subnormals
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),                             # largest finite
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),                             # tie at the top -> inf
    (-0.0, 0x8000), (float("inf"), 0x7F80),
])
def test_bf16_special_cases(value, expect):
    assert int(oracle.f64_to_bf16(np.array([value]))[0]) == expect


def test_bf16_widening():
    b = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000], np.uint16)
    want = [1.0, -2.0, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127, -0.0]
    assert list(oracle.bf16_to_f64(b)) == want


# --------------------------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------------------------

def brute_route(logits, k, renorm):
    T, E = logits.shape
    ids = np.array([sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k] for t in range(T)],
                   np.int32).reshape(T, k)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    w = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return ids, w


@pytest.mark.parametrize("E,k,renorm,ties", [(8, 2, True, False), (60, 4, False, False),
                                              (512, 10, True, False), (16, 5, True, True),
                                              (512, 10, False, True), (3, 3, False, True),
                                              (1, 1, True, False)])
def test_route_brute_force(E, k, renorm, ties):
    rng = np.random.default_rng(E * 100 + k)
    T = 37
    if ties:
        lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32)   # many equal logits
    else:
        lg = syn.bf16_bits_to_f32(bits(rng.standard_normal((T, E))))
    ids, w = oracle.route(lg, k, renorm)
    bids, bw = brute_route(lg, k, renorm)
    assert np.array_equal(ids, bids)
    np.testing.assert_allclose(w, bw, rtol=1e-13, atol=0)


def test_route_ties_prefer_lower_id():
    lg = np.zeros((1, 6), np.float32)
    lg[0, [1, 3, 4]] = 2.0
    ids, w = oracle.route(lg, 2, False)
    assert ids.tolist() == [[1, 3]]
    assert w[0, 0] == w[0, 1]


# --------------------------------------------------------------------------------------------
# sort + pad
# --------------------------------------------------------------------------------------------

def brute_align(ids, E, S, BM):
    T, k = ids.shape
    NP = T * (k + S)
    owner = [int(ids.reshape(-1)[i]) if i < T * k else E + (i - T * k) // T for i in range(NP)]
    order = sorted(range(NP), key=lambda i: (owner[i], i))
    rows, bexp = [], []
    for e in range(E + S):
        mine = [i for i in order if owner[i] == e]
        if not mine:
            continue
        nb = -(-len(mine) // BM)
        rows += mine + [NP] * (nb * BM - len(mine))
        bexp += [e] * nb
    inv = np.empty(NP, np.int32)
    for r, i in enumerate(rows):
        if i < NP:
            inv[i] = r
    return np.array(rows, np.int32), np.array(bexp, np.int32), inv


@pytest.mark.parametrize("T,E,k,S,BM", [(16, 8, 2, 0, 4), (37, 60, 4, 4, 16), (5, 512, 10, 1, 128),
                                         (64, 8, 2, 0, 128), (1, 60, 4, 4, 1), (0, 8, 2, 1, 16),
                                         (33, 3, 3, 2, 7)])
def test_align_brute_force_and_invariants(T, E, k, S, BM):
    rng = np.random.default_rng(T + 7 * E)
    ids = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32).reshape(T, k)
    got = oracle.align(ids, E, S, BM)
    rows, bexp, inv = brute_align(ids, E, S, BM)
    assert np.array_equal(got["sorted_ids"], rows)
    assert np.array_equal(got["block_expert"], bexp)
    NP = T * (k + S)
    if NP:
        assert np.array_equal(got["inv"], inv)
    n = got["n_padded"]
    # invariants: every pair exactly once, pads are the sentinel, each block one expert
    real = got["sorted_ids"][got["sorted_ids"] < NP]
    assert sorted(real.tolist()) == list(range(NP))
    assert int((got["sorted_ids"] == NP).sum()) == n - NP
    counts = np.bincount(ids.reshape(-1), minlength=E).tolist() + [T] * S
    assert n == sum(BM * -(-c // BM) for c in counts)
    assert n % BM == 0 and len(got["block_expert"]) == n // BM


# --------------------------------------------------------------------------------------------
# FFN and the whole layer
# --------------------------------------------------------------------------------------------

def silu(z):
    return z * scipy.special.expit(z)


def swiglu_np(W1, W3, W2, x):
    """Textbook SwiGLU MLP in float64: W2 (silu(W1 x) * (W3 x))."""
    return W2 @ (silu(W1 @ x) * (W3 @ x))


def test_two_expert_golden():
    g = json.load(open(os.path.join(GOLDEN, "two_expert.json")))
    W1, W3, W2 = (bits(np.array(g[n])) for n in ("W1", "W3", "W2"))
    L = oracle.Layer(W1, W3, W2, g["k"], g["renormalize"])
    res = L.forward(bits(np.array(g["hidden"])), np.array(g["logits"], np.float32), round_h=False)
    assert res["ids"].tolist() == g["expected_ids"]
    p0 = 1.0 / (1.0 + math.exp(-1.0))
    p1 = 1.0 - p0
    h0 = 2.0 * (1.0 / (1.0 + math.exp(-1.0)))          # 2 * silu(1)
    h1 = -1.0 / (1.0 + math.exp(1.0))                   # silu(-1)
    want = [p0 * h0 + p1 * 2.0 * h1, -p0 * h0 + p1 * 0.5 * h1]
    np.testing.assert_allclose(res["w"][0], [p0, p1], rtol=1e-15)
    np.testing.assert_allclose(res["out_f64"][0], want, rtol=1e-14)
    # with h rounded to bf16: 2*silu(1) = 1.46211... -> 1.4609375 (187/128); silu(-1) = -0.26894...
    # -> -0.26953125 (-69/256)
    res_r = L.forward(bits(np.array(g["hidden"])), np.array(g["logits"], np.float32), round_h=True)
    hr0, hr1 = 187 / 128, -69 / 256
    np.testing.assert_allclose(res_r["out_f64"][0],
                               [p0 * hr0 + p1 * 2.0 * hr1, -p0 * hr0 + p1 * 0.5 * hr1], rtol=1e-14)


def _rand_layer(rng, d, f, E, S=0, scale=0.5):
    W1 = bits(rng.standard_normal((E, f, d)) * scale)
    W3 = bits(rng.standard_normal((E, f, d)) * scale)
    W2 = bits(rng.standard_normal((E, d, f)) * scale)
    sh = {}
    if S:
        sh = dict(W1s=bits(rng.standard_normal((S * f, d)) * scale),
                  W3s=bits(rng.standard_normal((S * f, d)) * scale),
                  W2s=bits(rng.standard_normal((d, S * f)) * scale), S=S)
    return W1, W3, W2, sh


def test_single_expert_is_swiglu_mlp():
    rng = np.random.default_rng(5)
    d, f = 24, 40          # f != d so a transposed operand cannot pass
    W1, W3, W2, _ = _rand_layer(rng, d, f, 1)
    x = bits(rng.standard_normal((3, d)))
    L = oracle.Layer(W1, W3, W2, 1, True)
    res = L.forward(x, np.zeros((3, 1), np.float32), round_h=False)
    for t in range(3):
        want = swiglu_np(f64(W1[0]), f64(W3[0]), f64(W2[0]), f64(x[t]))
        np.testing.assert_allclose(res["out_f64"][t], want, rtol=1e-12, atol=1e-14)
    y = oracle.expert_ffn(W1[0], W3[0], W2[0], x[0], round_h=False)
    np.testing.assert_allclose(y, swiglu_np(f64(W1[0]), f64(W3[0]), f64(W2[0]), f64(x[0])),
                               rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("renorm", [False, True])
def test_dense_mixture_closed_form(renorm):
    # top_k = E: out = sum_e softmax(logits)_e * FFN_e(x) (+ shared), with or without
    # renormalisation (the probabilities already sum to one).
    rng = np.random.default_rng(11)
    d, f, E, S = 16, 12, 5, 2
    W1, W3, W2, sh = _rand_layer(rng, d, f, E, S)
    T = 6
    x = bits(rng.standard_normal((T, d)))
    lg = rng.standard_normal((T, E)).astype(np.float32)
    L = oracle.Layer(W1, W3, W2, E, renorm, **sh)
    res = L.forward(x, lg, round_h=False)
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    for t in range(T):
        xt = f64(x[t])
        want = sum(p[t, e] * swiglu_np(f64(W1[e]), f64(W3[e]), f64(W2[e]), xt) for e in range(E))
        want = want + swiglu_np(f64(sh["W1s"]), f64(sh["W3s"]), f64(sh["W2s"]), xt)
        np.testing.assert_allclose(res["out_f64"][t], want, rtol=1e-11, atol=1e-12)


def test_topk_selects_and_weights():
    # k < E: only the k largest logits contribute, with their softmax probability over ALL E.
    rng = np.random.default_rng(12)
    d, f, E, k = 8, 8, 6, 2
    W1, W3, W2, _ = _rand_layer(rng, d, f, E)
    x = bits(rng.standard_normal((1, d)))
    lg = np.array([[0.1, 2.0, -1.0, 1.5, 0.0, 1.5]], np.float32)  # top-2 = {1, 3} (3 beats 5)
    p = scipy.special.softmax(lg[0].astype(np.float64))
    for renorm in (False, True):
        res = oracle.Layer(W1, W3, W2, k, renorm).forward(x, lg, round_h=False)
        assert res["ids"].tolist() == [[1, 3]]
        w = np.array([p[1], p[3]])
        if renorm:
            w = w / w.sum()
        want = sum(w[j] * swiglu_np(f64(W1[e]), f64(W3[e]), f64(W2[e]), f64(x[0]))
                   for j, e in enumerate([1, 3]))
        np.testing.assert_allclose(res["out_f64"][0], want, rtol=1e-12, atol=1e-14)


def test_output_rounding_is_rne_of_sum():
    rng = np.random.default_rng(13)
    W1, W3, W2, sh = _rand_layer(rng, 32, 16, 4, 1)
    L = oracle.Layer(W1, W3, W2, 2, False, **sh)
    x = bits(rng.standard_normal((5, 32)))
    res = L.forward(x, rng.standard_normal((5, 4)).astype(np.float32))
    # the fp32 rounding route agrees with the one-step route whenever the sum is fp32-exact;
    # check the exact property instead: out_bf16 is the bf16 nearest to out_f64
    up = oracle.bf16_to_f64(res["out_bf16"])
    err = np.abs(up - res["out_f64"])
    ulp = np.ldexp(1.0, np.frexp(res["out_f64"])[1] - 8)
    assert np.all(err <= ulp / 2 + 1e-300)


def test_per_token_loop_equals_grouped_loop():
    rng = np.random.default_rng(14)
    d, f, E, k, S = 24, 16, 7, 3, 2
    W1, W3, W2, sh = _rand_layer(rng, d, f, E, S, scale=0.3)
    T = 19
    x = bits(rng.standard_normal((T, d)))
    lg = syn.bf16_bits_to_f32(bits(rng.standard_normal((T, E))))
    L = oracle.Layer(W1, W3, W2, k, True, **sh)
    for round_h in (False, True):
        a = L.forward(x, lg, round_h=round_h, nthreads=3)
        b = L.forward_grouped(x, lg, BM=4, round_h=round_h)
        np.testing.assert_allclose(a["out_f64"], b["out_f64"], rtol=1e-12, atol=1e-13)
        diff = np.abs(a["out_bf16"].astype(np.int32) - b["out_bf16"].astype(np.int32))
        assert diff.max() <= 1


def test_thread_count_does_not_change_result():
    cfg = syn.CONFIGS["tiny"]
    w = syn.make_weights(cfg)
    h, lg = syn.make_tokens(cfg, 16)
    L = oracle.Layer(w.W1, w.W3, w.W2, cfg.k, cfg.renormalize)
    a = L.forward(h, lg, nthreads=1)
    b = L.forward(h, lg, nthreads=5)
    assert np.array_equal(a["out_bf16"], b["out_bf16"])
    assert np.array_equal(a["out_f64"], b["out_f64"])

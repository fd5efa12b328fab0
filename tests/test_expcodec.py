"""Exponent-only Huffman codec for bf16 expert pages (FluxMoE, awesome-system-papers, "核心方法":
sign and mantissa kept, exponent Huffman-coded).

Part 1 pins the oracle: textbook Huffman lengths (CLRS's six-symbol example), deflate's canonical
code assignment (RFC 1951's eight-symbol example), the Kraft equality, the 12-bit length limit on
Fibonacci counts, optimality against brute force on tiny alphabets, and bit-exact round trips
including NaN, infinities, zeros and subnormals.  Part 2: the native host encoder writes the very
bytes the oracle writes.  The GPU decoder is tested in tests/test_gpu_expcodec.py.
"""
import itertools

import numpy as np
import pytest

from oracle import expcodec as ec
from paged_moe_expert_gb300 import _lib, build

CLRS = {0: 45, 1: 13, 2: 12, 3: 16, 4: 9, 5: 5}           # a..f, CLRS 16.3
CLRS_LENGTHS = {0: 1, 1: 3, 2: 3, 3: 3, 4: 4, 5: 4}


def counts_of(d):
    c = [0] * 256
    for s, k in d.items():
        c[s] = k
    return c


def test_textbook_huffman_lengths():
    L = ec.huffman_lengths(counts_of(CLRS))
    assert {s: L[s] for s in CLRS} == CLRS_LENGTHS
    assert sum(L) == sum(CLRS_LENGTHS.values())


def test_deflate_canonical_codes():
    # RFC 1951 section 3.2.2: lengths (3,3,3,3,3,2,4,4) for A..H give
    # A 010, B 011, C 100, D 101, E 110, F 00, G 1110, H 1111
    lengths = [0] * 256
    for s, L in zip(range(65, 73), (3, 3, 3, 3, 3, 2, 4, 4)):
        lengths[s] = L
    codes = ec.canonical_codes(lengths)
    assert [codes[s] for s in range(65, 73)] == [0b010, 0b011, 0b100, 0b101, 0b110, 0b00, 0b1110, 0b1111]


def test_kraft_equality_and_length_limit():
    fib = [1, 1]
    while len(fib) < 40:
        fib.append(fib[-1] + fib[-2])
    c = [0] * 256
    for i, f in enumerate(fib):
        c[100 + i] = f                                       # unlimited depth would be 39
    L = ec.huffman_lengths(c)
    assert max(L) == ec.LMAX
    assert sum(2.0 ** -x for x in L if x) == 1.0              # a complete prefix code
    one = ec.huffman_lengths(counts_of({7: 100}))
    assert one[7] == 1 and sum(one) == 1


def test_lengths_are_optimal_on_tiny_alphabets():
    rng = np.random.default_rng(0)
    for _ in range(30):
        k = int(rng.integers(2, 6))
        cnt = rng.integers(1, 50, size=k)
        L = ec.huffman_lengths(counts_of(dict(enumerate(cnt))))
        cost = sum(int(c) * L[s] for s, c in enumerate(cnt))
        best = min(sum(int(c) * l for c, l in zip(cnt, ls))
                   for ls in itertools.product(range(1, k + 1), repeat=k)
                   if sum(2.0 ** -l for l in ls) <= 1.0)
        assert cost == best


def bf16_normal(rng, n, scale=0.02):
    w = (rng.standard_normal(n) * scale).astype(np.float32).view(np.uint32)
    return ((w + 0x7FFF + ((w >> 16) & 1)) >> 16).astype(np.uint16)


SPECIALS = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x807F, 0x3F80,
                     0x7F7F, 0x0080], dtype=np.uint16)


@pytest.mark.parametrize("n", [0, 1, 7, 255, 256, 257, 1000, 4096 + 9])
def test_round_trip_is_bit_exact(n):
    rng = np.random.default_rng(n)
    v = bf16_normal(rng, n)
    v[: min(n, SPECIALS.size)] = SPECIALS[: min(n, SPECIALS.size)]
    blob = ec.encode(v)
    assert np.array_equal(ec.decode(blob), v)
    lut_o, offs_o, sm_o, bits_o = ec.layout(n)
    assert len(blob) == bits_o + 4 * ((int.from_bytes(blob[264:272], "little") + 31) // 32 + 2)


def test_round_trip_uniform_bits_and_single_symbol():
    rng = np.random.default_rng(9)
    v = rng.integers(0, 1 << 16, size=3000, dtype=np.uint16)     # every exponent value
    assert np.array_equal(ec.decode(ec.encode(v)), v)
    same = np.full(600, 0x3C00, dtype=np.uint16)                 # one exponent: 1 bit each
    blob = ec.encode(same)
    assert int.from_bytes(blob[264:272], "little") == 600
    assert np.array_equal(ec.decode(blob), same)


def test_weights_compress():
    v = bf16_normal(np.random.default_rng(3), 200000)
    ratio = len(ec.encode(v)) / (2 * v.size)
    assert 0.65 < ratio < 0.8                                    # exponent at ~3 of 8 bits


def test_planted_mistakes_are_caught():
    class Reversed:                                              # codes assigned in reverse order
        @staticmethod
        def codes(lengths):
            c = ec.canonical_codes(lengths)
            return [(1 << lengths[s]) - 1 - c[s] if lengths[s] else 0 for s in range(256)]
    lengths = [0] * 256
    for s, L in zip(range(65, 73), (3, 3, 3, 3, 3, 2, 4, 4)):
        lengths[s] = L
    assert [Reversed.codes(lengths)[s] for s in range(65, 73)] != \
        [0b010, 0b011, 0b100, 0b101, 0b110, 0b00, 0b1110, 0b1111]
    # a swapped sign/exponent split does not round-trip
    v = bf16_normal(np.random.default_rng(4), 100)
    exp, sm = ec.split(v)
    assert not np.array_equal(ec.join(sm, exp), v)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


@pytest.mark.parametrize("n", [0, 1, 255, 256, 257, 5000, 65536 + 300])
def test_native_encoder_writes_the_oracle_bytes(lib, n):
    from paged_moe_expert_gb300 import expcodec as nc
    rng = np.random.default_rng(100 + n)
    v = bf16_normal(rng, n, scale=float(rng.choice([0.02, 1.0, 1e-3])))
    v[: min(n, SPECIALS.size)] = SPECIALS[: min(n, SPECIALS.size)]
    assert bytes(nc.encode(v)) == ec.encode(v)


def test_native_encoder_length_limit(lib):
    from paged_moe_expert_gb300 import expcodec as nc
    fib = [1, 1]
    while len(fib) < 30:
        fib.append(fib[-1] + fib[-2])
    v = np.concatenate([np.full(f, (100 + i) << 7, dtype=np.uint16) for i, f in enumerate(fib)])
    np.random.default_rng(1).shuffle(v)
    blob = bytes(nc.encode(v))
    assert blob == ec.encode(v) and max(blob[:256]) == ec.LMAX

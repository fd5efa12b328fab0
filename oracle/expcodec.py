"""CPU oracle of the exponent-only Huffman codec for bf16 expert pages -- TEST INFRASTRUCTURE ONLY.

Only the test-suite may import this module.  FluxMoE (awesome-system-papers, section "核心方法",
observation 3 and the compressed GPU backend): the exponent bits of bf16 expert weights have low
entropy and the mantissa is nearly uniform, so only the exponent is Huffman-coded while sign and
mantissa stay as they are (about 20% of the storage saved), and the GPU decompresses.  The page
fixes no format; this module is the format's definition, written as plainly as possible:

* a bf16 value v splits into its exponent byte (v >> 7) & 0xFF and the byte
  (sign << 7) | mantissa = ((v >> 8) & 0x80) | (v & 0x7F); the decoder joins them back.
* code lengths: a Huffman tree over the exponent counts (the two least frequent nodes merge
  first; a tie goes to the node made earlier, leaves made first in symbol order), each symbol's
  length its depth; a single symbol gets length 1.  While the longest code exceeds 12 bits every
  nonzero count is halved (rounding up) and the tree rebuilt.
* canonical codes (the deflate rule): codes of one length are consecutive integers in symbol
  order, and the first code of length L is (first code of length L-1 + count of length L-1) << 1.
* chunks: the values are taken in groups of 65536 (the last group may be smaller); a group of v
  values has g = ceil(v / 256) chunks, its values form runs of 8 (the last may be shorter), and
  run R of the group belongs to chunk R mod g, as that chunk's run number R div g.  So a chunk
  holds at most 256 values, and the GPU threads decoding the g chunks of a group side by side
  read and write neighbouring runs.
* the exponent stream is written chunk after chunk, each chunk's codes in its run order, most
  significant code bit first, into 32-bit words filled from bit 31 down; the bit offset where
  each chunk starts is stored so chunks decode independently.
* a 4096-entry table maps the next 12 bits of the stream to (symbol | length << 8).

Byte layout of one compressed page of n values (sections 16-byte aligned):
  [0, 256)        code length of each exponent value (0: absent)
  [256, 264)      n (little-endian int64)
  [264, 272)      total bits of the exponent stream (int64)
  [272, ...)      the 4096-entry decode table, uint16 each
  then            chunk start bit offsets, uint32 [ceil(n / 256) + 1] (the last = total bits)
  then            the sign|mantissa bytes, uint8 [n], in value order
  then            the exponent stream, uint32 words (big-endian bit order inside each word),
                  followed by two zero words (a decoder may read one word past its last code)
"""
from __future__ import annotations

import heapq

import numpy as np

CHUNK = 256
LMAX = 12
LUT_BITS = 12


def _align16(x: int) -> int:
    return (x + 15) & ~15


def layout(n: int):
    """Byte offsets of the sections (table, chunk offsets, sign|mantissa, stream) for n values."""
    n_chunks = (n + CHUNK - 1) // CHUNK
    lut = 272
    offs = _align16(lut + 2 * (1 << LUT_BITS))
    sm = _align16(offs + 4 * (n_chunks + 1))
    bits = _align16(sm + n)
    return lut, offs, sm, bits


GROUP = 65536
RUN = 8


def chunk_values(n: int) -> list[list[int]]:
    """The value indices of every chunk, chunk by chunk, each in its coding order."""
    chunks = []
    for g0 in range(0, n, GROUP):
        v = min(GROUP, n - g0)
        g = (v + CHUNK - 1) // CHUNK
        runs = (v + RUN - 1) // RUN
        for c in range(g):
            vals = []
            for R in range(c, runs, g):
                start = g0 + RUN * R
                vals += list(range(start, min(start + RUN, n)))
            chunks.append(vals)
    return chunks


def huffman_lengths(counts) -> list[int]:
    """Code length of each of the 256 symbols from their counts (0 for absent symbols)."""
    counts = [int(c) for c in counts]
    while True:
        present = [s for s in range(256) if counts[s] > 0]
        lengths = [0] * 256
        if len(present) == 1:
            lengths[present[0]] = 1
            return lengths
        if not present:
            return lengths
        # heap items: (count, creation order, node); leaves are created first in symbol order
        heap = [(counts[s], i, ("leaf", s)) for i, s in enumerate(present)]
        heapq.heapify(heap)
        order = len(present)
        while len(heap) > 1:
            c1, _, a = heapq.heappop(heap)
            c2, _, b = heapq.heappop(heap)
            heapq.heappush(heap, (c1 + c2, order, ("node", a, b)))
            order += 1
        stack = [(heap[0][2], 0)]
        while stack:
            node, depth = stack.pop()
            if node[0] == "leaf":
                lengths[node[1]] = depth
            else:
                stack.append((node[1], depth + 1))
                stack.append((node[2], depth + 1))
        if max(lengths) <= LMAX:
            return lengths
        counts = [(c + 1) // 2 if c > 0 else 0 for c in counts]


def canonical_codes(lengths) -> list[int]:
    """Code of each symbol from the code lengths (deflate's canonical rule)."""
    bl_count = [0] * (LMAX + 2)
    for L in lengths:
        if L:
            bl_count[L] += 1
    next_code = [0] * (LMAX + 2)
    code = 0
    for L in range(1, LMAX + 1):
        code = (code + bl_count[L - 1]) << 1
        next_code[L] = code
    codes = [0] * 256
    for s in range(256):
        L = lengths[s]
        if L:
            codes[s] = next_code[L]
            next_code[L] += 1
    return codes


def decode_table(lengths) -> np.ndarray:
    codes = canonical_codes(lengths)
    lut = np.zeros(1 << LUT_BITS, dtype=np.uint16)
    for s in range(256):
        L = lengths[s]
        if L:
            lo = codes[s] << (LUT_BITS - L)
            lut[lo:lo + (1 << (LUT_BITS - L))] = s | (L << 8)
    return lut


def split(values: np.ndarray):
    v = np.asarray(values, dtype=np.uint16)
    exp = ((v >> 7) & 0xFF).astype(np.uint8)
    sm = (((v >> 8) & 0x80) | (v & 0x7F)).astype(np.uint8)
    return exp, sm


def join(exp: np.ndarray, sm: np.ndarray) -> np.ndarray:
    exp = exp.astype(np.uint16)
    sm = sm.astype(np.uint16)
    return ((sm & 0x80) << 8) | (exp << 7) | (sm & 0x7F)


def encode(values) -> bytes:
    v = np.ascontiguousarray(values, dtype=np.uint16).reshape(-1)
    n = v.size
    exp, sm = split(v)
    lengths = huffman_lengths(np.bincount(exp, minlength=256))
    codes = canonical_codes(lengths)
    # the exponent stream, chunk by chunk in each chunk's order, and each chunk's starting bit
    n_chunks = (n + CHUNK - 1) // CHUNK
    starts = []
    bitpos = 0
    words = []
    acc, acc_bits = 0, 0            # pending bits, most significant first
    chunks = chunk_values(n)
    assert len(chunks) == n_chunks and all(len(c) <= CHUNK for c in chunks)
    ex = exp.tolist()
    for vals in chunks:
        starts.append(bitpos)
        for i in vals:
            s = ex[i]
            L = lengths[s]
            acc = (acc << L) | codes[s]
            acc_bits += L
            bitpos += L
            while acc_bits >= 32:
                words.append((acc >> (acc_bits - 32)) & 0xFFFFFFFF)
                acc_bits -= 32
                acc &= (1 << acc_bits) - 1
    if acc_bits:
        words.append((acc << (32 - acc_bits)) & 0xFFFFFFFF)
    words += [0, 0]
    starts.append(bitpos)
    assert len(starts) == n_chunks + 1
    lut_o, offs_o, sm_o, bits_o = layout(n)
    out = bytearray(bits_o + 4 * len(words))
    out[0:256] = bytes(lengths)
    out[256:264] = int(n).to_bytes(8, "little")
    out[264:272] = int(bitpos).to_bytes(8, "little")
    out[lut_o:lut_o + 2 * (1 << LUT_BITS)] = decode_table(lengths).astype("<u2").tobytes()
    out[offs_o:offs_o + 4 * len(starts)] = np.asarray(starts, dtype="<u4").tobytes()
    out[sm_o:sm_o + n] = sm.tobytes()
    out[bits_o:] = np.asarray(words, dtype="<u4").tobytes()
    return bytes(out)


def decode(blob: bytes) -> np.ndarray:
    """Reads the stream code by code, walking the canonical code tree bit by bit (no table)."""
    lengths = list(blob[0:256])
    n = int.from_bytes(blob[256:264], "little")
    codes = canonical_codes(lengths)
    by_code = {(lengths[s], codes[s]): s for s in range(256) if lengths[s]}
    lut_o, offs_o, sm_o, bits_o = layout(n)
    sm = np.frombuffer(blob[sm_o:sm_o + n], dtype=np.uint8)
    words = np.frombuffer(blob[bits_o:], dtype="<u4")
    starts = np.frombuffer(blob[offs_o:offs_o + 4 * ((n + CHUNK - 1) // CHUNK + 1)], dtype="<u4")

    def bit(p):
        return (int(words[p >> 5]) >> (31 - (p & 31))) & 1

    exp = np.empty(n, dtype=np.uint8)
    for c, vals in enumerate(chunk_values(n)):
        p = int(starts[c])
        for i in vals:
            code, L = 0, 0
            while (L, code) not in by_code:
                code = (code << 1) | bit(p)
                p += 1
                L += 1
                assert L <= LMAX
            exp[i] = by_code[(L, code)]
    return join(exp, sm)

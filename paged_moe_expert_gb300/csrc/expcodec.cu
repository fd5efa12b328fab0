// Exponent-only Huffman compression of bf16 expert pages: the host encoder and the GPU decoder.
//
// FluxMoE (awesome-system-papers, section "核心方法", observation 3 and the compressed GPU
// backend): the exponent bits of bf16 expert weights have low entropy while the mantissa is close
// to uniform, so only the exponent is Huffman-coded and sign and mantissa are stored as they are;
// the GPU decompresses before the weights are used.  The page fixes no format; this file's is:
//
//   value v -> exponent byte (v >> 7) & 0xFF, and (sign << 7) | mantissa
//   code lengths from a Huffman tree over the exponent counts (two least frequent nodes merge
//   first, ties to the node made earlier, leaves made first in symbol order; one symbol ->
//   length 1); counts halved (rounding up) and the tree rebuilt while a code exceeds 12 bits
//   canonical codes (consecutive within a length, in symbol order)
//   chunks of at most 256 values, one per GPU thread: values in groups of 65536, a group of v
//   values has g = ceil(v/256) chunks, and its run R of 8 values belongs to chunk R mod g (as its
//   run R div g), so the threads of a group read and write neighbouring runs
//   the exponent stream chunk by chunk with the start bit of each chunk; 32-bit words filled
//   from bit 31 down, then two zero words
//   bytes: [0,256) lengths | [256,264) n | [264,272) stream bits | [272,...) 4096-entry table
//   (symbol | length << 8, uint16, indexed by the next 12 stream bits) | chunk start bits, uint32
//   [chunks + 1] | sign|mantissa bytes [n] in value order | stream words; each section 16-byte
//   aligned.
#include <algorithm>
#include <cstring>
#include <queue>
#include <vector>

#include "pmoe_internal.cuh"

namespace pmoe {
namespace {

constexpr int kChunk = 256;
constexpr int kGroup = 65536;            // values per group of 256 chunks
constexpr int kRun = 8;                  // values per run
constexpr int kLmax = 12;
constexpr int kLutBits = 12;
constexpr int kThreads = 256;             // one chunk per thread
constexpr int kMaxPages = 128;            // pages per decode launch (kernel parameter space)

struct Layout {
    int64_t lut, offs, sm, bits, n_chunks;
};

__host__ __device__ inline int64_t align16(int64_t x) { return (x + 15) & ~(int64_t)15; }

__host__ __device__ inline Layout layout_of(int64_t n) {
    Layout L;
    L.n_chunks = (n + kChunk - 1) / kChunk;
    L.lut = 272;
    L.offs = align16(L.lut + 2 * (1 << kLutBits));
    L.sm = align16(L.offs + 4 * (L.n_chunks + 1));
    L.bits = align16(L.sm + n);
    return L;
}

// Chunk `chunk`'s place: its group's first value, the group's chunk count g and run count, and
// its index c inside the group (its runs are c, c + g, c + 2g, ...).
struct ChunkPlace {
    int64_t g0;
    int64_t g, runs, c;
};
__host__ __device__ inline ChunkPlace place_of(int64_t n, int64_t chunk) {
    ChunkPlace P;
    const int64_t grp = chunk / 256;
    P.g0 = grp * kGroup;
    const int64_t v = n - P.g0 < kGroup ? n - P.g0 : kGroup;
    P.g = (v + kChunk - 1) / kChunk;
    P.runs = (v + kRun - 1) / kRun;
    P.c = chunk % 256;
    return P;
}

// Huffman code lengths of the 256 symbols from their counts.
void huffman_lengths(std::vector<uint64_t> counts, uint8_t* lengths) {
    for (;;) {
        std::memset(lengths, 0, 256);
        std::vector<int> present;
        for (int s = 0; s < 256; ++s)
            if (counts[s]) present.push_back(s);
        if (present.empty()) return;
        if (present.size() == 1) {
            lengths[present[0]] = 1;
            return;
        }
        // nodes: leaves first (symbol order), then merged nodes in creation order
        std::vector<int> parent(2 * present.size(), -1);
        typedef std::pair<uint64_t, int> Item;   // (count, creation order = node id)
        std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
        for (size_t i = 0; i < present.size(); ++i) heap.push(Item(counts[present[i]], (int)i));
        int next = (int)present.size();
        while (heap.size() > 1) {
            const Item a = heap.top(); heap.pop();
            const Item b = heap.top(); heap.pop();
            parent[a.second] = next;
            parent[b.second] = next;
            heap.push(Item(a.first + b.first, next));
            ++next;
        }
        int longest = 0;
        for (size_t i = 0; i < present.size(); ++i) {
            int depth = 0;
            for (int v = (int)i; parent[v] >= 0; v = parent[v]) ++depth;
            lengths[present[i]] = (uint8_t)depth;
            longest = std::max(longest, depth);
        }
        if (longest <= kLmax) return;
        for (int s = 0; s < 256; ++s)
            if (counts[s]) counts[s] = (counts[s] + 1) / 2;
    }
}

void canonical_codes(const uint8_t* lengths, uint32_t* codes) {
    int bl_count[kLmax + 2] = {0};
    for (int s = 0; s < 256; ++s)
        if (lengths[s]) bl_count[lengths[s]] += 1;
    uint32_t next_code[kLmax + 2] = {0};
    uint32_t code = 0;
    for (int L = 1; L <= kLmax; ++L) {
        code = (code + (uint32_t)bl_count[L - 1]) << 1;
        next_code[L] = code;
    }
    for (int s = 0; s < 256; ++s) codes[s] = lengths[s] ? next_code[lengths[s]]++ : 0;
}

struct DecodeArgs {
    const uint8_t* src[kMaxPages];
    int64_t src_bytes[kMaxPages];
    uint16_t* dst[kMaxPages];
    int64_t n;
    int ctas_per_page;
    int32_t* err;
};

// One thread per chunk: lookups on the next 12 bits of a 64-bit window, eight values joined and
// stored (16 bytes) at a time.  Each CTA first turns the page's table into a table of code pairs:
// entry w holds the symbol and length of the code at the front of w and, when the next code also
// fits in the 12 bits, that second symbol and the pair's length, so one lookup usually yields two
// values (bits 0-7 first symbol, 8-15 second, 16-19 first length, 20-23 pair length, 28 pair).
__global__ void __launch_bounds__(kThreads) exp_decode_kernel(const __grid_constant__ DecodeArgs a) {
    __shared__ uint16_t lut[1 << kLutBits];
    __shared__ uint32_t lut2[1 << kLutBits];
    const int page = blockIdx.x / a.ctas_per_page;
    const int64_t chunk = (int64_t)(blockIdx.x % a.ctas_per_page) * kThreads + threadIdx.x;
    const uint8_t* src = a.src[page];
    const Layout L = layout_of(a.n);
    {
        const uint4* t4 = reinterpret_cast<const uint4*>(src + L.lut);
        uint4* s4 = reinterpret_cast<uint4*>(lut);
        for (int i = threadIdx.x; i < (2 << kLutBits) / 16; i += kThreads) s4[i] = t4[i];
    }
    __syncthreads();
    for (int w = threadIdx.x; w < (1 << kLutBits); w += kThreads) {
        const uint32_t e1 = lut[w];
        const uint32_t l1 = e1 >> 8;
        uint32_t v = (e1 & 0xFFu) | (l1 << 16) | (l1 << 20);
        if (l1 >= 1 && l1 < (uint32_t)kLutBits) {
            const uint32_t e2 = lut[(w << l1) & ((1 << kLutBits) - 1)];
            const uint32_t l2 = e2 >> 8;
            if (l2 >= 1 && l1 + l2 <= (uint32_t)kLutBits)
                v = (e1 & 0xFFu) | ((e2 & 0xFFu) << 8) | (l1 << 16) | ((l1 + l2) << 20) | (1u << 28);
        }
        lut2[w] = v;
    }
    __syncthreads();
    if (chunk >= L.n_chunks) return;
    // (the host checked that the header sections for n lie inside the blob)
    const int64_t n_hdr = *reinterpret_cast<const int64_t*>(src + 256);
    const int64_t total = *reinterpret_cast<const int64_t*>(src + 264);
    const int64_t words_avail = (a.src_bytes[page] - L.bits) / 4;
    // a header that does not match the blob is reported, not read; inside the stream every
    // word read is checked against the blob's end (a corrupt table cannot walk past it)
    if (n_hdr != a.n || total > 32 * (words_avail - 2)) {
        if (a.err) atomicCAS(a.err, 0, (int)PMOE_ERR_INVALID_ARG);
        return;
    }
    const uint32_t* starts = reinterpret_cast<const uint32_t*>(src + L.offs);
    const int64_t start = starts[chunk];
    if (start > total) {
        if (a.err) atomicCAS(a.err, 0, (int)PMOE_ERR_INVALID_ARG);
        return;
    }
    const uint32_t* words = reinterpret_cast<const uint32_t*>(src + L.bits);
    const ChunkPlace P = place_of(a.n, chunk);
    const uint8_t* sm = src + L.sm;
    uint16_t* dst = a.dst[page];
    int64_t wi = start >> 5;
    int pos = (int)(start & 31);
    // the 64-bit window holds words wi and wi+1; word wi+2 is loaded one refill ahead, so the
    // load's latency hides behind the ~12 values decoded before it is needed
    uint64_t cur = ((uint64_t)__ldg(words + wi) << 32) | __ldg(words + wi + 1);
    uint32_t nxt = wi + 2 < words_avail ? __ldg(words + wi + 2) : 0u;
    auto advance = [&](int len) {
        pos += len;
        if (pos >= 32) {
            pos -= 32;
            ++wi;
            cur = (cur << 32) | nxt;
            nxt = wi + 2 < words_avail ? __ldg(words + wi + 2) : 0u;
        }
    };
    auto next_exp = [&]() -> uint32_t {
        const uint32_t e = lut2[(uint32_t)((cur << pos) >> (64 - kLutBits))];
        advance((int)((e >> 16) & 0xFu));
        return e & 0xFFu;
    };
    auto join = [](uint32_t ex, uint32_t s) -> uint32_t {
        return ((s & 0x80u) << 8) | (ex << 7) | (s & 0x7Fu);
    };
    // the chunk's runs; neighbouring threads hold neighbouring runs, so each warp's 8-byte loads
    // and 16-byte stores cover one contiguous range
    for (int64_t R = P.c; R < P.runs; R += P.g) {
        const int64_t v0 = P.g0 + kRun * R;
        if (v0 + kRun <= a.n) {
            const uint2 s8 = __ldg(reinterpret_cast<const uint2*>(sm + v0));
            // the run's 8 exponents, one or two per lookup
            uint64_t ex = 0;
            for (int got = 0; got < kRun;) {
                const uint32_t e = lut2[(uint32_t)((cur << pos) >> (64 - kLutBits))];
                const bool two = ((e >> 28) & 1u) && got < kRun - 1;
                ex |= (uint64_t)(two ? (e & 0xFFFFu) : (e & 0xFFu)) << (8 * got);
                advance((int)(two ? (e >> 20) & 0xFu : (e >> 16) & 0xFu));
                got += two ? 2 : 1;
            }
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t sw = q < 2 ? s8.x : s8.y;
                const int sh = (q & 1) * 16;
                const uint32_t e0 = (uint32_t)(ex >> (16 * q)) & 0xFFu;
                const uint32_t e1 = (uint32_t)(ex >> (16 * q + 8)) & 0xFFu;
                o[q] = join(e0, (sw >> sh) & 0xFFu) | (join(e1, (sw >> (sh + 8)) & 0xFFu) << 16);
            }
            *reinterpret_cast<uint4*>(dst + v0) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            for (int64_t v = v0; v < a.n; ++v) dst[v] = (uint16_t)join(next_exp(), sm[v]);
        }
    }
}

}  // namespace
}  // namespace pmoe

using namespace pmoe;

extern "C" size_t pmoe_exp_encode_bound(int64_t n) {
    if (n < 0) return 0;
    const Layout L = layout_of(n);
    return (size_t)(L.bits + 4 * (((n * kLmax + 31) >> 5) + 2));
}

extern "C" pmoe_status pmoe_exp_encode(const uint16_t* values, int64_t n, void* out, size_t cap,
                                       size_t* bytes) {
    if (n < 0 || (n > 0 && !values) || !out || !bytes)
        return record_failure(PMOE_ERR_INVALID_ARG, "pmoe_exp_encode: NULL argument or n < 0");
    if (cap < pmoe_exp_encode_bound(n))
        return record_failure(PMOE_ERR_INVALID_ARG, "pmoe_exp_encode: cap < pmoe_exp_encode_bound(n)");
    if ((uint64_t)n * kLmax >= (1ull << 32))
        return record_failure(PMOE_ERR_INVALID_ARG, "pmoe_exp_encode: page too large for 32-bit offsets");
    std::vector<uint64_t> counts(256, 0);
    for (int64_t i = 0; i < n; ++i) counts[(values[i] >> 7) & 0xFF] += 1;
    uint8_t lengths[256];
    huffman_lengths(counts, lengths);
    uint32_t codes[256];
    canonical_codes(lengths, codes);
    const Layout L = layout_of(n);
    uint8_t* o = static_cast<uint8_t*>(out);
    std::memset(o, 0, (size_t)L.bits);
    std::memcpy(o, lengths, 256);
    std::memcpy(o + 256, &n, 8);
    uint16_t* lut = reinterpret_cast<uint16_t*>(o + L.lut);
    for (int s = 0; s < 256; ++s) {
        if (!lengths[s]) continue;
        const uint32_t lo = codes[s] << (kLutBits - lengths[s]);
        for (uint32_t j = 0; j < (1u << (kLutBits - lengths[s])); ++j)
            lut[lo + j] = (uint16_t)(s | (lengths[s] << 8));
    }
    uint32_t* starts = reinterpret_cast<uint32_t*>(o + L.offs);
    uint8_t* sm = o + L.sm;
    for (int64_t i = 0; i < n; ++i) sm[i] = (uint8_t)(((values[i] >> 8) & 0x80) | (values[i] & 0x7F));
    uint32_t* words = reinterpret_cast<uint32_t*>(o + L.bits);
    uint64_t acc = 0;
    int acc_bits = 0;
    int64_t bitpos = 0, nw = 0;
    for (int64_t chunk = 0; chunk < L.n_chunks; ++chunk) {
        starts[chunk] = (uint32_t)bitpos;
        const ChunkPlace P = place_of(n, chunk);
        for (int64_t R = P.c; R < P.runs; R += P.g) {
            const int64_t v0 = P.g0 + kRun * R;
            for (int64_t i = v0; i < v0 + kRun && i < n; ++i) {
                const int s = (values[i] >> 7) & 0xFF;
                acc = (acc << lengths[s]) | codes[s];
                acc_bits += lengths[s];
                bitpos += lengths[s];
                if (acc_bits >= 32) {
                    words[nw++] = (uint32_t)(acc >> (acc_bits - 32));
                    acc_bits -= 32;
                    acc &= (acc_bits ? ((1ull << acc_bits) - 1) : 0);
                }
            }
        }
    }
    if (acc_bits) words[nw++] = (uint32_t)(acc << (32 - acc_bits));
    words[nw++] = 0;
    words[nw++] = 0;
    starts[L.n_chunks] = (uint32_t)bitpos;
    std::memcpy(o + 264, &bitpos, 8);
    *bytes = (size_t)(L.bits + 4 * nw);
    return PMOE_OK;
}

extern "C" pmoe_status pmoe_exp_decode_async(int32_t n_pages, int64_t n, const void* const* src,
                                             const int64_t* src_bytes, void* const* dst,
                                             int32_t* device_error, pmoe_stream_t stream) {
    if (n_pages < 0 || n_pages > kMaxPages || n < 1 || (n_pages > 0 && (!src || !src_bytes || !dst)))
        return record_failure(PMOE_ERR_INVALID_ARG,
                              "pmoe_exp_decode_async: 0 <= n_pages <= 128, n >= 1, arrays non-NULL");
    if (n_pages == 0) return PMOE_OK;
    DecodeArgs a{};
    const Layout L = layout_of(n);
    for (int p = 0; p < n_pages; ++p) {
        if (!src[p] || !dst[p] || (reinterpret_cast<uintptr_t>(src[p]) & 15) ||
            (reinterpret_cast<uintptr_t>(dst[p]) & 15))
            return record_failure(PMOE_ERR_INVALID_ARG,
                                  "pmoe_exp_decode_async: pointers must be non-NULL and 16-byte aligned");
        if (src_bytes[p] < L.bits + 8)
            return record_failure(PMOE_ERR_INVALID_ARG, "pmoe_exp_decode_async: blob smaller than its header");
        a.src[p] = static_cast<const uint8_t*>(src[p]);
        a.src_bytes[p] = src_bytes[p];
        a.dst[p] = static_cast<uint16_t*>(dst[p]);
    }
    a.n = n;
    a.ctas_per_page = (int)((L.n_chunks + kThreads - 1) / kThreads);
    a.err = device_error;
    const int64_t grid = (int64_t)n_pages * a.ctas_per_page;
    if (grid > INT32_MAX) return record_failure(PMOE_ERR_INVALID_ARG, "pmoe_exp_decode_async: too large");
    exp_decode_kernel<<<(unsigned)grid, kThreads, 0, (cudaStream_t)stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return record_failure(PMOE_ERR_CUDA, cudaGetErrorString(e));
    return PMOE_OK;
}

// Top-k softmax routing and the stable sort-and-pad of (token, slot) pairs by expert.
//
// Both steps sit ahead of the paged GEMMs of Rimuru's fused MoE kernel (paper-daily.com/en,
// "Expert weights are scattered across pages. How does the kernel read them?": the paged kernel
// runs on identical inputs and routing to the contiguous one).  Integer outputs are bit-exact
// and independent of thread scheduling: routing compares fp32 values exactly, and the sort
// ranks every pair by (expert, pair index) with warp ballots, not by atomic arrival order.
#include <math.h>

#include "pmoe_internal.cuh"
#include "route_common.cuh"

namespace pmoe {

template <int EPL>
__global__ void __launch_bounds__(128) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int renorm, int32_t* __restrict__ ids,
                                                    float* __restrict__ wout) {
    pdl_wait_prev();
    pdl_allow_next();
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    route_token<EPL>(logits + (int64_t)t * E, E, k, renorm, lane, ids + (int64_t)t * k,
                     wout + (int64_t)t * k);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                         float* w, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)((T + 3) / 4)), block(128);
    if (E <= 32) return launch_pdl(route_kernel<1>, grid, block, 0, s, logits, T, E, k, renorm, ids, w);
    else if (E <= 64) return launch_pdl(route_kernel<2>, grid, block, 0, s, logits, T, E, k, renorm, ids, w);
    else if (E <= 128) return launch_pdl(route_kernel<4>, grid, block, 0, s, logits, T, E, k, renorm, ids, w);
    else if (E <= 256) return launch_pdl(route_kernel<8>, grid, block, 0, s, logits, T, E, k, renorm, ids, w);
    else if (E <= 512) return launch_pdl(route_kernel<16>, grid, block, 0, s, logits, T, E, k, renorm, ids, w);
    else return launch_pdl(route_kernel<32>, grid, block, 0, s, logits, T, E, k, renorm, ids, w);
}

// ---------------------------------------------------------------------------------------------
// Sort + pad, one CTA of kAlignWarps warps.
//   pass A  warp w counts the routed pairs of its contiguous segment per expert (cw[w][e]);
//   scan    per expert: exclusive prefix of cw over warps; padded offsets off[e] over experts;
//   pass B  warp w walks its segment 32 pairs at a time; lanes with the same expert get their
//           rank from a match mask, so every pair lands at off[e] + (pairs of e before it).
// Shared-chunk pairs are already in order (token t of chunk s is its t-th pair) and pads fill
// the tail of each expert's last block.  The page resolution for the forward call (which map
// and page each active expert's three matrices come from, with range checks) runs here too,
// because it needs the per-expert counts.
// ---------------------------------------------------------------------------------------------
constexpr int kAlignWarps = 16;

// Where matrix j of active expert e lives for this call: (map, page) from the buffer slot or the
// page table, with range checks (a bad entry raises the error word and yields {-1, -1}).
__device__ __forceinline__ ExpertLoc resolve_loc(const ResolveArgs& rs, int E, int e, int j) {
    if (rs.contiguous) return ExpertLoc{0, 3 * e + j};
    const int bs = e < E ? rs.buf_slot[e] : -1;
    if (bs >= 0) {
        const int b = rs.slots_per_buffer > 0 ? bs / rs.slots_per_buffer : 2;
        const bool have = (b == 0 && rs.have_buf0) || (b == 1 && rs.have_buf1);
        if (b < 2 && have) return ExpertLoc{1 + b, 3 * (bs % rs.slots_per_buffer) + j};
        raise_error(rs.err, PMOE_ERR_SLOT_OOB);
    } else if (bs == -1) {
        const int p = rs.page_table[e * 3 + j];
        if (p >= 0 && p < rs.num_pages) return ExpertLoc{0, p};
        raise_error(rs.err, PMOE_ERR_PAGE_OOB);
    } else {
        raise_error(rs.err, PMOE_ERR_SLOT_OOB);
    }
    return ExpertLoc{-1, -1};
}

// The whole CTA: packed locations of every active expert's three matrices into sloc [ES][3].
__device__ __forceinline__ void resolve_all(const ResolveArgs& rs, int E, int ES, const int32_t* cnt,
                                            int32_t* sloc, int tid, int nt) {
    for (int idx = tid; idx < ES * 3; idx += nt)
        sloc[idx] = cnt[idx / 3] > 0 ? pack_loc(resolve_loc(rs, E, idx / 3, idx % 3)) : -1;
}

// One warp: the work units of the CTA-pair path from the padded offsets.  Per expert, in order,
// its pairs of consecutive 128-row blocks, then its odd last block, each with the expert and its
// three weight locations (sloc: packed, [ES][3], resolved by the whole CTA beforehand), so a GEMM
// finds everything about a tile in one load.  meta[kMetaPairs] = units, meta[kMetaSingles] =
// single-block units.
__device__ __forceinline__ void write_unit_list(const int32_t* off, int ES, int block_m,
                                                const ResolveArgs& rs, const int32_t* sloc,
                                                int32_t* meta, int lane) {
    const int per = (ES + 31) / 32;
    const int e0 = lane * per, e1 = min(ES, e0 + per);
    int nu = 0, ns = 0;
    for (int e = e0; e < e1; ++e) {
        const int nb = (off[e + 1] - off[e]) / block_m;
        nu += (nb + 1) >> 1;
        ns += nb & 1;
    }
    int iu = nu, is = ns;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, iu, o);
        const int b = __shfl_up_sync(0xffffffffu, is, o);
        if (lane >= o) { iu += a; is += b; }
    }
    int uu = iu - nu;
    for (int e = e0; e < e1; ++e) {
        const int b0 = off[e] / block_m, nb = (off[e + 1] - off[e]) / block_m;
        if (nb == 0) continue;
        const int p0 = sloc[3 * e], p1 = sloc[3 * e + 1], p2 = sloc[3 * e + 2];
        const int2 grp = make_int2(uu, (nb + 1) >> 1);
        for (int j = 0; j < (nb >> 1); ++j) {
            if (rs.unit_group) rs.unit_group[uu] = grp;
            rs.units[uu] = make_int4((b0 + 2 * j) << 1, e, p0, p1);
            rs.unit_w2[uu++] = p2;
        }
        if (nb & 1) {
            if (rs.unit_group) rs.unit_group[uu] = grp;
            rs.units[uu] = make_int4(((b0 + nb - 1) << 1) | 1, e, p0, p1);
            rs.unit_w2[uu++] = p2;
        }
    }
    if (lane == 31) {
        meta[kMetaPairs] = iu;
        meta[kMetaSingles] = is;
    }
}

// Phase time stamps of the one-CTA sort for performance work (compiled in only with
// -DPMOE_ALIGN_TRACE): globaltimer readings by thread 0 at the milestones named where ATRACE is used.
#ifdef PMOE_ALIGN_TRACE
__device__ unsigned long long g_align_trace[16];
__device__ __forceinline__ unsigned long long atrace_time() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    return t;
}
#define ATRACE(i) do { if (threadIdx.x == 0) g_align_trace[(i)] = atrace_time(); } while (0)
#else
#define ATRACE(i) ((void)0)
#endif

// Exclusive scan over experts of their padded row counts (cnt[e] rounded up to block_m) into
// off[0..ES], by the whole CTA: each thread sums a contiguous run of experts, warps scan their
// threads' sums with shuffles and warp 0 scans the warps' totals (wsum: kAlignWarps words).
// Every thread must call it; off is complete after the caller's next __syncthreads.
__device__ __forceinline__ void padded_offsets(const int32_t* cnt, int32_t* off, int ES, int block_m,
                                               int32_t* wsum) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, NT = kAlignWarps * 32;
    const int per = (ES + NT - 1) / NT;
    const int e0 = tid * per, e1 = min(ES, e0 + per);
    int local = 0;
    for (int e = e0; e < e1; ++e) local += (cnt[e] + block_m - 1) / block_m * block_m;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    if (w == 0) {
        int v = lane < kAlignWarps ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (lane < kAlignWarps) wsum[lane] = v;
    }
    __syncthreads();
    int run = incl - local + (w > 0 ? wsum[w - 1] : 0);
    for (int e = e0; e < e1; ++e) {
        off[e] = run;
        run += (cnt[e] + block_m - 1) / block_m * block_m;
    }
    if (tid == 0) off[ES] = wsum[kAlignWarps - 1];
}

// Pad rows, block map and valid rows per block of experts e = first, first + step, ... (one
// calling warp): lane i reads the offsets of the i-th expert of each group of 32, then the warp
// takes the group's experts that have rows one at a time, its lanes over the expert's pad rows
// and blocks (coalesced stores).
__device__ __forceinline__ void fill_blocks(const int32_t* off, const int32_t* cnt, int first, int step,
                                            int ES, int block_m, int32_t pad, int32_t* sorted_ids,
                                            int32_t* block_expert, int32_t* block_rows, int lane) {
    for (int g = first; g < ES; g += 32 * step) {
        const int e = g + lane * step;
        int o = 0, n = 0, end = 0;
        if (e < ES) {
            o = off[e];
            n = cnt[e];
            end = off[e + 1];
        }
        const int b0 = o / block_m, b1 = end / block_m;
        for (unsigned act = __ballot_sync(0xffffffffu, end > o); act; act &= act - 1) {
            const int src = __ffs(act) - 1;
            const int ee = g + src * step;
            const int oo = __shfl_sync(0xffffffffu, o, src), nn = __shfl_sync(0xffffffffu, n, src);
            const int en = __shfl_sync(0xffffffffu, end, src);
            const int bb0 = __shfl_sync(0xffffffffu, b0, src), bb1 = __shfl_sync(0xffffffffu, b1, src);
            for (int r = oo + nn + lane; r < en; r += 32) sorted_ids[r] = pad;
            for (int b = bb0 + lane; b < bb1; b += 32) {
                block_expert[b] = ee;
                if (block_rows) block_rows[b] = min(block_m, oo + nn - b * block_m);
            }
        }
    }
}

// `after_count` runs in every thread once the pairs are counted, before the CTA synchronises
// (the one-CTA sort stores its page tables to shared memory there, so their loads overlap the
// count).
template <typename AfterCount>
__device__ __forceinline__ void align_block(
    const int32_t* __restrict__ ids, int T, int k, int E, int S, int block_m,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ block_expert,
    int32_t* __restrict__ inv, int32_t* __restrict__ meta, const ResolveArgs& rs, int do_resolve,
    int32_t* smem, AfterCount&& after_count) {
    const int ES = E + S;
    int32_t* cw = smem;                         // [kAlignWarps][ES]
    int32_t* cnt = cw + kAlignWarps * ES;       // [ES]
    int32_t* off = cnt + ES;                    // [ES + 1]
    int32_t* wsum = off + ES + 1;               // [kAlignWarps]
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int NT = kAlignWarps * 32;
    const int64_t NR = (int64_t)T * k;
    const int64_t NP = (int64_t)T * (k + S);

    ATRACE(0);   // start
    {
        // shared memory is 16-byte aligned and kAlignWarps * ES is a multiple of 4
        int4* cw4 = reinterpret_cast<int4*>(cw);
        for (int i = tid; i < kAlignWarps * ES / 4; i += NT) cw4[i] = make_int4(0, 0, 0, 0);
    }
    __syncthreads();
    ATRACE(1);   // counters zeroed

    const int64_t seg = (NR + kAlignWarps - 1) / kAlignWarps;
    const int64_t s0 = (int64_t)w * seg;
    const int64_t s1 = s0 + seg < NR ? s0 + seg : NR;
    for (int64_t i = s0 + lane; i < s1; i += 32) {
        int e = ids[i];
        if (e < 0 || e >= E) e = 0;  // routing output is in range; guard the test entry point
        atomicAdd(&cw[w * ES + e], 1);
    }
    after_count();
    __syncthreads();
    ATRACE(2);   // counted

    for (int e = tid; e < ES; e += NT) {
        int c = 0;
        for (int ww = 0; ww < kAlignWarps; ++ww) {
            const int x = cw[ww * ES + e];
            cw[ww * ES + e] = c;
            c += x;
        }
        cnt[e] = e < E ? c : T;
    }
    __syncthreads();
    ATRACE(3);   // per-warp prefix

    padded_offsets(cnt, off, ES, block_m, wsum);
    __syncthreads();
    ATRACE(4);   // offsets

    const unsigned lt_mask = (1u << lane) - 1u;
    for (int64_t base = s0; base < s1; base += 32) {
        const int64_t i = base + lane;
        const bool valid = i < s1;
        int e = valid ? ids[i] : -1 - lane;
        if (valid && (e < 0 || e >= E)) e = 0;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (valid) {
            const int pos = off[e] + cw[w * ES + e] + __popc(peers & lt_mask);
            sorted_ids[pos] = (int32_t)i;
            inv[i] = pos;
        }
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) cw[w * ES + e] += __popc(peers);
        __syncwarp();
    }
    ATRACE(5);   // routed pairs placed
    for (int64_t idx = tid; idx < (int64_t)S * T; idx += NT) {
        const int s = (int)(idx / T), t = (int)(idx % T);
        const int pos = off[E + s] + t;
        sorted_ids[pos] = (int32_t)(NR + idx);
        inv[NR + idx] = pos;
    }
    ATRACE(6);   // shared pairs placed
    fill_blocks(off, cnt, w, kAlignWarps, ES, block_m, (int32_t)NP, sorted_ids, block_expert,
                rs.block_rows, lane);
    if (tid == 0) meta[kMetaNPadded] = off[ES];
    ATRACE(7);   // pads and block map
    if (rs.units) {
        __syncthreads();   // the per-warp counters are free: they hold the locations now
        resolve_all(rs, E, ES, cnt, cw, tid, NT);
        __syncthreads();
        if (w == 0) write_unit_list(off, ES, block_m, rs, cw, meta, lane);
    }

    if (do_resolve) {
        for (int idx = tid; idx < ES * 3; idx += NT) {
            const int e = idx / 3, j = idx % 3;
            rs.loc[idx] = cnt[e] > 0 ? resolve_loc(rs, E, e, j) : ExpertLoc{-1, -1};
        }
    }
    ATRACE(8);   // resolved
}

constexpr int kPrepTabPerThread = 8;   // (E + 3*(E+S)) / threads for E + S <= 1024
static_assert(kPrepTabPerThread * kAlignWarps * 32 >= 4 * kMaxExpertsTotal,
              "every buffer-slot and page-table entry needs a thread's table register");

__host__ __device__ constexpr int align_words(int ES) { return kAlignWarps * ES + 2 * ES + 1 + kAlignWarps; }

// The one-CTA sort.  With page resolution, the buffer-slot and page tables are loaded at the
// start (a few loads per thread, in flight while the pairs are counted) and kept in shared
// memory after the sort's own words, so the resolution at the end reads shared memory only.
__global__ void __launch_bounds__(kAlignWarps * 32) align_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int S, int block_m,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ block_expert,
    int32_t* __restrict__ inv, int32_t* __restrict__ meta, ResolveArgs rs, int do_resolve) {
    extern __shared__ int32_t smem[];
    const int ES = E + S;
    int32_t* s_bs = smem + align_words(ES);   // [E]
    int32_t* s_pt = s_bs + E;                 // [ES*3]
    pdl_wait_prev();
    pdl_allow_next();
    const int tid = threadIdx.x;
    constexpr int NT = kAlignWarps * 32;
    const int ntab = do_resolve && !rs.contiguous ? E + 3 * ES : 0;
    int32_t tv[kPrepTabPerThread];
#pragma unroll
    for (int i = 0; i < kPrepTabPerThread; ++i) {
        const int idx = tid + i * NT;
        tv[i] = idx < ntab ? (idx < E ? rs.buf_slot[idx] : rs.page_table[idx - E]) : 0;
    }
    auto stash = [&]() {
#pragma unroll
        for (int i = 0; i < kPrepTabPerThread; ++i) {
            const int idx = tid + i * NT;
            if (idx < ntab) {
                if (idx < E) s_bs[idx] = tv[i];
                else s_pt[idx - E] = tv[i];
            }
        }
    };
    ResolveArgs local = rs;
    if (ntab > 0) {
        local.buf_slot = s_bs;
        local.page_table = s_pt;
    }
    align_block(ids, T, k, E, S, block_m, sorted_ids, block_expert, inv, meta, local, do_resolve, smem,
                stash);
}

// ---------------------------------------------------------------------------------------------
// Sort + pad over many CTAs (large T).  The routed pairs are cut into C contiguous segments.
//   count    CTA c histograms its segment by expert (shared-memory atomics) -> part[c][e];
//   scatter  CTA c sums part over all CTAs (expert totals, padded exclusive offsets off[e]) and
//            over CTAs before it (its base inside each expert), then places its segment exactly
//            like the single-CTA pass B: per-warp counts, prefix over warps, match-mask ranks.
//            The result is the same stable order as the single-CTA kernel.  Shared-chunk pairs,
//            pads, the block map and the page resolution are split across the C CTAs.
// ---------------------------------------------------------------------------------------------
constexpr int kAlignMaxCtas = 64;
constexpr int kAlignOneCtaPairs = 2048;   // up to this many routed pairs: the one-CTA kernel
// above: one CTA per max(512, 2 * (E + S)) pairs, at most 64 -- every scatter CTA also sums the
// histograms of the CTAs before it over all experts, so CTAs get dearer with more experts
// (measured at 4096 tokens: 60 experts 20 -> 16 us going from 8 to 32 CTAs; 513 experts 16 -> 18
// us going from 20 to 64)
constexpr int kAlignPairsPerCta = 512;

__global__ void __launch_bounds__(kAlignWarps * 32) align_count_kernel(
    const int32_t* __restrict__ ids, int NR, int E, int ES, int seg, int32_t* __restrict__ part) {
    extern __shared__ int32_t h[];
    pdl_wait_prev();
    pdl_allow_next();
    const int tid = threadIdx.x, NT = kAlignWarps * 32, c = blockIdx.x;
    for (int e = tid; e < ES; e += NT) h[e] = 0;
    __syncthreads();
    const int64_t s0 = (int64_t)c * seg, s1 = s0 + seg < NR ? s0 + seg : NR;
    for (int64_t i = s0 + tid; i < s1; i += NT) {
        int e = ids[i];
        if (e < 0 || e >= E) e = 0;
        atomicAdd(&h[e], 1);
    }
    __syncthreads();
    for (int e = tid; e < ES; e += NT) part[(int64_t)c * ES + e] = h[e];
}

__global__ void __launch_bounds__(kAlignWarps * 32) align_scatter_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int S, int block_m, int seg, int C,
    const int32_t* __restrict__ part, int32_t* __restrict__ sorted_ids,
    int32_t* __restrict__ block_expert, int32_t* __restrict__ inv, int32_t* __restrict__ meta,
    ResolveArgs rs, int do_resolve) {
    extern __shared__ int32_t sm[];
    const int ES = E + S;
    int32_t* off = sm;                 // [ES + 1]
    int32_t* cnt = off + ES + 1;       // [ES]
    int32_t* base = cnt + ES;          // [ES]
    int32_t* cw = base + ES;           // [kAlignWarps][ES]
    int32_t* wsum = cw + kAlignWarps * ES;   // [kAlignWarps]
    pdl_wait_prev();
    pdl_allow_next();
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, NT = kAlignWarps * 32;
    const int c = blockIdx.x;
    const int64_t NR = (int64_t)T * k, NP = (int64_t)T * (k + S);
    for (int e = tid; e < ES; e += NT) {
        int tot = 0, mine = 0;
        if (e < E) {
            // the C histograms' entries of expert e, eight loads in flight (each an L2 round trip)
            for (int c0 = 0; c0 < C; c0 += 8) {
                int v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = c0 + q < C ? part[(int64_t)(c0 + q) * ES + e] : 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (c0 + q < c) mine += v[q];
                    tot += v[q];
                }
            }
        } else {
            tot = T;
        }
        cnt[e] = tot;
        base[e] = mine;
    }
    for (int i = tid; i < kAlignWarps * ES; i += NT) cw[i] = 0;
    __syncthreads();
    padded_offsets(cnt, off, ES, block_m, wsum);
    // this CTA's segment, split into per-warp sub-segments
    const int64_t c0 = (int64_t)c * seg, c1 = c0 + seg < NR ? c0 + seg : NR;
    const int64_t sub = (c1 - c0 + kAlignWarps - 1) / kAlignWarps;
    const int64_t s0 = c0 + (int64_t)w * sub < c1 ? c0 + (int64_t)w * sub : c1;
    const int64_t s1 = s0 + sub < c1 ? s0 + sub : c1;
    for (int64_t i = s0 + lane; i < s1; i += 32) {
        int e = ids[i];
        if (e < 0 || e >= E) e = 0;
        atomicAdd(&cw[w * ES + e], 1);
    }
    __syncthreads();
    for (int e = tid; e < ES; e += NT) {
        int run = off[e] + base[e];
        for (int ww = 0; ww < kAlignWarps; ++ww) {
            const int x = cw[ww * ES + e];
            cw[ww * ES + e] = run;
            run += x;
        }
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int64_t b = s0; b < s1; b += 32) {
        const int64_t i = b + lane;
        const bool valid = i < s1;
        int e = valid ? ids[i] : -1 - lane;
        if (valid && (e < 0 || e >= E)) e = 0;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (valid) {
            const int pos = cw[w * ES + e] + __popc(peers & lt_mask);
            sorted_ids[pos] = (int32_t)i;
            inv[i] = pos;
        }
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) cw[w * ES + e] += __popc(peers);
        __syncwarp();
    }
    // shared-chunk pairs, pads, block map, resolution: split across the CTAs
    for (int64_t idx = (int64_t)c * NT + tid; idx < (int64_t)S * T; idx += (int64_t)C * NT) {
        const int s = (int)(idx / T), t = (int)(idx % T);
        const int pos = off[E + s] + t;
        sorted_ids[pos] = (int32_t)(NR + idx);
        inv[NR + idx] = pos;
    }
    fill_blocks(off, cnt, c * kAlignWarps + w, C * kAlignWarps, ES, block_m, (int32_t)NP, sorted_ids,
                block_expert, rs.block_rows, lane);
    if (c == 0 && tid == 0) meta[kMetaNPadded] = off[ES];
    if (c == 0 && rs.units) {
        __syncthreads();   // the per-warp counters are free: they hold the locations now
        resolve_all(rs, E, ES, cnt, cw, tid, NT);
        __syncthreads();
        if (w == 0) write_unit_list(off, ES, block_m, rs, cw, meta, lane);
    }
    if (do_resolve) {
        for (int idx = c * NT + tid; idx < ES * 3; idx += C * NT) {
            const int e = idx / 3, j = idx % 3;
            rs.loc[idx] = cnt[e] > 0 ? resolve_loc(rs, E, e, j) : ExpertLoc{-1, -1};
        }
    }
}

// Copy the hidden row of every (token, expert) pair to its sorted row: X[inv[i]] = hidden[token
// of pair i].  Pad rows are left as they are: in both MMA orientations a pad row only feeds
// outputs of its own row, which nothing reads.
__device__ __forceinline__ void gather_pair(const uint16_t* __restrict__ hidden,
                                            const int32_t* __restrict__ inv, int i, int T, int k,
                                            int d, int lane, uint16_t* __restrict__ x) {
    const int NR = T * k;
    const int t = i < NR ? i / k : (i - NR) % T;
    const uint4* src = reinterpret_cast<const uint4*>(hidden + (int64_t)t * d);
    uint4* dst = reinterpret_cast<uint4*>(x + (int64_t)inv[i] * d);
    for (int c = lane; c < (d >> 3); c += 32) dst[c] = src[c];
}

__global__ void __launch_bounds__(256) gather_pairs_kernel(const uint16_t* __restrict__ hidden,
                                                           const int32_t* __restrict__ inv, int T,
                                                           int k, int S, int d,
                                                           uint16_t* __restrict__ x) {
    pdl_wait_prev();
    pdl_allow_next();
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (i >= T * (k + S)) return;
    gather_pair(hidden, inv, i, T, k, d, threadIdx.x & 31, x);
}

// Small batches: routing and sort + pad (with page resolution) in one CTA, so a decode step spends
// one launch on them instead of two.  The page-table loads are issued before the routing so the
// two latencies overlap; the routing ids and the tables then stay in shared memory for the sort.
// When the gathered rows are small, the row gather runs here too (x != NULL).

template <int EPL>
__global__ void __launch_bounds__(kAlignWarps * 32) prep_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renorm, int32_t* __restrict__ ids,
    float* __restrict__ wout, int S, int block_m, int32_t* __restrict__ sorted_ids,
    int32_t* __restrict__ block_expert, int32_t* __restrict__ inv, int32_t* __restrict__ meta,
    ResolveArgs rs, const uint16_t* __restrict__ hidden, int d, uint16_t* __restrict__ x) {
    extern __shared__ int32_t smem[];
    const int ES = E + S;
    int32_t* s_align = smem;
    int32_t* s_ids = s_align + align_words(ES);   // [T*k]
    int32_t* s_bs = s_ids + T * k;                // [E]
    int32_t* s_pt = s_bs + E;                     // [ES*3]
    pdl_wait_prev();
    pdl_allow_next();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int NT = kAlignWarps * 32;
    const int ntab = rs.contiguous ? 0 : E + 3 * ES;
    int32_t tv[kPrepTabPerThread];
#pragma unroll
    for (int i = 0; i < kPrepTabPerThread; ++i) {
        const int idx = tid + i * NT;
        tv[i] = idx < ntab ? (idx < E ? rs.buf_slot[idx] : rs.page_table[idx - E]) : 0;
    }
    ATRACE(9);   // prep: tables loading, routing starts
    for (int t = warp; t < T; t += kAlignWarps)
        route_token<EPL>(logits + (int64_t)t * E, E, k, renorm, lane, s_ids + t * k,
                         wout + (int64_t)t * k);
    ATRACE(10);   // prep: thread 0's warp routed
#pragma unroll
    for (int i = 0; i < kPrepTabPerThread; ++i) {
        const int idx = tid + i * NT;
        if (idx < ntab) {
            if (idx < E) s_bs[idx] = tv[i];
            else s_pt[idx - E] = tv[i];
        }
    }
    __syncthreads();
    for (int i = tid; i < T * k; i += NT) ids[i] = s_ids[i];
    ResolveArgs local = rs;
    if (!rs.contiguous) {
        local.buf_slot = s_bs;
        local.page_table = s_pt;
    }
    align_block(s_ids, T, k, E, S, block_m, sorted_ids, block_expert, inv, meta, local, 1, s_align,
                [] {});
    if (x) {
        __syncthreads();
        const int NP = T * (k + S);
        for (int i = warp; i < NP; i += kAlignWarps) gather_pair(hidden, inv, i, T, k, d, lane, x);
    }
    ATRACE(11);   // prep: rows gathered
}

#ifdef PMOE_ALIGN_TRACE
extern "C" int pmoe_align_trace_read(unsigned long long* host) {
    return (int)cudaMemcpyFromSymbol(host, g_align_trace, sizeof(unsigned long long) * 16);
}
#endif

// the one-CTA sort's words and its copy of the buffer-slot and page tables (E <= ES)
static size_t align_smem_bytes(int ES) { return sizeof(int32_t) * ((size_t)align_words(ES) + 4 * (size_t)ES); }

static size_t prep_smem_bytes(int T, int E, int k, int S) {
    return sizeof(int32_t) * ((size_t)align_words(E + S) + (size_t)T * k + E + 3 * (size_t)(E + S));
}

static cudaError_t allow_align_smem(const void* fn, std::atomic<unsigned long long>* done) {
    return raise_smem_limit(fn, (int)prep_smem_bytes(128, kMaxExpertsTotal, kMaxTopK, 0), done);
}

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int S, int block_m,
                         int32_t* sorted_ids, int32_t* block_expert, int32_t* inv,
                         int32_t* meta, const ResolveArgs* resolve, cudaStream_t s) {
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(align_kernel),
                                     (int)align_smem_bytes(kMaxExpertsTotal), &attr);
    if (e != cudaSuccess) return e;
    ResolveArgs rs{};
    if (resolve) rs = *resolve;
    return launch_pdl(align_kernel, dim3(1), dim3(kAlignWarps * 32), align_smem_bytes(E + S), s,
                      ids, T, k, E, S, block_m, sorted_ids, block_expert, inv, meta, rs,
                      resolve ? 1 : 0);
}

int align_ctas(int64_t NR, int ES) {
    if (NR <= kAlignOneCtaPairs) return 1;
    const int64_t per = 2 * (int64_t)ES > kAlignPairsPerCta ? 2 * (int64_t)ES : kAlignPairsPerCta;
    int64_t c = (NR + per - 1) / per;
    if (c < 1) c = 1;
    if (c > kAlignMaxCtas) c = kAlignMaxCtas;
    return (int)c;
}

size_t align_part_bytes() { return sizeof(int32_t) * (size_t)kAlignMaxCtas * kMaxExpertsTotal; }

cudaError_t launch_align_multi(const int32_t* ids, int T, int k, int E, int S, int block_m,
                               int32_t* part, int32_t* sorted_ids, int32_t* block_expert,
                               int32_t* inv, int32_t* meta, const ResolveArgs* resolve,
                               cudaStream_t s) {
    const int64_t NR = (int64_t)T * k;
    const int C = align_ctas(NR, E + S);
    if (C == 1)
        return launch_align(ids, T, k, E, S, block_m, sorted_ids, block_expert, inv, meta, resolve, s);
    const int ES = E + S;
    const int seg = (int)((NR + C - 1) / C);
    const size_t sm2 = sizeof(int32_t) * ((size_t)(kAlignWarps + 3) * ES + 1 + kAlignWarps);
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e0 = raise_smem_limit(reinterpret_cast<const void*>(align_scatter_kernel),
                                      (int)(sizeof(int32_t) * ((size_t)(kAlignWarps + 3) * kMaxExpertsTotal + 1 + kAlignWarps)),
                                      &attr);
    if (e0 != cudaSuccess) return e0;
    ResolveArgs rs{};
    if (resolve) rs = *resolve;
    cudaError_t e = launch_pdl(align_count_kernel, dim3(C), dim3(kAlignWarps * 32),
                               sizeof(int32_t) * ES, s, ids, (int)NR, E, ES, seg, part);
    if (e != cudaSuccess) return e;
    return launch_pdl(align_scatter_kernel, dim3(C), dim3(kAlignWarps * 32), sm2, s, ids, T, k, E, S,
                      block_m, seg, C, (const int32_t*)part, sorted_ids, block_expert, inv, meta, rs,
                      resolve ? 1 : 0);
}

cudaError_t launch_gather_pairs(const uint16_t* hidden, const int32_t* inv, int T, int k, int S,
                                int d, uint16_t* x, cudaStream_t s) {
    const int64_t np = (int64_t)T * (k + S);
    if (np == 0) return cudaSuccess;
    return launch_pdl(gather_pairs_kernel, dim3((unsigned)((np + 7) / 8)), dim3(256), 0, s, hidden,
                      inv, T, k, S, d, x);
}

template <int EPL>
static cudaError_t prep_small_epl(const float* logits, int T, int E, int k, int renorm,
                                  int32_t* ids, float* w, int S, int block_m, int32_t* sorted_ids,
                                  int32_t* block_expert, int32_t* inv, int32_t* meta,
                                  const ResolveArgs& rs, const uint16_t* hidden, int d,
                                  uint16_t* x, cudaStream_t s) {
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = allow_align_smem(reinterpret_cast<const void*>(prep_small_kernel<EPL>), &attr);
    if (e != cudaSuccess) return e;
    return launch_pdl(prep_small_kernel<EPL>, dim3(1), dim3(kAlignWarps * 32),
                      prep_smem_bytes(T, E, k, S), s, logits, T, E, k, renorm, ids, w, S, block_m,
                      sorted_ids, block_expert, inv, meta, rs, hidden, d, x);
}

cudaError_t launch_prep_small(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                              float* w, int S, int block_m, int32_t* sorted_ids,
                              int32_t* block_expert, int32_t* inv, int32_t* meta,
                              const ResolveArgs& rs, const uint16_t* hidden, int d, uint16_t* x,
                              cudaStream_t s) {
#define PREP(EPL) prep_small_epl<EPL>(logits, T, E, k, renorm, ids, w, S, block_m, sorted_ids, \
                                      block_expert, inv, meta, rs, hidden, d, x, s)
    if (E <= 32) return PREP(1);
    if (E <= 64) return PREP(2);
    if (E <= 128) return PREP(4);
    if (E <= 256) return PREP(8);
    if (E <= 512) return PREP(16);
    return PREP(32);
#undef PREP
}

}  // namespace pmoe

// Paged grouped expert GEMMs on CTA pairs (tcgen05.mma.cta_group::2, sm_103a).
//
// Same operation as the single-CTA kernel in tc_gemm.cu -- Rimuru's paged MoE GEMMs
// (paper-daily.com/en, "Expert weights are scattered across pages. How does the kernel read
// them?"; page rule addr_e(n,t) = B_P + p_e(n)*f*d + (n mod f)*d + t as one TMA row coordinate
// per tile) -- with each 256x256 output tile computed by a pair of CTAs on two SMs.  The pair
// shares one B operand: each CTA stages half of it, the tensor cores of both SMs read both
// halves, so every SM moves 32 KB per k-block instead of 48 KB and the shared-memory traffic per
// MMA drops by a third.  A tile's 256 rows are two consecutive 128-row blocks of one expert (one
// per CTA, M = 256).  An expert's odd last block is a unit of its own in the same launch, right
// after the expert's pairs so that it finds the expert's weights in L2, with the operands'
// roles swapped: 256 weight rows on the MMA's M side (128 per CTA) and the block's 128 tokens on
// N (64 staged by each CTA), so it fills the tensor cores as a pair does at half the work (an
// M = 128 MMA, 64 token rows per CTA, ran at half rate and cost as much as a pair).
//
//   pair, gate/up: B = [128 rows of the W1 page | 128 rows of the W3 page] for output columns
//            n0..n0+127: the leader CTA stages the W1 half, its peer the W3 half; every CTA's
//            accumulator holds gate (columns 0..127) and up (128..255) for its own 128 rows.
//   pair, down: B = 256 rows of the W2 page, 128 staged by each CTA.
//   single block, gate/up: A = [64 W1 rows | 64 W3 rows] of output columns n0 + 64*rank .. +63
//            on each CTA; TMEM lanes 0..63 hold gate, 64..127 up, columns the 128 tokens; the up
//            lanes hand their values to the gate lanes through shared memory.
//   single block, down: A = 128 W2 rows (output columns) on each CTA, as the pair's B halves.
//
// Protocol: both CTAs' TMA loads complete on the leader's full barrier; the leader issues the
// MMAs and commits them to the empty and accumulator-full barriers of both CTAs (multicast);
// each CTA's epilogue reads its own TMEM and releases the accumulator on the leader's barrier.
// Every mbarrier wait is bounded; on a time-out the pair unwinds through the same cluster
// barriers and TMEM release as a normal exit.
#include <math.h>

#include "tc_common.cuh"

namespace pmoe {

namespace {

using namespace tc;

constexpr int BK = 64;
constexpr int BN = 256;
constexpr int STAGES = 6;
constexpr int A_BYTES = 128 * BK * 2;  // 16 KB: this CTA's 128 rows
constexpr int B_BYTES = 128 * BK * 2;  // 16 KB: this CTA's half of B
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 192;
constexpr int kTileRing = 4;          // tiles handed from the producer to the MMA and epilogue
constexpr uint32_t kTmemCols = 512;
constexpr int kYBox = 32 * 64 * 2;   // down epilogue: one 32-row x 64-column bf16 store box
constexpr int kXchBytes = 16 * 64 * 4;                  // single gate/up: up values of 16 tokens
// ring, alignment slack, barriers (1 KB, keeping what follows 1024-byte aligned) and, for the down
// GEMM, two store boxes per epilogue warp (gate/up: the single blocks' exchange buffer)
template <int kMode>
constexpr int smem_bytes() { return STAGES * STAGE_BYTES + 1024 + 1024 + (kMode == 2 ? 4 * 2 * kYBox : kXchBytes); }
constexpr uint32_t kIdesc = idesc_bf16(256, BN);      // pair of blocks: 128 rows on each CTA
constexpr uint32_t kIdescSwap = idesc_bf16(256, 128);   // single block: weights on M, tokens on N
constexpr int A64_BYTES = 64 * BK * 2;                  // 8 KB: 64 rows of a 64-column k-block

enum { kGateUp = 1, kDown = 2 };
constexpr size_t kRasterBytes = (size_t)32 << 20;   // a quarter of the 129 MB L2, rounded down

// Per-tile time stamps for performance work (compiled in only with -DPMOE_GEMM_TRACE), as in the
// single-CTA kernel: [0] accumulator free, [1] first k-block landed, [2] last MMA issued (all
// globaltimer, the leader's MMA issuer), [3] SM cycles it waited for loads, [4] accumulator
// released and [6] accumulator seen full (the leader's first epilogue warp), [5] SM id, [7] wait
// for the accumulator begun.
#ifdef PMOE_GEMM_TRACE
constexpr int kTraceTiles = 8192;
constexpr int kTraceWords = 8;
__device__ unsigned long long g_gemm2_trace[2][kTraceTiles][kTraceWords];
#define GTRACE(t, i, v) \
    do { if ((t) < kTraceTiles) g_gemm2_trace[kMode - 1][(t)][(i)] = (unsigned long long)(v); } while (0)
#else
#define GTRACE(t, i, v) ((void)0)
#endif

struct Tc2Args {
    const int4* units;             // {(first block << 1) | single, expert, W1 loc, W3 loc}
    const int32_t* unit_w2;        // W2 loc of each unit (locations packed by pack_loc)
    const int2* unit_group;        // {first unit, units} of each unit's expert
    int raster;                    // 1: tiles ordered by expert, N tile, then unit (see below)
    int shared_units;              // the last units of the list belong to shared chunks
    const int32_t* meta;
    void* out;
    int f, d;
    int k_blocks;
    int n_tiles;
    int32_t* err;
    SharedRows sh;      // gate/up: shared-chunk blocks straight from hidden
};

struct Tc2Maps {
    CUtensorMap a;      // X_sorted [cap][d] or h [cap][f], 128-row boxes
    CUtensorMap w[3];   // pool / buffer 0 / buffer 1 weight views, 128-row boxes
    CUtensorMap hid;    // hidden [T][d], 128-row boxes, when args.sh.direct
    CUtensorMap y;      // down: y bf16 [cap][d], 32-row x 64-column boxes, 128-byte swizzle
    CUtensorMap a64;    // the same views with 64-row boxes (single blocks: 64 rows per CTA)
    CUtensorMap hid64;
    CUtensorMap w64[3]; // gate/up weight views with 64-row boxes
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// TMA load into this CTA's shared memory that completes on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive (once) on the barrier at this shared-memory offset in both CTAs when the MMAs issued so
// far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

template <int kMode, bool kContig>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_gemm2sm_kernel(const __grid_constant__ Tc2Maps maps, const Tc2Args args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + STAGES * STAGE_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sgen + STAGES * STAGE_BYTES + 8 * (2 * STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // tile ring: the producer hands each tile's unit and N tile to the MMA issuer and the epilogue
    // warps, which then need no global loads of their own between tiles
    auto mfull_bar = [&](int j) { return bar0 + 256u + 8u * j; };
    auto mempty_bar = [&](int j) { return bar0 + 256u + 8u * (kTileRing + j); };
    int4* tile_ring = reinterpret_cast<int4*>(sgen + STAGES * STAGE_BYTES + 256 + 16 * kTileRing);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);     // used on the leader: its producer's expect_tx
            mbar_init(empty_bar(s), 1);    // the leader's multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);    // the leader's multicast commit
            mbar_init(tempty_bar(a), 8);   // used on the leader: 4 epilogue warps x 2 CTAs
        }
        for (int j = 0; j < kTileRing; ++j) {
            mbar_init(mfull_bar(j), 1);                      // this CTA's producer
            mbar_init(mempty_bar(j), rank == 0 ? 5 : 4);     // epilogue warps (+ the MMA issuer)
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        // one warp of each CTA allocates the pair's tensor memory together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();            // the peer's barriers exist before anyone signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_wait_prev();
    pdl_allow_next();

    const int nunits = args.meta[kMetaPairs];
    const int64_t ntiles = (int64_t)nunits * args.n_tiles;
    const int64_t cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    // Work order.  Experts whose matrices fit in L2 (args.raster == 0): unit by unit, each unit's
    // N tiles in turn, with the shared chunks' units (weights resident in L2, tensor-bound) spread
    // evenly among the routed experts' units (weights streamed from HBM), so HBM streams over the
    // whole launch; an expert's pairs and its odd block stay together and share its weights in L2.
    // Experts larger than L2 (args.raster == 1): expert by expert, and within an expert N tile by
    // N tile with the expert's units innermost, so the pairs running at once share a few weight
    // tiles and the expert's token rows in L2 instead of each unit streaming all of the expert's
    // weights from HBM again.
    const int nrouted = nunits - args.shared_units;
    const bool mix = !args.raster && args.shared_units > 0 && nrouted > 0;
    auto pos_of = [&](int64_t t) -> int {
        int i = (int)(t / args.n_tiles);
        if (mix) {
            const int r = (int)(((int64_t)i * nrouted) / nunits);          // routed units before i
            const bool routed = (int)(((int64_t)(i + 1) * nrouted) / nunits) > r;
            i = routed ? r : nrouted + (i - r);
        }
        return i;
    };

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int pend_phase[STAGES];
            for (int s = 0; s < STAGES; ++s) pend_phase[s] = -1;
            int mslot = 0;
            uint32_t mphase = 0;
            bool ok = true;
            // hands one tile (or, with pb < 0, the end of the work) to this CTA's consumers
            auto publish = [&](int pb, bool single, int nt, int64_t t) -> bool {
                if (!mbar_wait(mempty_bar(mslot), mphase ^ 1u, abort_flag, args.err)) return false;
                tile_ring[mslot] = make_int4(pb < 0 ? -1 : (pb << 1) | (single ? 1 : 0), nt, (int)t, 0);
                mbar_arrive(mfull_bar(mslot));
                if (++mslot == kTileRing) { mslot = 0; mphase ^= 1u; }
                return true;
            };
            const int npad = args.meta[kMetaNPadded];
            // Everything about a tile is in its unit's record (one 16-byte load, plus the W2
            // location for down); the next tile's record is loaded at the start of this tile,
            // so its latency (a microsecond or two while the GEMM loads L2) hides behind this
            // tile's copies.  A chain of dependent loads here (unit, then expert, then page
            // location) drained the ring: the paged gate/up ran 5% behind fixed addressing.
            struct TileMeta {
                int pb, single, e, nt;
                ExpertLoc l0, l1;
            };
            auto meta_load = [&](TileMeta& m, int64_t tt) {
                int i;
                if (args.raster) {
                    const int2 g = args.unit_group[(int)(tt / args.n_tiles)];
                    const int64_t local = tt - (int64_t)g.x * args.n_tiles;
                    m.nt = (int)(local / g.y);
                    i = g.x + (int)(local - (int64_t)m.nt * g.y);
                } else {
                    i = pos_of(tt);
                    m.nt = (int)(tt % args.n_tiles);
                }
                const int4 r = args.units[i];
                const int32_t w2 = kMode == kDown && !kContig ? args.unit_w2[i] : -1;
                m.pb = r.x >> 1;
                m.single = r.x & 1;
                m.e = r.y;
                if (kContig) {
                    m.l0 = ExpertLoc{0, 3 * r.y + (kMode == kGateUp ? 0 : 2)};
                    m.l1 = ExpertLoc{0, 3 * r.y + (kMode == kGateUp ? 1 : 2)};
                } else if (kMode == kGateUp) {
                    m.l0 = unpack_loc(r.z);
                    m.l1 = unpack_loc(r.w);
                } else {
                    m.l0 = unpack_loc(w2);
                    m.l1 = m.l0;
                }
            };
            auto meta_valid = [&](const TileMeta& m) {
                return kMode == kGateUp ? (m.l0.map >= 0 && m.l1.map >= 0) : m.l0.map >= 0;
            };
            // the first tile from tt on with valid weights (false: none left)
            auto find_valid = [&](int64_t& tt, TileMeta& m) -> bool {
                for (; tt < ntiles; tt += ncl) {
                    meta_load(m, tt);
                    if (meta_valid(m)) return true;
                }
                return false;
            };
            int64_t t = cid;
            TileMeta cur;
            bool have = find_valid(t, cur);
            while (have && ok) {
                const int pb = cur.pb, nt = cur.nt;
                const bool single = cur.single != 0;
                const ExpertLoc l0 = cur.l0, l1 = cur.l1;
                if (!publish(pb, single, nt, t)) { ok = false; break; }
                // this CTA's token rows (a pair: its own block, the MMA's A; a single block: its
                // 64-row half, the MMA's B): sorted rows, or hidden itself for a shared-chunk block
                const CUtensorMap* am = single ? &maps.a64 : &maps.a;
                int row_a = single ? pb * 128 + (int)rank * 64 : (pb + (int)rank) * 128;
                if (kMode == kGateUp && args.sh.direct) {
                    const int e = cur.e;
                    if (e >= args.sh.E) {
                        am = single ? &maps.hid64 : &maps.hid;
                        row_a = shared_token_row(args.sh, e, row_a, npad);
                    }
                }
                const CUtensorMap* wm;
                const CUtensorMap* wm2 = nullptr;   // single gate/up: the W3 box after the W1 box
                int row_b, row_b2 = 0;
                if (kMode == kGateUp) {
                    if (single) {
                        wm = &maps.w64[l0.map];
                        wm2 = &maps.w64[l1.map];
                        row_b = l0.page * args.f + nt * 128 + (int)rank * 64;
                        row_b2 = l1.page * args.f + nt * 128 + (int)rank * 64;
                    } else {
                        wm = leader ? &maps.w[l0.map] : &maps.w[l1.map];
                        row_b = (leader ? l0.page : l1.page) * args.f + nt * 128;
                    }
                } else {
                    wm = &maps.w[l0.map];
                    row_b = l0.page * args.d + nt * BN + (int)rank * 128;
                }
                const uint32_t tx = single ? 2 * (A64_BYTES + B_BYTES) : 2 * STAGE_BYTES;
                int64_t tn = t + ncl;
                TileMeta nxt;
                if (tn < ntiles) meta_load(nxt, tn);
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
                    const uint32_t fb_leader = map_to_rank(full_bar(stage), 0);
                    if (leader) mbar_arrive_expect_tx(full_bar(stage), tx);
                    const uint32_t sa = sbase + stage * STAGE_BYTES;
                    if (single) {
                        // weights into the A half of the stage, the 64 token rows into the B half
                        tma_load_2d_pair(sa, wm, fb_leader, kb * BK, row_b);
                        if (wm2) tma_load_2d_pair(sa + A64_BYTES, wm2, fb_leader, kb * BK, row_b2);
                        tma_load_2d_pair(sa + A_BYTES, am, fb_leader, kb * BK, row_a);
                    } else {
                        tma_load_2d_pair(sa, am, fb_leader, kb * BK, row_a);
                        tma_load_2d_pair(sa + A_BYTES, wm, fb_leader, kb * BK, row_b);
                    }
                    pend_phase[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok || tn >= ntiles) break;
                if (!meta_valid(nxt)) {
                    tn += ncl;
                    if (!find_valid(tn, nxt)) break;
                }
                t = tn;
                cur = nxt;
            }
            if (ok) publish(-1, false, 0, 0);
            if (!ok && leader) {
                volatile int never = 0;
                for (int s = 0; s < STAGES; ++s)
                    if (pend_phase[s] >= 0) mbar_wait(full_bar(s), (uint32_t)pend_phase[s], &never, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int mslot = 0;
            uint32_t mphase = 0;
            bool ok = true;
            while (ok) {
                if (!mbar_wait(mfull_bar(mslot), mphase, abort_flag, args.err)) break;
                const int4 m = tile_ring[mslot];
                mbar_arrive(mempty_bar(mslot));
                if (++mslot == kTileRing) { mslot = 0; mphase ^= 1u; }
                if (m.x < 0) break;
                const int t = m.z;
                (void)t;
                const uint32_t idesc = (m.x & 1) ? kIdescSwap : kIdesc;
                GTRACE(t, 7, globaltimer());
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.err)) break;
                tc_fence_after();
                GTRACE(t, 0, globaltimer());
#ifdef PMOE_GEMM_TRACE
                long long waited = 0;
#endif
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < args.k_blocks; ++kb) {
#ifdef PMOE_GEMM_TRACE
                    const long long c0 = clock64();
#endif
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, args.err)) { ok = false; break; }
#ifdef PMOE_GEMM_TRACE
                    waited += clock64() - c0;
                    if (kb == 0) GTRACE(t, 1, globaltimer());
#endif
                    tc_fence_after();
                    const uint32_t sa = sbase + stage * STAGE_BYTES;
                    const uint64_t adesc = smem_desc(sa);
                    const uint64_t bdesc = smem_desc(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_pair(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                                 (kb | k) != 0 ? 1u : 0u);
                    mma_commit_pair(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair(tfull_bar(acc));
                GTRACE(t, 2, globaltimer());
                GTRACE(t, 3, waited);
#ifdef PMOE_GEMM_TRACE
                {
                    uint32_t smid;
                    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
                    GTRACE(t, 5, smid);
                }
#endif
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        int mslot = 0;
        uint32_t mphase = 0;
        const uint32_t ybox = bar0 + 1024u + (uint32_t)(quad * 2 * kYBox);   // down: this warp's boxes
        int ysel = 0;
        // lane 0 waits and the warp follows its verdict, so the warp never splits before the
        // warp-wide TMEM loads
        auto warp_wait = [&](uint32_t bar, uint32_t par) -> bool {
            int ok = 0;
            if (lane == 0) ok = mbar_wait(bar, par, abort_flag, args.err) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();   // orders lane 0's acquire before the other lanes' reads
            return ok != 0;
        };
        for (;;) {
            if (!warp_wait(mfull_bar(mslot), mphase)) break;
            const int4 m = tile_ring[mslot];
            __syncwarp();
            if (lane == 0) mbar_arrive(mempty_bar(mslot));
            if (++mslot == kTileRing) { mslot = 0; mphase ^= 1u; }
            if (m.x < 0) break;
            const int pb = m.x >> 1, nt = m.y, t = m.z;
            const bool single = (m.x & 1) != 0;
            (void)t;
            if (!warp_wait(tfull_bar(acc), acc_phase)) break;
            tc_fence_after();
            if (leader && lane == 0 && quad == 0) GTRACE(t, 6, globaltimer());
            const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
            if (single) {
                // TMEM lanes: this CTA's 128 weight rows; columns: the block's tokens
                // pb*128 + 0..127 (the leader's B rows first)
                if (kMode == kGateUp) {
                    // lanes 0..63 (quads 0, 1) gate, 64..127 (quads 2, 3) up, of the outputs
                    // n0 + 64*rank + fi; the up warps pass their values to the gate warps
                    const int fi = (quad & 1) * 32 + lane;
                    const bool up_half = quad >= 2;
                    float* xch = reinterpret_cast<float*>(sgen + STAGES * STAGE_BYTES + 1024);
                    uint16_t* hcol = static_cast<uint16_t*>(args.out) + (int64_t)pb * 128 * args.f +
                                     nt * 128 + (int)rank * 64 + fi;
#pragma unroll 1
                    for (int c0 = 0; c0 < 128; c0 += 16) {
                        float v[16];
                        tmem_ld16(taddr + c0, v);
                        tmem_wait_ld();
                        if (up_half) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) xch[j * 64 + fi] = v[j];
                        }
                        asm volatile("bar.sync 1, 128;" ::: "memory");
                        if (!up_half) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                hcol[(int64_t)(c0 + j) * args.f] = f32_to_bf16_bits(silu_mul(v[j], xch[j * 64 + fi]));
                        }
                        asm volatile("bar.sync 1, 128;" ::: "memory");
                    }
                } else {
                    // lanes: output columns nt*256 + rank*128 + quad*32 + lane
                    const int dcol = nt * BN + (int)rank * 128 + quad * 32 + lane;
                    const bool in = nt * BN + (int)rank * 128 + quad * 32 < args.d;   // whole warp
                    uint16_t* ycol = static_cast<uint16_t*>(args.out) + (int64_t)pb * 128 * args.d + dcol;
#pragma unroll 1
                    for (int c0 = 0; c0 < 128; c0 += 16) {
                        float v[16];
                        tmem_ld16(taddr + c0, v);
                        tmem_wait_ld();
                        if (in) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) ycol[(int64_t)(c0 + j) * args.d] = f32_to_bf16_bits(v[j]);
                        }
                    }
                }
            } else if (kMode == kGateUp) {
                const int64_t grow = (int64_t)(pb + (int)rank) * 128 + row;
                uint16_t* h = static_cast<uint16_t*>(args.out) + grow * args.f + nt * 128;
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    float g[16], u[16];
                    tmem_ld16(taddr + c0, g);
                    tmem_ld16(taddr + 128 + c0, u);
                    tmem_wait_ld();
                    uint32_t p[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        p[i] = pack_bf16(silu_mul(g[2 * i], u[2 * i]), silu_mul(g[2 * i + 1], u[2 * i + 1]));
                    uint4* dst = reinterpret_cast<uint4*>(h + c0);
                    dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                    dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                }
            } else {
                // bf16 rows through shared memory and TMA stores (whole 128-byte lines)
                const int r0 = nt * BN;
                const int yrow = (pb + (int)rank) * 128 + quad * 32;
#pragma unroll 1
                for (int c0 = 0; c0 < BN && r0 + c0 < args.d; c0 += 64) {
                    store_rows_bf16x64(&maps.y, ybox + (uint32_t)(ysel * kYBox), taddr + c0, lane, r0 + c0, yrow);
                    ysel ^= 1;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
            if (leader && lane == 0 && quad == 0) GTRACE(t, 4, globaltimer());
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (kMode == kDown && lane == 0) bulk_wait_all();   // stores done before the CTA exits
    }

    // the roles above run on one lane of their warp; the warp converges before the block barrier
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync();            // the leader's MMAs no longer read the peer's shared memory
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
    }
}

template <int kMode, bool kContig>
cudaError_t launch2(const Tc2Maps& maps, const Tc2Args& a, int grid, cudaStream_t s) {
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(tc_gemm2sm_kernel<kMode, kContig>),
                                     smem_bytes<kMode>(), &attr);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_gemm2sm_kernel<kMode, kContig>, dim3(grid), dim3(kThreads),
                      smem_bytes<kMode>(), s, maps, a);
}

}  // namespace

cudaError_t launch_tc_gemm2sm(int mode, bool contig, const CUtensorMap& act, const CUtensorMap& act64,
                              const CUtensorMap* wmaps, const CUtensorMap* wmaps64,
                              const int4* units, const int32_t* unit_w2, const int2* unit_group,
                              const int32_t* meta, void* out, int64_t out_rows, int f, int d,
                              int64_t units_max, int num_sms, int32_t* err, cudaStream_t s,
                              const CUtensorMap* hid, const CUtensorMap* hid64, SharedRows sh,
                              int shared_units) {
    Tc2Maps maps;
    maps.a = act;
    maps.a64 = act64;
    for (int i = 0; i < 3; ++i) {
        maps.w[i] = wmaps[i];
        maps.w64[i] = wmaps64[i];
    }
    maps.hid = hid ? *hid : act;
    maps.hid64 = hid64 ? *hid64 : act64;
    maps.y = act;
    if (mode == kDown && !encode_rows_map(&maps.y, out, out_rows, d, 32)) return cudaErrorInvalidValue;
    Tc2Args a{};
    a.units = units;
    a.unit_w2 = unit_w2;
    a.unit_group = unit_group;
    a.shared_units = shared_units;
    a.meta = meta;
    a.out = out;
    a.f = f;
    a.d = d;
    a.err = err;
    a.sh = hid ? sh : SharedRows{};
    if (mode == kGateUp) {
        a.k_blocks = d / BK;
        a.n_tiles = f / 128;
    } else {
        a.k_blocks = f / BK;
        a.n_tiles = (d + BN - 1) / BN;
    }
    // gate/up: the expert-major order once one expert's W1 | W3 take more than a quarter of L2
    // (Mixtral-shaped experts: 235 MB; the other layer shapes fit many times).  Measured on the
    // Mixtral-shaped layer at 8192 tokens: DRAM reads per launch 14.3 GB -> 2.1 GB, gate/up
    // 2.42 -> 2.09 ms.  The down GEMM keeps the unit-major order: its K (= f) makes a unit's h rows
    // as large as an N tile of W2, and the expert-major order made no measurable difference there
    // (3.5 against 2.9-3.4 GB read, 1.14 against 1.06-1.13 ms over three captures).
    a.raster = (mode == kGateUp && (size_t)2 * f * d * 2 > kRasterBytes) ? 1 : 0;
    const int64_t tiles = units_max * a.n_tiles;
    int64_t clusters = num_sms / 2;
    if (tiles < clusters) clusters = tiles > 0 ? tiles : 1;
    const int grid = (int)(2 * clusters);
    if (mode == kGateUp)
        return contig ? launch2<kGateUp, true>(maps, a, grid, s) : launch2<kGateUp, false>(maps, a, grid, s);
    return contig ? launch2<kDown, true>(maps, a, grid, s) : launch2<kDown, false>(maps, a, grid, s);
}

#ifdef PMOE_GEMM_TRACE
extern "C" int pmoe_gemm2_trace_read(int mode, unsigned long long* host, int n) {
    if (mode < 1 || mode > 2 || n > kTraceTiles * kTraceWords) return -1;
    return (int)cudaMemcpyFromSymbol(host, g_gemm2_trace, sizeof(unsigned long long) * n,
                                     sizeof(unsigned long long) * kTraceTiles * kTraceWords * (mode - 1));
}
extern "C" int pmoe_gemm2_trace_clear() {
    static unsigned long long zeros[2 * kTraceTiles * kTraceWords];
    return (int)cudaMemcpyToSymbol(g_gemm2_trace, zeros, sizeof(zeros));
}
#endif

}  // namespace pmoe

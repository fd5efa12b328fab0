// The paged MoE layer for a few tokens (T <= 16) in one persistent kernel whose CTAs own whole
// columns of the intermediate dimension.
//
// The layer is Rimuru's paged fused MoE (paper-daily.com/en, "Expert weights are scattered across
// pages. How does the kernel read them?"): every active expert's gate/up projection, SiLU-and-mul
// and down projection, with the expert's three matrices read in place from pool pages or
// load-buffer slots (addr_e(n, t) = B_P + p_e(n)*f*d + (n mod f)*d + t, one lookup per tile).  At
// a few tokens the layer is a stream of those pages.  The fused decode kernel (tc_fused.cu) splits
// that stream over the SMs by k-blocks, so most gate/up tiles are summed across CTAs before their
// h can feed the down projection, and that hand-off, not bandwidth, sets its time at one token.
// Here the split follows the intermediate dimension instead:
//
//   * the active experts' intermediate columns are cut into tiles of 64 (shared chunks first, then
//     the routed experts in ascending id); with NT tiles over G CTAs, CTA c < G' takes tiles c,
//     c + G', c + 2 G', ... where G' = ceil(NT / ceil(NT / G)), so the tiles divide evenly over
//     the CTAs that work (HBM, not the SM count, bounds the stream: 76 or more of the 152 SMs
//     stream a fixed volume as fast as all of them);
//   * a CTA computes the gate/up projection of its tiles over the whole K = d (no partial sums),
//     applies SiLU-and-mul (h = bf16(silu(g) * u), the activation every path feeds the down
//     projection) and the token's routing weight in the epilogue, and keeps h' = w_{t,e} * h in
//     its own shared memory as two bf16 parts, h'_hi + h'_lo, whose sum carries h' to 17 bits;
//   * it then computes the down projection restricted to its own columns, y_c = W2[:, its
//     columns] h'[its columns], for all d output rows, and stores that fp32 partial; after the one
//     grid barrier of the call each CTA sums a slice of the output over the partials in CTA order
//     and rounds it to bf16.
//
// The routing weight goes into h' because the down projection is linear, so one partial per CTA
// covers every expert it touched: out_t = sum_c y_c[t].  Rounding w * h itself to bf16 instead
// would move the rounding point off the definition's bf16(h) by up to 2^-9 per element, an error
// that grows from layer to layer of a model; the low part keeps it below 2^-17.  It takes the
// down MMA's rows after the tokens' own (N = 2 MT for at most MT = 8 or 16 tokens, one kernel
// instance each), so the down projection still needs one MMA per k-step.
//
// The first tile of each CTA c < g0 is a shared-chunk tile fixed before routing (tile c), so those
// CTAs stream it while the tokens are routed.  Roles: warp 0 the TMA producer, warp 1 the MMA
// issuer, warps 2..9 route every token (in every CTA), warps 2..5 then run the epilogues, and all
// eight the combine.  The MMA's M side holds 128 weight rows (64 W1 over the 64 W3 rows of the
// same columns for gate/up; 128 W2 rows for the down projection), its N side the 16 token slots
// (gate/up) or the MT tokens' h'_hi rows followed by their h'_lo rows (down projection).  All
// waits are bounded; a time-out sets the error word and the kernel unwinds.  The grid barrier
// needs every CTA resident: one CTA per SM.
#include <math.h>

#include "decode_common.cuh"
#include "route_common.cuh"
#include "tc_common.cuh"

namespace pmoe {

namespace {

using namespace tc;
using namespace dec;

constexpr int SBK = 64;                        // k-block (elements)
constexpr int BN = 16;                         // gate/up MMA N: token slots
constexpr int kThreads = 320;                  // 10 warps
constexpr int kW = 128 * SBK * 2;              // 16 KB weight operand per stage
constexpr int kAct = BN * SBK * 2;             // 2 KB token tile of a gate/up stage
constexpr int kStage = kW + kAct;
constexpr int kSmemMax = 232448;               // 227 KB opt-in dynamic shared memory

// shared-memory tables after the ring and the h' tiles (byte offsets)
constexpr int kTabMask = 0;                                  // u32 [1024] tokens of each expert
constexpr int kTabSlotOf = kTabMask + 4096;                  // i16 [1024] expert -> slot
constexpr int kTabSlotExpert = kTabSlotOf + 2048;            // i16 [1024] slot -> expert
constexpr int kTabIds = kTabSlotExpert + 2048;               // i32 [16][16] routing ids
constexpr int kTabW = kTabIds + 1024;                        // f32 [16][16] routing weights
constexpr int kTabMisc = kTabW + 1024;                       // i32 [64]
constexpr int kTabXch = kTabMisc + 256;                      // f32 [16][64] up -> gate lanes; after
                                                             // the barrier [4][8][32] combine sums
constexpr int kTabBytes = (kTabXch + BN * 64 * 4 + 127) / 128 * 128;
constexpr uint32_t kTmemCols = 512;            // gate/up accumulators 2 x 16, down <= 480 columns
constexpr uint32_t kIdesc = idesc_bf16(128, BN);

// The sizes that follow from MT, the most tokens a kernel instance takes (8 or 16).
template <int MT>
struct SCfg {
    static constexpr int DN = 2 * MT;                   // down MMA N: MT rows of h'_hi, MT of h'_lo
    static constexpr int HTILE = DN * SBK * 2;          // one h' tile (2 or 4 KB)
    static constexpr int PASS = MT == 8 ? 28 : 14;      // output blocks per down pass: 32 + PASS*DN <= 480
    static constexpr int GROUPS = (PASS + 3) / 4;       // the epilogue takes a pass's blocks four at a time
    static constexpr int STAGES_RAW = (kSmemMax - 1024 - kSliceMaxTiles * HTILE - kTabBytes - 512) / kStage;
    static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
    static constexpr uint32_t IDESC_DN = idesc_bf16(128, DN);
    static constexpr int SMEM = 1024 + STAGES * kStage + kSliceMaxTiles * HTILE + kTabBytes + 512;
    static_assert(kStage % 1024 == 0 && HTILE % 1024 == 0, "operands keep 1024-byte alignment");
    static_assert(SMEM <= kSmemMax, "shared memory budget");
    static_assert(32 + PASS * DN <= (int)kTmemCols, "tensor memory budget");
};

struct SMaps {
    CUtensorMap x;        // hidden [T][d], boxes of 16 rows x 64
    CUtensorMap w64[3];   // pool / load buffer 0 / 1 as [pages*f][d], boxes of 64 rows
    CUtensorMap wf[3];    // pool / load buffer 0 / 1 as [pages*d][f], boxes of 128 rows
};

// Barrier of the G CTAs of a call on one 64-bit counter that every call raises by exactly G
// (each CTA adds 1 once its partial is written, release): the call's target is the next multiple
// of G above the value its CTAs read at entry, which some of them may already have raised, never
// all.  Run by one thread per CTA; bounded: gives up after ~2 s (or when the CTA already
// aborted, after arriving), raising PMOE_ERR_TIMEOUT.
__device__ bool count_barrier(unsigned long long* ctr, unsigned long long target, volatile int* abort_flag,
                              int32_t* err) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(ctr) : "memory");
    if (*abort_flag) return false;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((it & 15u) == 0 && (*abort_flag || globaltimer() - t0 > 2000000000ull)) {
            if (!*abort_flag) {
                *abort_flag = 1;
                raise_error(err, PMOE_ERR_TIMEOUT);
            }
            return false;
        }
        __nanosleep(32);
    }
}

#ifdef PMOE_SLICE_TRACE
__device__ unsigned long long g_slice_trace[kFusedMaxGrid * 32];
// the time stamp is taken where the macro stands (the clobber keeps it after a preceding barrier)
__device__ __forceinline__ unsigned long long trace_time() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    return t;
}
#define TRACE(i) (g_slice_trace[blockIdx.x * 32 + (i)] = trace_time())
#define TRACEV(i, v) (g_slice_trace[blockIdx.x * 32 + (i)] = (unsigned long long)(v))
#else
#define TRACE(i) ((void)0)
#define TRACEV(i, v) ((void)0)
#endif

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    slice_decode_kernel(const __grid_constant__ SMaps maps, const FusedArgs args) {
    using C = SCfg<MT>;
    constexpr int kStages = C::STAGES;
    constexpr int kHTile = C::HTILE;
    constexpr int kPassTiles = C::PASS;
    constexpr int kPassGroups = C::GROUPS;
    constexpr int DN = C::DN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    const uint32_t hbase = sbase + kStages * kStage;   // h' tiles
    uint8_t* tab = sgen + kStages * kStage + kSliceMaxTiles * kHTile;
    uint32_t* tok_mask = reinterpret_cast<uint32_t*>(tab + kTabMask);
    int16_t* slot_of = reinterpret_cast<int16_t*>(tab + kTabSlotOf);
    int16_t* slot_expert = reinterpret_cast<int16_t*>(tab + kTabSlotExpert);
    int32_t* ids_s = reinterpret_cast<int32_t*>(tab + kTabIds);
    float* w_s = reinterpret_cast<float*>(tab + kTabW);
    int32_t* misc = reinterpret_cast<int32_t*>(tab + kTabMisc);
    float* xch = reinterpret_cast<float*>(tab + kTabXch);
    // misc: [0..7] scan scratch, [8] routed experts Ar, [9] abort, [10] TMEM address,
    //       [11] barrier decision, [12..13] arrival counter at entry (low, high), [14] CTAs
    //       that work (G'), [15] this CTA's tiles
    const uint32_t bar0 = sbase + kStages * kStage + kSliceMaxTiles * kHTile + kTabBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto gfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto gempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
    const uint32_t dempty_bar = bar0 + 8u * (2 * kStages + 4);
    const uint32_t route_bar = bar0 + 8u * (2 * kStages + 5);
    const uint32_t mmadone_bar = bar0 + 8u * (2 * kStages + 6);
    // down accumulators of output blocks 4q .. 4q+3 of a pass complete
    auto dfull_bar = [&](int q) { return bar0 + 8u * (2 * kStages + 7 + q); };
    auto hready_bar = [&](int j) { return bar0 + 8u * (2 * kStages + 7 + kPassGroups + j); };   // h' tile j written
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 9);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc + 10);
    volatile int* decision = reinterpret_cast<volatile int*>(misc + 11);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int T = args.T, E = args.E, S = args.S;
    const int F64 = args.f / SBK, KB1 = args.d / SBK;
    const int M2 = (args.d + 127) / 128;
    // the down projection's output blocks in passes of at most kPassTiles accumulators
    const int n_pass = (M2 + kPassTiles - 1) / kPassTiles;
    const int MP = (M2 + n_pass - 1) / n_pass;
    const uint32_t all_tok = (1u << T) - 1u;   // T <= MT <= 16
    const bool primed_tile = cta < args.g0;     // first tile = shared tile `cta`, known now

    if (threadIdx.x == 0) TRACE(25);   // entry
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(gfull_bar(a), 1);
            mbar_init(gempty_bar(a), 4);
        }
        for (int q = 0; q < kPassGroups; ++q) mbar_init(dfull_bar(q), 1);
        mbar_init(dempty_bar, 4);
        mbar_init(route_bar, 1);
        mbar_init(mmadone_bar, 1);
        for (int j = 0; j < kSliceMaxTiles; ++j) mbar_init(hready_bar(j), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    if (threadIdx.x == 0) TRACE(0);   // set-up done

    auto slot_expert_of = [&](int a) { return a < S ? E + a : (int)slot_expert[a]; };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int pend[kStages];       // parity of the last fill issued into each stage, -1: none
            for (int s = 0; s < kStages; ++s) pend[s] = -1;
            // expert pages are read once per call: keep them from displacing the partials and
            // tables in L2
            const uint64_t wpol = policy_evict_first();
            // before the previous kernel has finished: the first ring of the shared tile's
            // weights (tables and pages are inputs that no kernel of this library writes)
            int primed = 0;
            if (primed_tile) {
                const int a = cta / F64, ft = cta - (cta / F64) * F64;
                const int2 l0 = resolve(args, E + a, 0), l1 = resolve(args, E + a, 1);
                for (int kb = 0; kb < KB1 && kb < kStages; ++kb) {
                    const uint32_t sa = sbase + kb * kStage;
                    mbar_arrive_expect_tx(full_bar(kb), kStage);
                    tma_load_2d_hint(sa, &maps.w64[l0.x], full_bar(kb), kb * SBK, l0.y * args.f + ft * 64, wpol);
                    tma_load_2d_hint(sa + kW / 2, &maps.w64[l1.x], full_bar(kb), kb * SBK,
                                     l1.y * args.f + ft * 64, wpol);
                    pend[kb] = 0;
                    ++primed;
                }
            }
            pdl_wait_prev();
            pdl_allow_next();
            TRACE(1);   // producer: ring primed, previous kernel done
            bool ok = true;
            // gate/up of tile u (slot a = u / F64): W1 and W3 rows of its 64 columns and the
            // token tile, k-block by k-block; the first `skip` stages already hold the weights
            auto stream_gu = [&](int u, int skip) -> bool {
                const int a = u / F64, ft = u - a * F64;
                const int e = slot_expert_of(a);
                const int2 l0 = resolve(args, e, 0), l1 = resolve(args, e, 1);
                const int row0 = l0.y * args.f + ft * 64, row1 = l1.y * args.f + ft * 64;
                for (int kb = 0; kb < KB1; ++kb) {
                    const uint32_t fb = full_bar(stage);
                    const uint32_t sa = sbase + stage * kStage;
                    if (kb >= skip) {
                        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.err)) return false;
                        mbar_arrive_expect_tx(fb, kStage);
                        tma_load_2d_hint(sa, &maps.w64[l0.x], fb, kb * SBK, row0, wpol);
                        tma_load_2d_hint(sa + kW / 2, &maps.w64[l1.x], fb, kb * SBK, row1, wpol);
                    }
                    tma_load_2d(sa + kW, &maps.x, fb, kb * SBK, 0);
                    pend[stage] = (int)phase;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                return true;
            };
            int j0 = 0;
            if (primed_tile) {
                ok = stream_gu(cta, primed);
                j0 = 1;
            }
            if (ok && !mbar_wait(route_bar, 0, abort_flag, args.err)) ok = false;
            TRACE(2);   // producer: routing known
            const int Gw = ok ? misc[14] : 1, nt = ok ? misc[15] : 0;
            // down projection of tile j, pass p: 128 W2 rows of its 64 columns per output block
            int2 l2[kSliceMaxTiles];
            int ftj[kSliceMaxTiles];
            for (int j = 0; ok && j < nt; ++j) {
                const int u = cta + j * Gw, a = u / F64;
                ftj[j] = u - a * F64;
                l2[j] = resolve(args, slot_expert_of(a), 2);
            }
            auto stream_dn = [&](int p, int j) -> bool {
                const int m1 = min(M2, (p + 1) * MP);
                for (int m = p * MP; m < m1; ++m) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.err)) return false;
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, kW);
                    tma_load_2d_hint(sbase + stage * kStage, &maps.wf[l2[j].x], fb, ftj[j] * SBK,
                                     l2[j].y * args.d + m * 128, wpol);
                    pend[stage] = (int)phase;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                return true;
            };
            // the gate/up of tile j + 1 goes before the down projection of tile j, which then finds
            // tile j's h' written
            for (int j = j0; ok && j < nt; ++j) {
                ok = stream_gu(cta + j * Gw, 0);
                if (ok && j >= 1) ok = stream_dn(0, j - 1);
            }
            TRACE(3);   // producer: gate/up loads issued
            if (ok && nt > 0) ok = stream_dn(0, nt - 1);
            for (int p = 1; ok && p < n_pass; ++p)
                for (int j = 0; ok && j < nt; ++j) ok = stream_dn(p, j);
            TRACE(4);   // producer: all loads issued
            if (!ok) {
                // wait for this CTA's copies in flight before it may exit
                volatile int never = 0;
                for (int s = 0; s < kStages; ++s)
                    if (pend[s] >= 0) mbar_wait(full_bar(s), (uint32_t)pend[s], &never, nullptr);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        pdl_wait_prev();
        pdl_allow_next();
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            auto mma_gu = [&](int j) -> bool {
                const int g = j & 1;
                if (!mbar_wait(gempty_bar(g), (((uint32_t)j >> 1) & 1u) ^ 1u, abort_flag, args.err)) return false;
                tc_fence_after();
                const uint32_t d0 = tmem_base + (uint32_t)(g * BN);
                for (int kb = 0; kb < KB1; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, args.err)) return false;
                    tc_fence_after();
                    const uint32_t sa = sbase + stage * kStage;
                    const uint64_t wd = smem_desc(sa);
                    const uint64_t xd = smem_desc(sa + kW);
#pragma unroll
                    for (int k = 0; k < SBK / 16; ++k)
                        mma_bf16(d0, wd + (uint64_t)(2 * k), xd + (uint64_t)(2 * k), kIdesc,
                                 (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(empty_bar(stage));
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                mma_commit(gfull_bar(g));
                return true;
            };
            bool ok = true;
            int j0 = 0;
            if (primed_tile) {
                ok = mma_gu(0);
                j0 = 1;
            }
            if (ok && !mbar_wait(route_bar, 0, abort_flag, args.err)) ok = false;
            const int nt = ok ? misc[15] : 0;
            // down projection of tile j over the output blocks of pass p, accumulated over the
            // tiles in TMEM (columns 2 BN + DN * block of the pass)
            auto mma_dn = [&](int p, int j) -> bool {
                if (p == 0) {
                    if (!mbar_wait(hready_bar(j), 0, abort_flag, args.err)) return false;
                    tc_fence_after();
                } else if (j == 0) {
                    // the previous pass's accumulators have been read out
                    if (!mbar_wait(dempty_bar, (uint32_t)(p - 1) & 1u, abort_flag, args.err)) return false;
                    tc_fence_after();
                }
                const uint64_t bd = smem_desc(hbase + (uint32_t)(j * kHTile));
                const int m1 = min(M2, (p + 1) * MP);
                for (int m = p * MP; m < m1; ++m) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, args.err)) return false;
                    tc_fence_after();
                    const uint32_t d0 = tmem_base + (uint32_t)(2 * BN + (m - p * MP) * DN);
                    const uint64_t ad = smem_desc(sbase + stage * kStage);
                    // columns t and MT + t: W2 h'_hi and W2 h'_lo of token t
#pragma unroll
                    for (int k = 0; k < SBK / 16; ++k)
                        mma_bf16(d0, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), C::IDESC_DN,
                                 (j > 0 || k > 0) ? 1u : 0u);
                    mma_commit(empty_bar(stage));
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                    // the last tile completes output blocks four at a time for the epilogue
                    if (j == nt - 1 && ((m - p * MP) % 4 == 3 || m == m1 - 1)) mma_commit(dfull_bar((m - p * MP) / 4));
                }
                return true;
            };
            for (int j = j0; ok && j < nt; ++j) {
                ok = mma_gu(j);
                if (ok && j >= 1) ok = mma_dn(0, j - 1);
            }
            if (ok && nt > 0) ok = mma_dn(0, nt - 1);
            for (int p = 1; ok && p < n_pass; ++p)
                for (int j = 0; ok && j < nt; ++j) ok = mma_dn(p, j);
            TRACE(13);   // MMA: all issued
            // every MMA this thread issued has completed before the TMEM is released
            mma_commit(mmadone_bar);
            volatile int never = 0;
            mbar_wait(mmadone_bar, 0, &never, nullptr);
        }
    } else {
        // ------ warps 2..9: routing; warps 2..5 the epilogues; all eight the combine ------
        const int gi = threadIdx.x - 64, gw = warp - 2;
        const bool leader = gi == 0;
        // the page tables into L2 while the previous kernel finishes (inputs no kernel here writes)
        if (!args.contig) {
            const int nt = E + 3 * (E + S);
            for (int i = gi * 32; i < nt; i += kGroupThreads * 32) {
                const int32_t* p = i < E ? args.buf_slot + i : args.page_table + (i - E);
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
            }
        }
        pdl_wait_prev();
        pdl_allow_next();
        // the arrival counter as the previous call left it (read after that call finished)
        if (leader) {
            unsigned long long v;
            asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(args.arrive) : "memory");
            misc[12] = (int32_t)(uint32_t)v;
            misc[13] = (int32_t)(uint32_t)(v >> 32);
        }
        // routing of all T tokens (each CTA on its own)
        for (int e = gi; e < E; e += kGroupThreads) tok_mask[e] = 0u;
        group_bar();
        if (leader) TRACE(17);   // routing starts
        // warp gw routes token gw, and token gw + 8 with it when there is one (T <= 16)
        static_assert(kSliceMaxTokens <= 2 * kGroupWarps, "two tokens per routing warp at most");
        {
            const int t = gw, t2 = gw + kGroupWarps;
            if (t < T) {
                const float* lg = args.logits + (int64_t)t * E;
                int32_t* io = ids_s + t * kMaxTopK;
                float* wo = w_s + t * kMaxTopK;
                // (the 8-token instance never has a second token: no pair code in it)
                if (MT > kGroupWarps && t2 < T) {
                    const float* lg2 = args.logits + (int64_t)t2 * E;
                    int32_t* io2 = ids_s + t2 * kMaxTopK;
                    float* wo2 = w_s + t2 * kMaxTopK;
                    switch (args.epl) {
                        case 1: route_token_pair<1>(lg, lg2, E, args.k, args.renorm, lane, io, wo, io2, wo2); break;
                        case 2: route_token_pair<2>(lg, lg2, E, args.k, args.renorm, lane, io, wo, io2, wo2); break;
                        case 4: route_token_pair<4>(lg, lg2, E, args.k, args.renorm, lane, io, wo, io2, wo2); break;
                        case 8: route_token_pair<8>(lg, lg2, E, args.k, args.renorm, lane, io, wo, io2, wo2); break;
                        case 16: route_token_pair<16>(lg, lg2, E, args.k, args.renorm, lane, io, wo, io2, wo2); break;
                        default: route_token_pair<32>(lg, lg2, E, args.k, args.renorm, lane, io, wo, io2, wo2); break;
                    }
                } else {
                    switch (args.epl) {
                        case 1: route_token<1>(lg, E, args.k, args.renorm, lane, io, wo); break;
                        case 2: route_token<2>(lg, E, args.k, args.renorm, lane, io, wo); break;
                        case 4: route_token<4>(lg, E, args.k, args.renorm, lane, io, wo); break;
                        case 8: route_token<8>(lg, E, args.k, args.renorm, lane, io, wo); break;
                        case 16: route_token<16>(lg, E, args.k, args.renorm, lane, io, wo); break;
                        default: route_token<32>(lg, E, args.k, args.renorm, lane, io, wo); break;
                    }
                }
                __syncwarp();
                if (lane < args.k) atomicOr(&tok_mask[io[lane]], 1u << t);
                if (MT > kGroupWarps && t2 < T && lane < args.k)
                    atomicOr(&tok_mask[(ids_s + t2 * kMaxTopK)[lane]], 1u << t2);
            }
        }
        if (leader) TRACE(18);   // this warp's tokens routed
        group_bar();
        // active routed experts in ascending id -> slots S, S+1, ...; shared chunk s -> slot s
        {
            const int e0 = gi * 4;
            int c = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) c += (e0 + i < E && tok_mask[e0 + i] != 0u) ? 1 : 0;
            const int incl = group_scan<false>(c, lane, gw, misc);
            int r = S + incl - c;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = e0 + i;
                if (e < E && tok_mask[e] != 0u) {
                    slot_of[e] = (int16_t)r;
                    slot_expert[r] = (int16_t)e;
                    ++r;
                }
            }
            if (gi == kGroupThreads - 1) misc[8] = incl;
            if (gi < S) {
                slot_of[E + gi] = (int16_t)gi;
                slot_expert[gi] = (int16_t)(E + gi);
            }
            group_bar();
        }
        if (leader) TRACE(19);   // slots assigned
        const int A = S + misc[8];
        if (cta == 0) {
            // CTA 0's routing and slot table go to the workspace, where the other paths keep their
            // routing state, so the call can be inspected afterwards (nothing here reads them)
            for (int i = gi; i < T * args.k; i += kGroupThreads) {
                const int t = i / args.k, j = i - t * args.k;
                args.ids_out[i] = ids_s[t * kMaxTopK + j];
                args.w_out[i] = w_s[t * kMaxTopK + j];
            }
            for (int a = gi; a < A; a += kGroupThreads) args.active_out[a] = slot_expert_of(a);
            if (leader) args.meta_out[kMetaActive] = A;
        }
        // the tiles: NT over G' CTAs, ceil(NT / G) at most per CTA
        if (leader) {
            const int NT = A * F64;
            const int tpc = (NT + G - 1) / G;
            const int Gw = tpc > 0 ? (NT + tpc - 1) / tpc : 1;
            int nt = cta < Gw ? (NT - cta + Gw - 1) / Gw : 0;
            if (nt > kSliceMaxTiles || (primed_tile && nt < 1)) {
                raise_error(args.err, PMOE_ERR_INVALID_ARG);   // the host sizes the call against both
                nt = 0;
                *abort_flag = 1;
            }
            misc[14] = Gw;
            misc[15] = nt;
            mbar_arrive(route_bar);
            TRACE(5);   // routing done
            TRACEV(30, nt);
            TRACEV(31, primed_tile ? 1 : 0);
        }
        group_bar();
        const int Gw = misc[14], nt = misc[15];
        const unsigned long long entry = (unsigned long long)(uint32_t)misc[12] |
                                         ((unsigned long long)(uint32_t)misc[13] << 32);
        const unsigned long long target = (entry / (unsigned)G + 1ull) * (unsigned)G;

        if (gw < 4) {
            // ---- epilogues: gate/up accumulators -> h' tiles in shared memory; down
            // accumulators -> this CTA's fp32 partial ----
            const int quad = warp & 3;
            const int col = (quad & 1) * 32 + lane;   // column of the tile (gate lanes)
            bool ep_ok = true;
            for (int j = 0; j < nt; ++j) {
                const int g = j & 1;
                const int u = cta + j * Gw, a = u / F64;
                const int e = slot_expert_of(a);
                const uint32_t mask = a < S ? all_tok : tok_mask[e];
                if (ep_ok && !mbar_wait(gfull_bar(g), ((uint32_t)j >> 1) & 1u, abort_flag, args.err)) ep_ok = false;
                if (ep_ok) tc_fence_after();
                float v[16];
                if (ep_ok) {
                    tmem_ld16(tmem_base + (uint32_t)(g * BN) + ((uint32_t)(quad * 32) << 16), v);
                    tmem_wait_ld();
                    tc_fence_before();
                }
                // the accumulator is free for tile j + 2 as soon as it is read
                __syncwarp();
                if (lane == 0) mbar_arrive(gempty_bar(g));
                if (ep_ok && quad >= 2) {
#pragma unroll
                    for (int t = 0; t < BN; ++t) xch[t * 64 + col] = v[t];
                }
                epi_bar();
                if (quad < 2) {
                    // h = bf16(silu(gate) * up), the activation the down projection consumes, and
                    // h' = w_{t,e} * h (0 for tokens not routed to e) carried exactly enough as two
                    // bf16 parts, h'_hi = bf16(h') and h'_lo = bf16(h' - h'_hi) (17 bits together), so
                    // the down projection sees the routing weight applied to the rounded h; stored
                    // as the down MMA's K-major operand (row t and row MT + t, 16-byte chunk
                    // col/8 ^ t mod 8)
                    const uint32_t hb = hbase + (uint32_t)(j * kHTile) + (uint32_t)((col & 7) * 2);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        float hv = 0.f;
                        if (ep_ok && (mask >> t & 1u)) {
                            float wt = 1.f;
                            if (a >= S)
                                for (int q = 0; q < args.k; ++q)
                                    if (ids_s[t * kMaxTopK + q] == e) wt = w_s[t * kMaxTopK + q];
                            hv = wt * bf16_lo(f32_to_bf16_bits(silu_mul(v[t], xch[t * 64 + col])));
                        }
                        const uint16_t hi = f32_to_bf16_bits(hv);
                        const uint16_t lo = f32_to_bf16_bits(hv - bf16_lo(hi));
                        const uint32_t addr = hb + (uint32_t)(t * 128) + ((uint32_t)((col >> 3) ^ (t & 7)) << 4);
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(hi) : "memory");
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr + (uint32_t)(MT * 128)), "h"(lo) : "memory");
                    }
                    // h' is read by the tensor cores next: order the stores before the async proxy
                    fence_proxy_async_shared();
                }
                epi_bar();   // h' tile j complete; xch free for the next tile
                if (quad == 0 && lane == 0) mbar_arrive(hready_bar(j));
            }
            if (gw == 0 && lane == 0) TRACE(6);   // h' complete
            float* P = args.p2 + (int64_t)cta * T * args.d;
            for (int p = 0; nt > 0 && p < n_pass; ++p) {
                const int m1 = min(M2, (p + 1) * MP);
                for (int m = p * MP; m < m1; ++m) {
                    if ((m - p * MP) % 4 == 0) {
                        if (ep_ok && !mbar_wait(dfull_bar((m - p * MP) / 4), (uint32_t)p & 1u, abort_flag, args.err))
                            ep_ok = false;
                        if (ep_ok) tc_fence_after();
                    }
                    if (!ep_ok) break;
                    float v[DN];
                    const uint32_t ta = tmem_base + (uint32_t)(2 * BN + (m - p * MP) * DN) + ((uint32_t)(quad * 32) << 16);
#pragma unroll
                    for (int c0 = 0; c0 < DN; c0 += 16) tmem_ld16(ta + (uint32_t)c0, *reinterpret_cast<float(*)[16]>(v + c0));
                    tmem_wait_ld();
                    const int r = m * 128 + quad * 32 + lane;
                    if (r < args.d) {
#pragma unroll
                        for (int t = 0; t < MT; ++t)
                            if (t < T) __stcg(P + (int64_t)t * args.d + r, v[t] + v[t + MT]);
                    }
                }
                if (ep_ok) tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dempty_bar);
            }
            if (gw == 0 && lane == 0) TRACE(10);   // partial written
        }

        // the one grid barrier of the call: every partial is written
        __syncwarp();
        group_bar();
        if (leader) TRACE(26);   // arriving
        if (leader) *decision = count_barrier(args.arrive, target, abort_flag, args.err) ? 1 : 0;
        group_bar();
        if (*decision) {
            if (leader) TRACE(11);   // barrier
            // combine: out[t][r] = bf16(sum over c < G' of partial_c[t][r]); one item is a token
            // and 32 output rows, the CTA's items cta, cta + G, ... taken four at a time; warp w
            // sums the partials c = w, w + 8, ... of each in order, then warp j < 4 adds item j's
            // eight sums in order.  Four items' loads in flight at once: their round trips to L2,
            // not the bytes, set the combine's time.
            const int ch32 = (args.d + 31) / 32;
            const int n_items = T * ch32;
            const int64_t cstride = (int64_t)T * args.d;
            float* cred = xch;   // [4][8][32] warp sums (the gate/up exchange is no longer used)
            for (int i0 = cta; i0 < n_items; i0 += 4 * G) {
                const float* src[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int item = i0 + j * G < n_items ? i0 + j * G : i0;
                    const int t = item / ch32, r = (item - t * ch32) * 32 + lane;
                    src[j] = args.p2 + (int64_t)t * args.d + (r < args.d ? r : args.d - 1);
                }
                float sj[4] = {0.f, 0.f, 0.f, 0.f};
                int c = gw;
                for (; c + 24 < Gw; c += 32) {
                    float p[4][4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q) p[j][q] = __ldcg(src[j] + (int64_t)(c + 8 * q) * cstride);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q) sj[j] += p[j][q];
                }
                for (; c < Gw; c += 8) {
                    float p[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) p[j] = __ldcg(src[j] + (int64_t)c * cstride);
#pragma unroll
                    for (int j = 0; j < 4; ++j) sj[j] += p[j];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) cred[(j * kGroupWarps + gw) * 32 + lane] = sj[j];
                group_bar();
                if (gw < 4 && i0 + gw * G < n_items) {
                    const int item = i0 + gw * G;
                    const int t = item / ch32, r = (item - t * ch32) * 32 + lane;
                    float o = 0.f;
#pragma unroll
                    for (int w = 0; w < kGroupWarps; ++w) o += cred[(gw * kGroupWarps + w) * 32 + lane];
                    if (r < args.d) args.out[(int64_t)t * args.d + r] = f32_to_bf16_bits(o);
                }
                group_bar();
            }
            if (leader) TRACE(12);   // combine done
        }
    }

    // the roles above run on one lane of their warp; the warp converges before the block barrier
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) TRACE(24);   // every role done
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
        if (lane == 0) TRACE(27);   // TMEM released
    }
}

}  // namespace

cudaError_t launch_slice_decode(const CUtensorMap& xmap, const CUtensorMap* w64, const CUtensorMap* wf,
                                const FusedArgs& a, int grid, cudaStream_t s) {
    if (grid < 1 || grid > kFusedMaxGrid || a.T < 1 || a.T > kSliceMaxTokens || kSliceMaxTokens > 16 || a.g0 < 0 ||
        a.g0 > grid)
        return cudaErrorInvalidValue;
    SMaps m;
    m.x = xmap;
    for (int i = 0; i < 3; ++i) {
        m.w64[i] = w64[i];
        m.wf[i] = wf[i];
    }
    if (a.T <= 8) {
        static std::atomic<unsigned long long> attr8{0};
        cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(slice_decode_kernel<8>), SCfg<8>::SMEM, &attr8);
        if (e != cudaSuccess) return e;
        return launch_pdl(slice_decode_kernel<8>, dim3(grid), dim3(kThreads), SCfg<8>::SMEM, s, m, a);
    }
    static std::atomic<unsigned long long> attr16{0};
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(slice_decode_kernel<16>), SCfg<16>::SMEM, &attr16);
    if (e != cudaSuccess) return e;
    return launch_pdl(slice_decode_kernel<16>, dim3(grid), dim3(kThreads), SCfg<16>::SMEM, s, m, a);
}

#ifdef PMOE_SLICE_TRACE
extern "C" int pmoe_slice_trace_read(unsigned long long* host, int n) {
    return (int)cudaMemcpyFromSymbol(host, g_slice_trace, sizeof(unsigned long long) * n);
}
#endif

}  // namespace pmoe

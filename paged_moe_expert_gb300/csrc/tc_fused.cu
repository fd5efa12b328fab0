// The whole paged MoE layer for decode-size batches (T <= 32 tokens) in one persistent kernel.
//
// At a few tokens the layer is a stream of expert pages (Rimuru, paper-daily.com/en, "Expert
// weights are scattered across pages. How does the kernel read them?": the kernel takes, per
// expert, a pool page or a load-buffer slot, and reads the rows at
// addr_e(n, t) = B_P + p_e(n)*f*d + (n mod f)*d + t, one page lookup per tile).  What limits a
// chain of short kernels there is not bandwidth but the gaps: routing before any routed page can
// be fetched, a ramp-up and a tail at every kernel boundary, and tiles that do not divide evenly
// over the SMs.  This kernel removes them:
//
//   * every CTA routes all tokens itself (the same warp routine as the routing kernel), while its
//     producer is already streaming the shared expert's pages, which need no routing;
//   * the weight stream of each projection is split evenly over the CTAs by k-block iterations
//     (stream-K), not by tiles: CTA c takes iterations [start(c), start(c+1)) of the I iterations
//     of all active experts, so every SM streams about the same number of bytes;
//   * a piece of a gate/up tile that one CTA computes is stored as an fp32 partial; the CTA whose
//     piece completes a tile (an epoch-tagged counter per tile) sums the partials, applies
//     SiLU-and-mul and publishes that tile of h with a ready word, and a helper thread issues each
//     down-projection stage's h tile as soon as its ready word is set, so the down projection of
//     finished tiles overlaps the gate/up of the rest and no grid-wide barrier sits between them;
//   * down-projection pieces are fp32 partials too, summed by the combine after the one grid
//     barrier of the call.
//
// Iteration spaces: 0 = gate/up of the shared chunks (known before routing; spread over the
// first G0 CTAs only, so pieces stay large), 1 = gate/up of the routed experts (after routing;
// split so that space 0 + space 1 is even over all CTAs), 2 = down of every active expert.
//
// Operands as in the small-batch kernels: the MMA's M side holds 128 weight rows (64 W1 rows
// stacked over the 64 W3 rows of the same output columns for gate/up; 128 W2 rows for down), its
// N side all BN tokens of the batch (rows >= T read as zeros).  A token not routed to an expert is
// computed and discarded: the tensor cores have time to spare at these sizes, and it spares the
// row gather.  Partials, h and the output are written only for routed (token, expert) pairs.
//
// Sums have a fixed order that depends only on the routing, the shapes and the grid size, so the
// output does not depend on where the pages are.  All waits (mbarriers, ready words, the grid
// barrier) are bounded; a timeout sets the error word and the kernel unwinds.  Waiting on other
// CTAs needs all CTAs resident at once: the grid is one CTA per SM, and each CTA's gate/up work
// never waits on another CTA.
#include <math.h>

#include "decode_common.cuh"
#include "route_common.cuh"
#include "tc_common.cuh"

namespace pmoe {

namespace {

using namespace tc;
using namespace dec;

constexpr int FBK = 64;                        // k-block (elements)
constexpr int kThreads = 320;                  // 10 warps
constexpr int kW = 128 * FBK * 2;              // 16 KB weight operand per stage
constexpr int kSmemMax = 232448;               // 227 KB opt-in dynamic shared memory
constexpr int kStartsLen = kFusedMaxGrid + 1;

// shared-memory tables after the ring (byte offsets)
constexpr int kTabMask = 0;                                  // u32 [1024] tokens of each expert
constexpr int kTabSlotOf = kTabMask + 4096;                  // i16 [1024] expert -> slot
constexpr int kTabSlotExpert = kTabSlotOf + 2048;            // i16 [1024] slot -> expert
constexpr int kTabIds = kTabSlotExpert + 2048;               // i32 [32][16] routing ids
constexpr int kTabW = kTabIds + 2048;                        // f32 [32][16] routing weights
constexpr int kTabStarts = kTabW + 2048;                     // i32 [3][257] CTA ranges
constexpr int kTabMisc = kTabStarts + 3 * 4 * kStartsLen + 4;   // i32 [64]
constexpr int kTabXch = (kTabMisc + 256 + 15) / 16 * 16;        // f32 [32][64] up -> gate lanes
constexpr int kTabBytes = (kTabXch + 32 * 64 * 4 + 127) / 128 * 128;

template <int BN>
struct FCfg {
    static constexpr int ACT = BN * FBK * 2;
    static constexpr int STAGE = kW + ACT;
    static constexpr int STAGES_RAW = (kSmemMax - 1024 - kTabBytes - 512) / STAGE;
    static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
    static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
    static constexpr uint32_t IDESC = idesc_bf16(128, BN);
    static constexpr int SMEM = 1024 + STAGES * STAGE + kTabBytes + 512;
};

struct Maps {
    CUtensorMap x;        // hidden [T][d], boxes of BN rows x 64
    CUtensorMap h;        // h [A_max*BN][f] in the workspace, boxes of BN rows x 64
    CUtensorMap w64[3];   // pool / load buffer 0 / 1 as [pages*f][d], boxes of 64 rows
    CUtensorMap wf[3];    // pool / load buffer 0 / 1 as [pages*d][f], boxes of 128 rows
};

// Next piece of the range [it, hi): unit u, k-blocks [kb0, kb1).  Iteration counts fit in 31
// bits (at most 1024 slots x 1024 tiles x 256 k-blocks).
__device__ __forceinline__ bool next_piece(int32_t& it, int32_t hi, int KB, int32_t& u, int& kb0,
                                           int& kb1) {
    if (it >= hi) return false;
    u = it / KB;
    kb0 = it - u * KB;
    const int32_t rem = hi - it;
    kb1 = rem < KB - kb0 ? kb0 + rem : KB;
    it += kb1 - kb0;
    return true;
}

// floor(c * I / G) without 64-bit division (c, G <= 256, I < 2^31).
__device__ __forceinline__ int32_t split_at(int32_t I, int G, int c) {
    const int32_t q = I / G, r = I - q * G;
    return c * q + (c * r) / G;
}

// Start of CTA c's share of space 0: the first G0 CTAs split its I0 iterations evenly.
__device__ __forceinline__ int32_t start0(int32_t I0, int G0, int c) {
    return split_at(I0, G0, c < G0 ? c : G0);
}

// cta_of for an even split (space 2): an estimate from the ratio, corrected against the table.
__device__ __forceinline__ int cta_of_even(const int32_t* starts, int G, int32_t x, float ratio) {
    int c = (int)((float)x * ratio);
    c = c < 0 ? 0 : (c > G - 1 ? G - 1 : c);
    while (c > 0 && starts[c] > x) --c;
    while (c < G - 1 && starts[c + 1] <= x) ++c;
    return c;
}

// The CTA whose range holds iteration x: the largest c < G with starts[c] <= x (non-empty then).
__device__ __forceinline__ int cta_of(const int32_t* starts, int G, int32_t x) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (starts[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Phase time stamps for performance work (compiled in only with -DPMOE_FUSED_TRACE): per CTA,
// 32 globaltimer readings at the milestones named where TRACE is used.
#ifdef PMOE_FUSED_TRACE
__device__ unsigned long long g_fused_trace[kFusedMaxGrid * 32];
#define TRACE(i) (g_fused_trace[blockIdx.x * 32 + (i)] = globaltimer())
#else
#define TRACE(i) ((void)0)
#endif

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    fused_decode_kernel(const __grid_constant__ Maps maps, const FusedArgs args) {
    using C = FCfg<BN>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    uint8_t* tab = sgen + STAGES * C::STAGE;
    uint32_t* tok_mask = reinterpret_cast<uint32_t*>(tab + kTabMask);
    int16_t* slot_of = reinterpret_cast<int16_t*>(tab + kTabSlotOf);
    int16_t* slot_expert = reinterpret_cast<int16_t*>(tab + kTabSlotExpert);
    int32_t* ids_s = reinterpret_cast<int32_t*>(tab + kTabIds);
    float* w_s = reinterpret_cast<float*>(tab + kTabW);
    int32_t* starts = reinterpret_cast<int32_t*>(tab + kTabStarts);   // [3][kStartsLen]
    int32_t* misc = reinterpret_cast<int32_t*>(tab + kTabMisc);
    float* xch = reinterpret_cast<float*>(tab + kTabXch);
    // misc: [0..7] scan scratch, [8] routed experts Ar, [9] abort, [10] TMEM address,
    //       [11] barrier decision, [12] epoch word at entry, [13] down stages armed,
    //       [14] first down stage, [15] producer done, [20..23] gate/up pieces written per
    //       epilogue warp
    const uint32_t bar0 = sbase + STAGES * C::STAGE + kTabBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t route_bar = bar0 + 8u * (2 * STAGES + 4);
    const uint32_t mmadone_bar = bar0 + 8u * (2 * STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 9);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc + 10);
    volatile int* decision = reinterpret_cast<volatile int*>(misc + 11);
    volatile int* w2_count = reinterpret_cast<volatile int*>(misc + 13);
    volatile int* p2_stage0 = reinterpret_cast<volatile int*>(misc + 14);
    volatile int* prod_done = reinterpret_cast<volatile int*>(misc + 15);
    volatile int* epi_cnt = reinterpret_cast<volatile int*>(misc + 20);   // [4] per epilogue warp

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int T = args.T, E = args.E, S = args.S;
    const int F64 = args.f / FBK, KB1 = args.d / FBK, KB2 = args.f / FBK;
    const int M2 = (args.d + 127) / 128;
    const uint32_t all_tok = T >= 32 ? 0xffffffffu : ((1u << T) - 1u);
    const int32_t I0 = S * F64 * KB1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4);
        }
        mbar_init(route_bar, 1);
        mbar_init(mmadone_bar, 1);
        *abort_flag = 0;
        *w2_count = 0;
        *p2_stage0 = 0;
        *prod_done = 0;
        for (int q = 0; q < 4; ++q) epi_cnt[q] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    if (threadIdx.x == 0) TRACE(0);   // set-up done

    // this CTA's range of space sp (space 0 in closed form; spaces 1, 2 from the tables, which
    // are complete once route_bar has completed)
    auto range = [&](int sp, int32_t& lo, int32_t& hi) {
        if (sp == 0) {
            lo = start0(I0, args.g0, cta);
            hi = start0(I0, args.g0, cta + 1);
        } else {
            lo = starts[sp * kStartsLen + cta];
            hi = starts[sp * kStartsLen + cta + 1];
        }
    };
    auto space_KB = [&](int sp) { return sp == 2 ? KB2 : KB1; };
    auto slot_expert_of = [&](int a) { return a < S ? E + a : (int)slot_expert[a]; };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int pend[STAGES];        // parity of the last fill issued into each stage, -1: none
            for (int s = 0; s < STAGES; ++s) pend[s] = -1;
            bool ok = true;
            // expert pages are read once per call: keep them from displacing the partials, h and
            // the tables in L2
            const uint64_t wpol = policy_evict_first();
            auto load_w = [&](int sp, int2 l0, int2 l1, int row0, int row1, int kb) {
                const uint32_t sa = sbase + stage * C::STAGE;
                if (sp < 2) {
                    tma_load_2d_hint(sa, &maps.w64[l0.x], full_bar(stage), kb * FBK, row0, wpol);
                    tma_load_2d_hint(sa + kW / 2, &maps.w64[l1.x], full_bar(stage), kb * FBK, row1, wpol);
                } else {
                    tma_load_2d_hint(sa, &maps.wf[l0.x], full_bar(stage), kb * FBK, row0, wpol);
                }
            };
            // pre-wait: the first ring of shared-chunk weights (tables and pages are inputs that no
            // kernel of this library writes)
            int primed = 0;
            {
                int32_t it, hi, u;
                range(0, it, hi);
                int kb0, kb1;
                while (primed < STAGES && next_piece(it, hi, KB1, u, kb0, kb1)) {
                    const int a = u / F64, ft = u % F64;
                    const int2 l0 = resolve(args, E + a, 0), l1 = resolve(args, E + a, 1);
                    const int row0 = l0.y * args.f + ft * 64, row1 = l1.y * args.f + ft * 64;
                    for (int kb = kb0; kb < kb1 && primed < STAGES; ++kb) {
                        mbar_arrive_expect_tx(full_bar(stage), C::STAGE);
                        load_w(0, l0, l1, row0, row1, kb);
                        pend[stage] = (int)phase;
                        ++primed;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                }
                stage = 0;
                phase = 0;
            }
            pdl_wait_prev();
            pdl_allow_next();
            TRACE(1);   // producer: first ring primed, previous kernel done
            int step = 0, n_w2 = 0;
            for (int sp = 0; sp < 3 && ok; ++sp) {
                if (sp == 1) {
                    if (!mbar_wait(route_bar, 0, abort_flag, args.err)) { ok = false; break; }
                    TRACE(2);   // producer: routing known
                }
                if (sp == 2) {
                    TRACE(3);   // producer: gate/up loads issued
                    *p2_stage0 = stage;   // the h issuer follows the down stages from here
                }
                const int KB = space_KB(sp);
                int32_t it, hi, u;
                range(sp, it, hi);
                int kb0, kb1;
                while (ok && next_piece(it, hi, KB, u, kb0, kb1)) {
                    int a, tile;
                    if (sp == 2) { a = u / M2; tile = u % M2; }
                    else { a = (sp == 1 ? S : 0) + u / F64; tile = u % F64; }
                    const int e = slot_expert_of(a);
                    int2 l0, l1;
                    int row0, row1;
                    if (sp < 2) {
                        l0 = resolve(args, e, 0);
                        l1 = resolve(args, e, 1);
                        row0 = l0.y * args.f + tile * 64;
                        row1 = l1.y * args.f + tile * 64;
                    } else {
                        l0 = resolve(args, e, 2);
                        l1 = l0;
                        row0 = l0.y * args.d + tile * 128;
                        row1 = row0;
                    }
                    for (int kb = kb0; kb < kb1; ++kb, ++step) {
                        const uint32_t fb = full_bar(stage);
                        const uint32_t sa = sbase + stage * C::STAGE;
                        if (sp == 0 && step < primed) {
                            tma_load_2d(sa + kW, &maps.x, fb, kb * FBK, 0);
                        } else {
                            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.err)) {
                                ok = false;
                                break;
                            }
                            // the stage's bytes: weights now, and the activation tile -- the token
                            // rows for gate/up here, the h tile for down from the h issuer
                            mbar_arrive_expect_tx(fb, C::STAGE);
                            load_w(sp, l0, l1, row0, row1, kb);
                            if (sp < 2) {
                                tma_load_2d(sa + kW, &maps.x, fb, kb * FBK, 0);
                            } else {
                                __threadfence_block();
                                *w2_count = ++n_w2;
                            }
                        }
                        pend[stage] = (int)phase;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                }
            }
            *prod_done = 1;
            TRACE(4);   // producer: all loads issued
            if (!ok) {
                // the h issuer completes every down stage issued here; wait for this CTA's copies
                volatile int never = 0;
                for (int s = 0; s < STAGES; ++s)
                    if (pend[s] >= 0) mbar_wait(full_bar(s), (uint32_t)pend[s], &never, nullptr);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        pdl_wait_prev();
        pdl_allow_next();
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int sp = 0; sp < 3 && ok; ++sp) {
                if (sp == 1 && !mbar_wait(route_bar, 0, abort_flag, args.err)) break;
                const int KB = space_KB(sp);
                int32_t it, hi, u;
                range(sp, it, hi);
                int kb0, kb1;
                while (ok && next_piece(it, hi, KB, u, kb0, kb1)) {
                    if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d0 = tmem_base + (uint32_t)(acc * BN);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(full_bar(stage), phase, abort_flag, args.err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t sa = sbase + stage * C::STAGE;
                        const uint64_t wd = smem_desc(sa);
                        const uint64_t xd = smem_desc(sa + kW);
#pragma unroll
                        for (int k = 0; k < FBK / 16; ++k)
                            mma_bf16(d0, wd + (uint64_t)(2 * k), xd + (uint64_t)(2 * k), C::IDESC,
                                     (kb > kb0 || k > 0) ? 1u : 0u);
                        mma_commit(empty_bar(stage));
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    mma_commit(tfull_bar(acc));
                    if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                }
            }
            TRACE(13);   // MMA: all issued
            // every MMA this thread issued has completed before the TMEM is released
            mma_commit(mmadone_bar);
            volatile int never = 0;
            mbar_wait(mmadone_bar, 0, &never, nullptr);
        }
    } else {
        // ------ warps 2..9: routing; warps 2..5 epilogues and h; warp 6 the h issuer; combine ------
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
        // this CTA's barrier word as the previous call left it (read after that call finished)
        if (leader) misc[12] = (int32_t)ld_relaxed(args.flags + cta);
        if (leader) TRACE(16);   // barrier count read
        // routing of all T tokens (each CTA on its own)
        for (int e = gi; e < E; e += kGroupThreads) tok_mask[e] = 0u;
        group_bar();
        if (leader) TRACE(17);   // routing starts
        for (int t = gw; t < T; t += kGroupWarps) {
            const float* lg = args.logits + (int64_t)t * E;
            int32_t* io = ids_s + t * kMaxTopK;
            float* wo = w_s + t * kMaxTopK;
            switch (args.epl) {
                case 1: route_token<1>(lg, E, args.k, args.renorm, lane, io, wo); break;
                case 2: route_token<2>(lg, E, args.k, args.renorm, lane, io, wo); break;
                case 4: route_token<4>(lg, E, args.k, args.renorm, lane, io, wo); break;
                case 8: route_token<8>(lg, E, args.k, args.renorm, lane, io, wo); break;
                case 16: route_token<16>(lg, E, args.k, args.renorm, lane, io, wo); break;
                default: route_token<32>(lg, E, args.k, args.renorm, lane, io, wo); break;
            }
            __syncwarp();
            if (lane < args.k) atomicOr(&tok_mask[io[lane]], 1u << t);
        }
        if (leader) TRACE(18);   // this warp's tokens routed
        group_bar();
        if (leader) TRACE(28);   // all warps routed
        // active routed experts in ascending id -> slots S, S+1, ...; shared chunk s -> slot s
        int32_t Ar;
        {
            const int e0 = gi * 4;
            int c = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) c += (e0 + i < E && tok_mask[e0 + i] != 0u) ? 1 : 0;
            const int incl = group_scan<false>(c, lane, gw, misc);
            if (leader) TRACE(29);   // slot scan
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
            Ar = misc[8];
        }
        if (leader) TRACE(19);   // slots assigned
        const int A = S + Ar;
        const int32_t I1 = Ar * F64 * KB1, I2 = A * M2 * KB2;
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
        // CTA ranges: space 0 closed form (first G0 CTAs); space 1 so that spaces 0 + 1 are even
        // over all CTAs (a prefix maximum keeps the starts non-decreasing); space 2 even
        {
            int32_t* st0 = starts;
            int32_t* st1 = starts + kStartsLen;
            int32_t* st2 = starts + 2 * kStartsLen;
            const int32_t tot = I0 + I1;
            int32_t cand = 0, s0 = 0;
            if (gi < G) {
                s0 = start0(I0, args.g0, gi);
                cand = split_at(tot, G, gi) - s0;
                cand = cand < 0 ? 0 : (cand > I1 ? I1 : cand);
            }
            const int32_t pm = group_scan<true>(cand, lane, gw, misc);
            if (gi < G) {
                st0[gi] = s0;
                st1[gi] = pm;
                st2[gi] = split_at(I2, G, gi);
            }
            if (leader) {
                st0[G] = I0;
                st1[G] = I1;
                st2[G] = I2;
            }
        }
        group_bar();
        if (leader) {
            mbar_arrive(route_bar);
            TRACE(5);   // routing done
        }
        const uint32_t bar_base = (uint32_t)misc[12];
        const uint32_t epoch = bar_base + 1u;   // tags this call's tile counters and ready words

        if (gw < 4) {
            // ---- epilogues: accumulator columns of routed tokens -> fp32 partials; the CTA that
            // completes a gate/up tile sums its partials into h and sets the tile's ready word ----
            const int quad = warp & 3;
            const int row = quad * 32 + lane;
            int acc = 0, n_epi = 0;
            uint32_t acc_phase = 0;
            bool ep_ok = true;
            for (int sp = 0; sp < 3; ++sp) {
                const int KB = space_KB(sp);
                int32_t it, hi, u;
                range(sp, it, hi);
                int kb0, kb1;
                float* P = sp == 2 ? args.p2 : args.p1 + (sp == 1 ? args.p1_base1 : 0) * (int64_t)BN * 128;
                // every epilogue warp walks all pieces and passes the same barriers; after a
                // failed wait (abort) it skips the work but keeps the barrier sequence
                while (next_piece(it, hi, KB, u, kb0, kb1)) {
                    const int a = sp == 2 ? u / M2 : (sp == 1 ? S : 0) + u / F64;
                    const uint32_t mask = a < S ? all_tok : tok_mask[slot_expert[a]];
                    // a gate/up piece that covers its whole tile is the tile's only piece: its h
                    // comes straight from the accumulator (lanes 0..63 gate, 64..127 up of the
                    // same 64 columns; the up lanes pass their values through shared memory)
                    const bool whole = sp < 2 && kb0 == 0 && kb1 == KB;
                    if (ep_ok && !mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.err)) ep_ok = false;
                    if (ep_ok) tc_fence_after();
                    const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
                    if (whole) {
                        const int col = (quad & 1) * 32 + lane;
                        const int ft = u % F64;
                        uint16_t* hrow = args.h + (int64_t)a * BN * args.f + ft * 64 + col;
#pragma unroll
                        for (int c0 = 0; c0 < BN; c0 += 16) {
                            float v[16];
                            if (ep_ok) {
                                tmem_ld16(taddr + c0, v);
                                tmem_wait_ld();
                                if (quad >= 2) {
#pragma unroll
                                    for (int j = 0; j < 16; ++j) xch[(c0 + j) * 64 + col] = v[j];
                                }
                            }
                            epi_bar();
                            if (ep_ok && quad < 2) {
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    if (mask >> (c0 + j) & 1u)
                                        hrow[(int64_t)(c0 + j) * args.f] =
                                            f32_to_bf16_bits(silu_mul(v[j], xch[(c0 + j) * 64 + col]));
                            }
                            epi_bar();
                        }
                        if (quad < 2) fence_proxy_async_global();   // h is read by TMA next
                        epi_bar();
                        if (ep_ok && quad == 0 && lane == 0)
                            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(args.hflag + a * F64 + ft),
                                         "r"(epoch)
                                         : "memory");
                        if (ep_ok) tc_fence_before();
                    } else if (ep_ok) {
                        float* dst = P + ((int64_t)(u + cta) * BN) * 128 + row;
#pragma unroll
                        for (int c0 = 0; c0 < BN; c0 += 16) {
                            float v[16];
                            tmem_ld16(taddr + c0, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (mask >> (c0 + j) & 1u) dst[(c0 + j) * 128] = v[j];
                        }
                        tc_fence_before();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(acc));
                    if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                    if (sp == 2) continue;
                    // gate/up: tell the tile completers this piece's partials are written
                    if (lane == 0) {
                        __threadfence_block();
                        epi_cnt[quad] = ++n_epi;
                    }
                }
                if (sp == 1 && leader) TRACE(6);   // gate/up epilogues done
            }
            if (leader) TRACE(10);   // down epilogues done
        } else if (gw >= 5) {
            // ---- tile completers (warps 7..9, gate/up pieces round-robin): count each piece of
            // this CTA into its tile once its partials are written; the piece that completes a
            // tile sums the tile's partials into h and sets its ready word ----
            const int nw = kGroupWarps - 5, wsel = gw - 5;
            int idx = 0;
            bool ok = true;
            for (int sp = 0; sp < 2 && ok; ++sp) {
                const int32_t* st = starts + sp * kStartsLen;
                const float* P = args.p1 + (sp == 1 ? args.p1_base1 : 0) * (int64_t)BN * 128;
                int32_t it, hi, u;
                range(sp, it, hi);
                int kb0, kb1;
                while (ok && next_piece(it, hi, KB1, u, kb0, kb1)) {
                    const int my = idx++;
                    if (my % nw != wsel) continue;
                    if (kb0 == 0 && kb1 == KB1) continue;   // a whole tile: its epilogue wrote h
                    const uint64_t t0 = globaltimer();
                    for (uint32_t w = 1;; ++w) {
                        const bool done = epi_cnt[0] > my && epi_cnt[1] > my && epi_cnt[2] > my && epi_cnt[3] > my;
                        if (done) break;
                        if ((w & 63u) == 0 && (*abort_flag || globaltimer() - t0 > 2000000000ull)) {
                            ok = false;
                            break;
                        }
                        __nanosleep(20);
                    }
                    if (!ok) break;
                    const int a = (sp == 1 ? S : 0) + u / F64, ft = u % F64;
                    const int gu = a * F64 + ft;
                    const int c_lo = cta_of(st, G, u * KB1), c_hi = cta_of(st, G, u * KB1 + KB1 - 1);
                    int last = 0;
                    if (lane == 0) {
                        int npieces = 0;
                        for (int c = c_lo; c <= c_hi; ++c) npieces += st[c] < st[c + 1] ? 1 : 0;
                        __threadfence();
                        unsigned long long* cw = args.ucnt + gu;
                        unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(cw), nv;
                        for (;;) {
                            nv = (uint32_t)(old >> 32) == epoch ? old + 1ull
                                                                 : (((unsigned long long)epoch << 32) | 1ull);
                            const unsigned long long prev = atomicCAS(cw, old, nv);
                            if (prev == old) break;
                            old = prev;
                        }
                        __threadfence();
                        last = (int)(uint32_t)nv == npieces ? 1 : 0;
                    }
                    last = __shfl_sync(0xffffffffu, last, 0);
                    if (!last) continue;
                    // h[a][n][ft*64 + 2l, +1] = bf16(silu(sum of gate partials) * sum of up partials)
                    const uint32_t mask = a < S ? all_tok : tok_mask[slot_expert[a]];
                    for (uint32_t mrem = mask; mrem;) {
                        int nn[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            nn[q] = mrem ? __ffs(mrem) - 1 : -1;
                            if (mrem) mrem &= mrem - 1;
                        }
                        float2 g[4], up[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) g[q] = up[q] = make_float2(0.f, 0.f);
                        for (int c = c_lo; c <= c_hi; ++c) {
                            const bool live = st[c] < st[c + 1];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int n = nn[q] < 0 ? 0 : nn[q];
                                const float* src = P + ((int64_t)(u + c) * BN + n) * 128 + 2 * lane;
                                const float2 vg = __ldcg(reinterpret_cast<const float2*>(src));
                                const float2 vu = __ldcg(reinterpret_cast<const float2*>(src + 64));
                                if (live) {
                                    g[q].x += vg.x; g[q].y += vg.y;
                                    up[q].x += vu.x; up[q].y += vu.y;
                                }
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (nn[q] < 0) break;
                            const float h0 = silu_mul(g[q].x, up[q].x);
                            const float h1 = silu_mul(g[q].y, up[q].y);
                            reinterpret_cast<uint32_t*>(args.h + ((int64_t)a * BN + nn[q]) * args.f + ft * 64)[lane] =
                                pack_bf16(h0, h1);
                        }
                    }
                    fence_proxy_async_global();   // h is read by the tensor-copy engine next
                    __syncwarp();
                    if (lane == 0)
                        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(args.hflag + gu), "r"(epoch)
                                     : "memory");
                }
            }
            if (!ok && lane == 0 && !*abort_flag) {
                *abort_flag = 1;
                raise_error(args.err, PMOE_ERR_TIMEOUT);
            }
        } else if (gw == 4) {
            // ---- the h issuer (warp 6): the h tile of each down stage once its gate/up tile is
            // ready; down stage i of this CTA is iteration it0 + i of space 2, so its slot and
            // k-block follow from i, and one round of the warp checks the ready words of up to 32
            // armed stages with one load each ----
            const int32_t* st2 = starts + 2 * kStartsLen;
            const int32_t it0 = st2[cta], n_total = st2[cta + 1] - it0;
            int i = 0, stage0 = -1;
            bool ok = true;
            uint64_t t0 = globaltimer();
            while (ok && i < n_total) {
                const int armed = *w2_count;
                if (armed > i) {
                    if (stage0 < 0) stage0 = *p2_stage0;
                    const int window = min(min(armed, n_total) - i, 32);
                    bool ready = false;
                    int a = 0, kb = 0;
                    if (lane < window) {
                        const int32_t x = it0 + i + lane, uu = x / KB2;
                        a = uu / M2;
                        kb = x - uu * KB2;
                        ready = ld_acquire(args.hflag + a * F64 + kb) == epoch;
                    }
                    const uint32_t bal = __ballot_sync(0xffffffffu, ready);
                    const int p = __ffs(~bal) - 1;   // ready stages in order from i
                    if (p > 0) {
                        if (i == 0 && lane == 0) TRACE(21);   // first h tile issued
                        if (lane < p) {
                            fence_proxy_async_global();
                            const int s = (stage0 + i + lane) % STAGES;
                            tma_load_2d(sbase + s * C::STAGE + kW, &maps.h, full_bar(s), kb * FBK, a * BN);
                        }
                        i += p;
                        t0 = globaltimer();
                        continue;
                    }
                }
                if (__any_sync(0xffffffffu, *abort_flag || globaltimer() - t0 > 2000000000ull)) ok = false;
                __nanosleep(20);
            }
            if (!ok) {
                if (lane == 0 && !*abort_flag) {
                    *abort_flag = 1;
                    raise_error(args.err, PMOE_ERR_TIMEOUT);
                }
                // complete every stage the producer armed (the tile reads valid memory), so no copy
                // is left in flight when the CTA exits
                for (uint32_t w = 1; !*prod_done && w < (1u << 24); ++w) __nanosleep(64);
                const int n = *w2_count;
                if (stage0 < 0) stage0 = *p2_stage0;
                for (int j = i + lane; j < n; j += 32) {
                    const int s = (stage0 + j) % STAGES;
                    tma_load_2d(sbase + s * C::STAGE + kW, &maps.h, full_bar(s), 0, 0);
                }
            }
            if (lane == 0) TRACE(22);   // all h tiles issued
        }

        // the one grid barrier of the call (it also leaves this call's epoch in every CTA's word):
        // every down partial is written
        __syncwarp();
        group_bar();
        if (leader) TRACE(26);
        if (gw == 0) {
            const bool ok = !*abort_flag && grid_barrier(args.flags, G, cta, epoch, lane, abort_flag, args.err);
            if (leader) *decision = ok ? 1 : 0;
        }
        group_bar();
        if (*decision) {
            if (leader) TRACE(11);   // barrier
            // combine: out[t] = bf16(sum_j w[t,j] * y[t, e_j] + sum_s y[t, E+s]) in that order,
            // one warp per (token, 32 output rows); items go round-robin over the CTAs first
            const int32_t* st = starts + 2 * kStartsLen;
            const float ratio2 = (float)G / (float)I2;
            const int ch32 = (args.d + 31) / 32;
            const int npair = args.k + S;
            for (int32_t item = gw * G + cta; item < T * ch32; item += G * kGroupWarps) {
                const int t = item / ch32, m = (item - t * ch32) * 32 + lane;
                const int mt = m >> 7, r = m < args.d ? (m & 127) : 0;
                float acc_o = 0.f;
                for (int j0 = 0; j0 < npair; j0 += 8) {
                    int64_t u2[8];
                    int c0[8], c1[8];
                    float wj[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int j = j0 + q < npair ? j0 + q : npair - 1;
                        const int a = j < args.k ? slot_of[ids_s[t * kMaxTopK + j]] : j - args.k;
                        wj[q] = j < args.k ? w_s[t * kMaxTopK + j] : 1.f;
                        u2[q] = (int64_t)a * M2 + mt;
                        c0[q] = cta_of_even(st, G, (int32_t)(u2[q] * KB2), ratio2);
                        c1[q] = cta_of_even(st, G, (int32_t)(u2[q] * KB2 + KB2 - 1), ratio2);
                    }
                    // loads are unconditional (clamped to a written piece) so they all issue at
                    // once; what they contribute is selected afterwards
                    float p[8][4];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int c = c0[q] + i <= c1[q] ? c0[q] + i : c1[q];
                            const float v = __ldcg(args.p2 + ((u2[q] + c) * BN + t) * 128 + r);
                            p[q][i] = (c0[q] + i <= c1[q] && st[c] < st[c + 1]) ? v : 0.f;
                        }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (j0 + q >= npair) break;
                        float y = 0.f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) y += p[q][i];
                        for (int c = c0[q] + 4; c <= c1[q]; ++c)   // a unit split over > 4 CTAs
                            if (st[c] < st[c + 1]) y += __ldcg(args.p2 + ((u2[q] + c) * BN + t) * 128 + r);
                        acc_o = fmaf(wj[q], y, acc_o);
                    }
                }
                if (leader) TRACE(23);   // combine: first item's partials summed
                if (m < args.d) args.out[(int64_t)t * args.d + m] = f32_to_bf16_bits(acc_o);
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(C::TMEM_COLS)
                     : "memory");
    }
}

template <int BN>
cudaError_t launch_bn(const Maps& maps, const FusedArgs& a, int grid, cudaStream_t s) {
    using C = FCfg<BN>;
    static_assert(C::SMEM <= kSmemMax, "shared memory budget");
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(fused_decode_kernel<BN>), C::SMEM, &attr);
    if (e != cudaSuccess) return e;
    return launch_pdl(fused_decode_kernel<BN>, dim3(grid), dim3(kThreads), C::SMEM, s, maps, a);
}

}  // namespace

cudaError_t launch_fused_decode(const CUtensorMap& xmap, const CUtensorMap& hmap,
                                const CUtensorMap* w64, const CUtensorMap* wf, const FusedArgs& a,
                                int bn, int grid, cudaStream_t s) {
    if (grid < 1 || grid > kFusedMaxGrid || a.g0 < 1 || a.g0 > grid) return cudaErrorInvalidValue;
    Maps m;
    m.x = xmap;
    m.h = hmap;
    for (int i = 0; i < 3; ++i) {
        m.w64[i] = w64[i];
        m.wf[i] = wf[i];
    }
    if (bn == 16) return launch_bn<16>(m, a, grid, s);
    if (bn == 32) return launch_bn<32>(m, a, grid, s);
    return cudaErrorInvalidValue;
}

#ifdef PMOE_FUSED_TRACE
extern "C" int pmoe_fused_trace_read(unsigned long long* host, int n) {
    return (int)cudaMemcpyFromSymbol(host, g_fused_trace, sizeof(unsigned long long) * n);
}
#endif

}  // namespace pmoe

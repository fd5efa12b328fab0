// Paged expert GEMMs for small token counts on the tensor cores, with the operands swapped:
// the MMA's M side (128 lanes) holds expert weight rows and its N side holds the few tokens of
// a sorted block (BN = 16..128).  At decode sizes the layer is bound by streaming each active
// expert's pages once, so this kernel is a TMA streaming engine: a deep ring of weight tiles per
// SM keeps enough bytes in flight to saturate HBM, and the tensor cores do the dot products at no
// cost to the stream.
//
// The page rule is the one of Rimuru's paged kernel (paper-daily.com/en, "Expert weights are
// scattered across pages. How does the kernel read them?"): addr_e(n, t) = B_P + p_e(n)*f*d +
// (n mod f)*d + t.  A tile of expert e reads rows p_e*f + n0 .. +127 of the pool's (or a load
// buffer's) [pages*f, d] view -- one table lookup per tile, fixed strides after it.  The gate (W1)
// and up (W3) rows of the same output columns come from their two pages into two operand tiles
// that feed two accumulators, so silu(gate)*up pairs up in each epilogue thread's registers.
//
//   gate/up:  D_g[n][j] = sum_c W1_e[n0+n][c] x_j[c],  D_u likewise with W3 (x_j: the block's
//             gathered token rows);
//             h[row_j][n0+n] = bf16(silu(D_g) * D_u)
//   down:     D[r][j] = sum_{c in K split} W2_e[r0+r][c] h[row_j][c]  ->  y[split][row_j][r0+r]
//
// Warp roles as in the large-batch kernel: warp 0 TMA producer, warp 1 MMA issuer (and TMEM
// owner), warps 2-5 epilogue; two TMEM accumulator sets so the epilogue of one tile overlaps the
// next tile's loads and MMAs.  All mbarrier waits are bounded.
#include <math.h>

#include "tc_common.cuh"

namespace pmoe {

namespace {

using namespace tc;

constexpr int BK = 64;
constexpr int WROWS = 128;                  // weight rows per tile (MMA M)
constexpr int W_BYTES = WROWS * BK * 2;     // 16 KB per weight operand per stage
constexpr int kThreads = 192;
constexpr int kRingBytes = 204 * 1024;

// kGateUp:        tile = 128 W1 rows and 128 W3 rows, two accumulators (gate, up).
// kDown:          tile = 128 W2 rows.
// kGateUpStacked: tile = 64 W1 rows stacked over 64 W3 rows in one 128-row operand, one
//                 accumulator whose lanes 0..63 hold gate and 64..127 up; the epilogue pairs them
//                 through shared memory.  Half-size tiles: twice as many work items for few-token
//                 batches, so the persistent CTAs finish together.
enum { kGateUp = 1, kDown = 2, kGateUpStacked = 3 };

template <int kMode, int BN>
struct Cfg {
    static constexpr bool kGateFamily = kMode != kDown;
    static constexpr int WR = kMode == kGateUpStacked ? 64 : WROWS;   // weight rows per tile (per matrix)
    static constexpr int W_STAGE = kMode == kGateUp ? 2 * W_BYTES : W_BYTES;
    static constexpr int ACT_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = W_STAGE + ACT_BYTES;
    static constexpr int XCH_BYTES = kMode == kGateUpStacked ? 64 * BN * 4 : 0;
    static constexpr int STAGES_RAW = (kRingBytes - XCH_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
    static constexpr int ACC_COLS = (kMode == kGateUp ? 2 : 1) * BN;   // one accumulator set
    static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS < 32 ? 32 : 2 * ACC_COLS;
    static constexpr int SMEM = STAGES * STAGE_BYTES + XCH_BYTES + 1024 + 256;
    static constexpr uint32_t IDESC = idesc_bf16(WROWS, BN);
};

struct SwapArgs {
    const int32_t* sorted_ids;   // gate/up: token rows of each block are loaded straight from hidden
    int T, k, S;
    const int32_t* block_expert;
    const int32_t* meta;
    const ExpertLoc* loc;
    void* out;            // h (bf16, row stride f) or y (fp32, row stride d, split stride ystride)
    int f, d;
    int k_blocks;         // K / 64 over the whole reduction
    int w_tiles;          // weight-row tiles per block
    int splits;           // K splits (down projection only)
    int64_t ystride;      // rows per split of y
    int early;            // 1: the sort's outputs are complete at launch (see the priming below)
    int32_t* err;
    SharedRows sh;        // gate/up: shared-chunk blocks straight from hidden
    const int32_t* block_rows;   // tokens of each block (the rest of its BN rows are pads), or NULL
};

struct SwapMaps {
    CUtensorMap act;      // X_sorted [rows][d] or h [rows][f], boxes of BN rows
    CUtensorMap w[3];     // weights of pool / load buffer 0 / load buffer 1, boxes of 128 rows
    CUtensorMap hid;      // hidden [T][d], boxes of BN rows, when args.sh.direct
};

template <bool kContig>
__device__ __forceinline__ ExpertLoc loc_of(const ExpertLoc* loc, int e, int j) {
    if (kContig) return ExpertLoc{0, 3 * e + j};
    return loc[e * 3 + j];
}

template <int kMode, int BN, bool kContig>
__global__ void __launch_bounds__(kThreads, 1)
    tc_swap_kernel(const __grid_constant__ SwapMaps maps, const SwapArgs args) {
    using C = Cfg<kMode, BN>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw);
    // layout: ring | stacked-mode exchange buffer | barriers | TMEM address | abort flag
    const uint32_t bar0 = sbase + STAGES * C::STAGE_BYTES + C::XCH_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    uint32_t* tmem_holder =
        reinterpret_cast<uint32_t*>(sgen + STAGES * C::STAGE_BYTES + C::XCH_BYTES + 8 * (2 * STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4);
        }
        *abort_flag = 0;
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
    int nblocks = 0, per_block = 0, kb_per_split = 0;
    int64_t ntiles = 0;
    auto read_work = [&]() {
        nblocks = args.meta[kMetaNPadded] / BN;
        per_block = args.w_tiles * args.splits;
        ntiles = (int64_t)nblocks * per_block;
        kb_per_split = (args.k_blocks + args.splits - 1) / args.splits;
    };

    // tile t -> (block b, weight-row tile wt, split sp, k-block range)
    auto decode_tile = [&](int64_t t, int& b, int& wt, int& sp, int& kb0, int& kb1) {
        b = (int)(t / per_block);
        const int r = (int)(t % per_block);
        wt = r / args.splits;
        sp = r % args.splits;
        kb0 = sp * kb_per_split;
        kb1 = min(args.k_blocks, kb0 + kb_per_split);
    };
    auto tile_valid = [&](int b, ExpertLoc& l0, ExpertLoc& l1) {
        const int e = args.block_expert[b];
        if (C::kGateFamily) {
            l0 = loc_of<kContig>(args.loc, e, 0);
            l1 = loc_of<kContig>(args.loc, e, 1);
            return l0.map >= 0 && l1.map >= 0;
        }
        l0 = loc_of<kContig>(args.loc, e, 2);
        l1 = l0;
        return l0.map >= 0;
    };

    // The weight operand of one stage: gate/up two 128-row boxes (W1, W3); stacked a 64-row W1 box
    // over a 64-row W3 box; down one 128-row W2 box.
    auto load_weights = [&](uint32_t sa, uint32_t fb, int kb, const ExpertLoc& l0,
                            const ExpertLoc& l1, int row0, int row1) {
        tma_load_2d(sa, &maps.w[l0.map], fb, kb * BK, row0);
        if (kMode == kGateUp) tma_load_2d(sa + W_BYTES, &maps.w[l1.map], fb, kb * BK, row1);
        if (kMode == kGateUpStacked) tma_load_2d(sa + W_BYTES / 2, &maps.w[l1.map], fb, kb * BK, row1);
    };

    // Priming: expert weights do not depend on the previous kernel.  When the sort's outputs are
    // already complete at launch (args.early: the kernel before this one waited for them), the
    // producer fills the first round of the ring with weight tiles before waiting for the
    // previous kernel, whose output (the activations) only the other half of each stage needs.
    int primed = 0;
    if (args.early) {
        read_work();
        if (warp == 0 && lane == 0) {
            int stage = 0;
            for (int64_t t = blockIdx.x; t < ntiles && primed < STAGES; t += gridDim.x) {
                int b, wt, sp, kb0, kb1;
                decode_tile(t, b, wt, sp, kb0, kb1);
                ExpertLoc l0, l1;
                if (!tile_valid(b, l0, l1) || kb0 >= kb1) continue;
                const int rows_per_page = C::kGateFamily ? args.f : args.d;
                const int row0 = l0.page * rows_per_page + wt * C::WR;
                const int row1 = l1.page * rows_per_page + wt * C::WR;
                for (int kb = kb0; kb < kb1 && primed < STAGES; ++kb) {
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                    const uint32_t sa = sbase + stage * C::STAGE_BYTES;
                    load_weights(sa, fb, kb, l0, l1, row0, row1);
                    ++primed;
                    ++stage;
                }
            }
        }
    }
    // the prologue above touches no global memory the previous kernel writes
    pdl_wait_prev();
    pdl_allow_next();
    if (!args.early) read_work();

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int pend_phase[STAGES];
            for (int s = 0; s < STAGES; ++s) pend_phase[s] = -1;
            bool ok = true;
            int step = 0;   // (tile, k-block) steps issued; the first `primed` have their weights
            const int npad = args.meta[kMetaNPadded];
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                int b, wt, sp, kb0, kb1;
                decode_tile(t, b, wt, sp, kb0, kb1);
                ExpertLoc l0, l1;
                if (!tile_valid(b, l0, l1) || kb0 >= kb1) continue;
                const int rows_per_page = C::kGateFamily ? args.f : args.d;
                const int row0 = l0.page * rows_per_page + wt * C::WR;
                const int row1 = l1.page * rows_per_page + wt * C::WR;
                // the block's token rows: sorted rows, or hidden itself for a shared-chunk block
                const CUtensorMap* am = &maps.act;
                int arow = b * BN;
                if (C::kGateFamily && args.sh.direct) {
                    const int e = args.block_expert[b];
                    if (e >= args.sh.E) {
                        am = &maps.hid;
                        arow = shared_token_row(args.sh, e, b * BN, npad);
                    }
                }
                for (int kb = kb0; kb < kb1; ++kb, ++step) {
                    const uint32_t fb = full_bar(stage);
                    const uint32_t sa = sbase + stage * C::STAGE_BYTES;
                    if (step >= primed) {
                        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
                        mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                        load_weights(sa, fb, kb, l0, l1, row0, row1);
                    }
                    tma_load_2d(sa + C::W_STAGE, am, fb, kb * BK, arow);
                    pend_phase[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                volatile int never = 0;
                for (int s = 0; s < STAGES; ++s)
                    if (pend_phase[s] >= 0) mbar_wait(full_bar(s), (uint32_t)pend_phase[s], &never, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                int b, wt, sp, kb0, kb1;
                decode_tile(t, b, wt, sp, kb0, kb1);
                ExpertLoc l0, l1;
                if (!tile_valid(b, l0, l1) || kb0 >= kb1) continue;
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.err)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + (uint32_t)(acc * C::ACC_COLS);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, args.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = sbase + stage * C::STAGE_BYTES;
                    const uint64_t w0 = smem_desc(sa);
                    const uint64_t w1 = smem_desc(sa + W_BYTES);
                    const uint64_t xa = smem_desc(sa + C::W_STAGE);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
                        mma_bf16(d0, w0 + (uint64_t)(2 * k), xa + (uint64_t)(2 * k), C::IDESC, accum);
                        if (kMode == kGateUp)
                            mma_bf16(d0 + BN, w1 + (uint64_t)(2 * k), xa + (uint64_t)(2 * k), C::IDESC, accum);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar(acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else {
        const int quad = warp & 3;
        const int wrow = quad * 32 + lane;          // weight row within the tile
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            int b, wt, sp, kb0, kb1;
            decode_tile(t, b, wt, sp, kb0, kb1);
            ExpertLoc l0, l1;
            if (!tile_valid(b, l0, l1) || kb0 >= kb1) continue;
            // only the block's token columns are read out and stored: its pad columns feed rows
            // of h and y that nothing reads
            const int rows = args.block_rows ? args.block_rows[b] : BN;
            if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.err)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t)(acc * C::ACC_COLS) + ((uint32_t)(quad * 32) << 16);
            const int64_t row_base = (int64_t)b * BN;
            if (kMode == kGateUp) {
                uint16_t* h = static_cast<uint16_t*>(args.out) + wt * WROWS + wrow;
#pragma unroll 1
                for (int c0 = 0; c0 < rows; c0 += 16) {
                    float g[16], u[16];
                    tmem_ld16(taddr + c0, g);
                    tmem_ld16(taddr + BN + c0, u);
                    tmem_wait_ld();
                    uint16_t* hc = h + (row_base + c0) * args.f;
                    // (warp-uniform branch: whole chunks store without per-element tests)
                    if (rows - c0 >= 16) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) hc[(int64_t)j * args.f] = f32_to_bf16_bits(silu_mul(g[j], u[j]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < rows - c0) hc[(int64_t)j * args.f] = f32_to_bf16_bits(silu_mul(g[j], u[j]));
                    }
                }
            } else if (kMode == kGateUpStacked) {
                // lanes 64..127 (quads 2, 3) hold up, lanes 0..63 (quads 0, 1) gate, both for the
                // tile's 64 output columns: up goes through shared memory, token-major
                float* xch = reinterpret_cast<float*>(sgen + STAGES * C::STAGE_BYTES);
                const bool up_half = quad >= 2;
                const int r = wrow & 63;
                uint16_t* h = static_cast<uint16_t*>(args.out) + wt * 64 + r;
                // (rows is the same in all four epilogue warps, so each meets every named barrier)
#pragma unroll 1
                for (int c0 = 0; c0 < rows; c0 += 16) {
                    float v[16];
                    tmem_ld16(taddr + c0, v);
                    tmem_wait_ld();
                    if (up_half) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) xch[(c0 + j) * 64 + r] = v[j];
                    }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (!up_half) {
                        uint16_t* hc = h + (row_base + c0) * args.f;
                        if (rows - c0 >= 16) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                hc[(int64_t)j * args.f] = f32_to_bf16_bits(silu_mul(v[j], xch[(c0 + j) * 64 + r]));
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (j < rows - c0)
                                    hc[(int64_t)j * args.f] = f32_to_bf16_bits(silu_mul(v[j], xch[(c0 + j) * 64 + r]));
                        }
                    }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                }
            } else {
                const int r = wt * WROWS + wrow;
                float* y = static_cast<float*>(args.out) + (int64_t)sp * args.ystride * args.d + r;
#pragma unroll 1
                for (int c0 = 0; c0 < rows; c0 += 16) {
                    float v[16];
                    tmem_ld16(taddr + c0, v);
                    tmem_wait_ld();
                    if (r < args.d) {
                        float* yc = y + (row_base + c0) * args.d;
                        if (rows - c0 >= 16) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) yc[(int64_t)j * args.d] = v[j];
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (j < rows - c0) yc[(int64_t)j * args.d] = v[j];
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    // the roles above run on one lane of their warp; the warp converges before the block barrier
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(C::TMEM_COLS)
                     : "memory");
    }
}

template <int kMode, int BN, bool kContig>
cudaError_t launch_swap_one(const SwapMaps& maps, const SwapArgs& a, int grid, cudaStream_t s) {
    using C = Cfg<kMode, BN>;
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(tc_swap_kernel<kMode, BN, kContig>),
                                     C::SMEM, &attr);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_swap_kernel<kMode, BN, kContig>, dim3(grid), dim3(kThreads), C::SMEM, s, maps, a);
}

template <int kMode, bool kContig>
cudaError_t launch_swap_bn(int bn, const SwapMaps& maps, const SwapArgs& a, int grid, cudaStream_t s) {
    switch (bn) {
        case 16: return launch_swap_one<kMode, 16, kContig>(maps, a, grid, s);
        case 32: return launch_swap_one<kMode, 32, kContig>(maps, a, grid, s);
        case 64:
            if constexpr (kMode != kGateUpStacked) return launch_swap_one<kMode, 64, kContig>(maps, a, grid, s);
            return cudaErrorInvalidValue;
        case 128:
            if constexpr (kMode != kGateUpStacked) return launch_swap_one<kMode, 128, kContig>(maps, a, grid, s);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_tc_swap(int mode, bool contig, int bn, const CUtensorMap& act,
                           const CUtensorMap* wmaps, const int32_t* sorted_ids, int T, int k,
                           int S, const int32_t* block_expert, const int32_t* meta,
                           const ExpertLoc* loc, void* out, int f, int d, int splits,
                           int64_t ystride, int64_t nblk_max, int num_sms, int32_t* err,
                           int early, cudaStream_t s, const CUtensorMap* hid, SharedRows sh,
                           const int32_t* block_rows) {
    SwapMaps maps;
    maps.act = act;
    for (int i = 0; i < 3; ++i) maps.w[i] = wmaps[i];
    maps.hid = hid ? *hid : act;
    SwapArgs a{};
    a.sorted_ids = sorted_ids;
    a.T = T;
    a.k = k;
    a.S = S;
    a.block_expert = block_expert;
    a.meta = meta;
    a.loc = loc;
    a.out = out;
    a.f = f;
    a.d = d;
    a.err = err;
    a.ystride = ystride;
    a.early = early;
    a.sh = hid ? sh : SharedRows{};
    a.block_rows = block_rows;
    if (mode == kGateUp || mode == kGateUpStacked) {
        a.k_blocks = d / BK;
        a.w_tiles = f / (mode == kGateUp ? WROWS : 64);
        a.splits = 1;
    } else {
        a.k_blocks = f / BK;
        a.w_tiles = (d + WROWS - 1) / WROWS;
        a.splits = splits;
    }
    const int64_t tiles = nblk_max * a.w_tiles * a.splits;
    const int grid = (int)(tiles < num_sms ? (tiles > 0 ? tiles : 1) : num_sms);
    if (mode == kGateUp)
        return contig ? launch_swap_bn<kGateUp, true>(bn, maps, a, grid, s)
                      : launch_swap_bn<kGateUp, false>(bn, maps, a, grid, s);
    if (mode == kGateUpStacked) {
        if (bn > 32) return cudaErrorInvalidValue;   // stacked tiles serve few-token blocks
        return contig ? launch_swap_bn<kGateUpStacked, true>(bn, maps, a, grid, s)
                      : launch_swap_bn<kGateUpStacked, false>(bn, maps, a, grid, s);
    }
    return contig ? launch_swap_bn<kDown, true>(bn, maps, a, grid, s)
                  : launch_swap_bn<kDown, false>(bn, maps, a, grid, s);
}

}  // namespace pmoe

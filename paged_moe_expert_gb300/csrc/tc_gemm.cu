// Paged grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Rimuru's paged MoE kernel (paper-daily.com/en, "Expert weights are scattered across pages. How
// does the kernel read them?") resolves where an expert's weights live once per output tile and
// then reads inside a page at fixed strides:
//     addr_e(n, t) = B_P + p_e(n) * f * d + (n mod f) * d + t.
// Here that rule is a TMA coordinate: the pool (and each load buffer) is one tensor map over rows
// [pages * f, d] (gate/up pages) or [pages * d, f] (down pages), and an output tile of expert e
// loads its weight rows at row p_e * f + (n0 mod f).  The page table is read once per tile; every
// k-step after that is a fixed-stride TMA box.  Gate (W1) and up (W3) rows of the same output
// columns come from two different pages into the two halves of one B tile, so one 128x256 MMA
// produces both halves and the SiLU-and-mul epilogue pairs them in registers -- no concatenated
// copy of the weights exists anywhere.
//
// Structure: persistent CTAs (one per SM) walk the (sorted block, N tile) work list; warp 0 issues
// TMA loads into a 4-stage shared-memory ring, warp 1 issues tcgen05.mma into one of two TMEM
// accumulators (128 lanes x 256 fp32 columns each), warps 2-5 drain the other accumulator with
// tcgen05.ld and run the epilogue.  Every wait on an mbarrier is bounded; a wait that gives up
// raises the device error word and the CTA unwinds after its own copies have landed.
#include <math.h>

#include "tc_common.cuh"

namespace pmoe {

namespace {

using namespace tc;

constexpr int BM = kTcBlockM;          // 128 rows of sorted (token, expert) pairs
constexpr int BK = 64;                 // 64 bf16 = one 128-byte swizzle row
constexpr int BN = 256;                // MMA N
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_HALF = 128 * BK * 2;   // 16 KB (one TMA box of 128 rows)
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 192;          // 6 warps
constexpr uint32_t kTmemCols = 512;    // two 256-column fp32 accumulators
constexpr int kYBox = 32 * 64 * 2;     // down epilogue: one 32-row x 64-column bf16 store box
// ring, alignment slack, barriers (1 KB, keeping what follows 1024-byte aligned) and, for the down
// GEMM, two store boxes per epilogue warp
template <int kMode>
constexpr int smem_bytes() { return STAGES * STAGE_BYTES + 1024 + 1024 + (kMode == 2 ? 4 * 2 * kYBox : 0); }

constexpr uint32_t kIdesc = idesc_bf16(BM, BN);

enum { kGateUp = 1, kDown = 2 };

// Per-tile time stamps for performance work (compiled in only with -DPMOE_GEMM_TRACE): for each
// tile of the last launch of each mode, [0] globaltimer when its accumulator was free, [1] when
// its first k-block had landed, [2] after its last MMA was issued, [3] SM cycles the MMA issuer
// waited for loads, [4] globaltimer when the epilogue released the accumulator, [5] SM id,
// [6] globaltimer when the epilogue saw the accumulator full, [7] globaltimer when the MMA issuer
// began waiting for the accumulator.
#ifdef PMOE_GEMM_TRACE
constexpr int kTraceTiles = 8192;
constexpr int kTraceWords = 8;
__device__ unsigned long long g_gemm_trace[2][kTraceTiles][kTraceWords];
#define GTRACE(t, i, v) \
    do { if ((t) < kTraceTiles) g_gemm_trace[kMode - 1][(t)][(i)] = (unsigned long long)(v); } while (0)
#else
#define GTRACE(t, i, v) ((void)0)
#endif

__device__ __forceinline__ uint32_t sm_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

struct TcArgs {
    const int32_t* block_expert;
    const int32_t* meta;
    const ExpertLoc* loc;
    void* out;          // h (bf16 [cap][f]) or y (bf16 [cap][d])
    int f, d;
    int k_blocks;       // K / 64
    int n_tiles;        // N tiles per sorted block
    int32_t* err;
    SharedRows sh;         // gate/up: shared-chunk blocks straight from hidden
    const int32_t* block_rows;   // valid rows of each block (NULL: all 128)
};

struct TcMaps {
    CUtensorMap a;      // activations: X_sorted [cap][d] or h [cap][f]
    CUtensorMap w[3];   // weights of pool / load buffer 0 / load buffer 1
    CUtensorMap hid;    // hidden [T][d] (128-row boxes), when args.sh.direct
    CUtensorMap y;      // down: y bf16 [cap][d], 32-row x 64-column boxes, 128-byte swizzle
    CUtensorMap a16;    // the activation views with 16-row boxes (blocks with few valid rows)
    CUtensorMap hid16;
};

// Valid rows of block mb: the remainder of an expert's rows in its last block, 128 elsewhere.
__device__ __forceinline__ int valid_rows(const TcArgs& A, int mb) {
    return A.block_rows ? A.block_rows[mb] : BM;
}

template <bool kContig>
__device__ __forceinline__ ExpertLoc tile_loc(const ExpertLoc* loc, int e, int j) {
    if (kContig) return ExpertLoc{0, 3 * e + j};
    return loc[e * 3 + j];
}

// Location of the tile's weight matrices (gate/up: W1 and W3; down: W2), or invalid.
template <int kMode, bool kContig>
__device__ __forceinline__ bool tile_weights(const TcArgs& A, int mb, ExpertLoc& l0, ExpertLoc& l1) {
    const int e = A.block_expert[mb];
    if (kMode == kGateUp) {
        l0 = tile_loc<kContig>(A.loc, e, 0);
        l1 = tile_loc<kContig>(A.loc, e, 1);
        return l0.map >= 0 && l1.map >= 0;
    }
    l0 = tile_loc<kContig>(A.loc, e, 2);
    l1 = l0;
    return l0.map >= 0;
}

// ---- the kernel ------------------------------------------------------------------------------

template <int kMode, bool kContig>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps maps, const TcArgs args) {
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
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // the prologue above touches no global memory; from here on the previous kernel's results
    // are needed
    pdl_wait_prev();
    pdl_allow_next();

    const int nblocks = args.meta[kMetaNPadded] / BM;
    const int64_t ntiles = (int64_t)nblocks * args.n_tiles;
    auto block_of = [&](int64_t t) { return (int)(t / args.n_tiles); };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int pend_phase[STAGES];
            for (int s = 0; s < STAGES; ++s) pend_phase[s] = -1;
            bool ok = true;
            const int npad = args.meta[kMetaNPadded];
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int mb = block_of(t), nt = (int)(t % args.n_tiles);
                const int rows = valid_rows(args, mb);
                ExpertLoc l0, l1;
                if (!tile_weights<kMode, kContig>(args, mb, l0, l1)) continue;
                const CUtensorMap* w0 = &maps.w[l0.map];
                const CUtensorMap* w1 = &maps.w[l1.map];
                // the tile's token rows: sorted rows, or hidden itself for a shared-chunk block;
                // a block with fewer than 113 valid rows loads only those, in 16-row boxes (the
                // MMA's other rows hold stale data and only feed output rows nothing reads)
                const int n16 = (rows + 15) >> 4;
                const bool part = n16 < BM / 16;
                const CUtensorMap* am = part ? &maps.a16 : &maps.a;
                int arow = mb * BM;
                if (kMode == kGateUp && args.sh.direct) {
                    const int e = args.block_expert[mb];
                    if (e >= args.sh.E) {
                        am = part ? &maps.hid16 : &maps.hid;
                        arow = shared_token_row(args.sh, e, mb * BM, npad);
                    }
                }
                const uint32_t tx = (part ? (uint32_t)n16 * 16u * BK * 2u : (uint32_t)A_BYTES) + B_BYTES;
                int row0, row1;
                if (kMode == kGateUp) {
                    row0 = l0.page * args.f + nt * 128;   // W1 rows of output columns n0..n0+127
                    row1 = l1.page * args.f + nt * 128;   // W3 rows of the same columns
                } else {
                    row0 = l0.page * args.d + nt * BN;    // W2 rows (outputs) r0..r0+127
                    row1 = row0 + 128;                    // and r0+128..r0+255
                }
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, tx);
                    const uint32_t sa = sbase + stage * STAGE_BYTES;
                    if (part) {
                        for (int i = 0; i < n16; ++i)
                            tma_load_2d(sa + (uint32_t)i * 16u * BK * 2u, am, fb, kb * BK, arow + 16 * i);
                    } else {
                        tma_load_2d(sa, am, fb, kb * BK, arow);
                    }
                    tma_load_2d(sa + A_BYTES, w0, fb, kb * BK, row0);
                    tma_load_2d(sa + A_BYTES + B_HALF, w1, fb, kb * BK, row1);
                    pend_phase[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA unwinds
                volatile int never = 0;
                for (int s = 0; s < STAGES; ++s)
                    if (pend_phase[s] >= 0) mbar_wait(full_bar(s), (uint32_t)pend_phase[s], &never, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int mb = block_of(t);
                ExpertLoc l0, l1;
                if (!tile_weights<kMode, kContig>(args, mb, l0, l1)) continue;
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
                    for (int k = 0; k < BK / 16; ++k) {
                        // advance 16 elements (32 bytes) along K inside the swizzled row
                        mma_bf16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k),
                                 kIdesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar(acc));
                GTRACE(t, 2, globaltimer());
                GTRACE(t, 3, waited);
                GTRACE(t, 5, sm_id());
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else {
        // ---------------- epilogue: warps 2..5 ----------------
        const int quad = warp & 3;                 // TMEM lanes 32*quad .. 32*quad+31
        const int row = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t ybox = bar0 + 1024u + (uint32_t)(quad * 2 * kYBox);   // down: this warp's boxes
        int ysel = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int mb = block_of(t), nt = (int)(t % args.n_tiles);
            ExpertLoc l0, l1;
            if (!tile_weights<kMode, kContig>(args, mb, l0, l1)) continue;
            if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.err)) break;
            tc_fence_after();
            if (lane == 0 && quad == 0) GTRACE(t, 6, globaltimer());
            const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
            const int64_t grow = (int64_t)mb * BM + row;
            const int rows = valid_rows(args, mb);
            if (quad * 32 >= rows) {
                // no valid row in this warp's lanes: nothing to store
            } else if (kMode == kGateUp) {
                uint16_t* h = static_cast<uint16_t*>(args.out) + grow * args.f + nt * 128;
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    float g[16], u[16];
                    tmem_ld16(taddr + c0, g);          // gate columns n0 + c0 ..
                    tmem_ld16(taddr + 128 + c0, u);    // up columns of the same n
                    tmem_wait_ld();
                    uint32_t p[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float a0 = silu_mul(g[2 * i], u[2 * i]);
                        const float a1 = silu_mul(g[2 * i + 1], u[2 * i + 1]);
                        p[i] = pack_bf16(a0, a1);
                    }
                    if (row < rows) {
                        uint4* dst = reinterpret_cast<uint4*>(h + c0);
                        dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                        dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                    }
                }
            } else {
                // bf16 rows through shared memory and TMA stores: each store writes whole
                // 128-byte lines instead of one 16-byte piece of 32 different rows
                const int r0 = nt * BN;
                const int yrow = mb * BM + quad * 32;
#pragma unroll 1
                for (int c0 = 0; c0 < BN && r0 + c0 < args.d; c0 += 64) {
                    store_rows_bf16x64(&maps.y, ybox + (uint32_t)(ysel * kYBox), taddr + c0, lane, r0 + c0, yrow);
                    ysel ^= 1;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (lane == 0 && quad == 0) GTRACE(t, 4, globaltimer());
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (kMode == kDown && lane == 0) bulk_wait_all();   // stores done before the CTA exits
    }

    // the roles above run on one lane of their warp; the warp converges before the block barrier
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---- host side -------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

template <int kMode, bool kContig>
cudaError_t launch_one(const TcMaps& maps, const TcArgs& a, int grid, cudaStream_t s) {
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(tc_gemm_kernel<kMode, kContig>),
                                     smem_bytes<kMode>(), &attr);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_gemm_kernel<kMode, kContig>, dim3(grid), dim3(kThreads), smem_bytes<kMode>(),
                      s, maps, a);
}

}  // namespace

// A bf16 row-major matrix [rows][cols] as a TMA map with boxes of 64 columns x box_rows rows and
// 128-byte swizzle.
bool encode_rows_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiledFn fn = encoder();
    if (!fn || !base || rows <= 0 || cols <= 0 || (cols * 2) % 16 != 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


cudaError_t launch_tc_gemm(int mode, bool contig, const CUtensorMap& act, const CUtensorMap* wmaps,
                           const int32_t* block_expert, const int32_t* meta, const ExpertLoc* loc,
                           void* out, int64_t out_rows, int f, int d, int64_t nblk_max, int num_sms,
                           int32_t* err, cudaStream_t s, const CUtensorMap* hid, SharedRows sh,
                           const int32_t* block_rows, const CUtensorMap* act16,
                           const CUtensorMap* hid16) {
    TcMaps maps;
    maps.a = act;
    for (int i = 0; i < 3; ++i) maps.w[i] = wmaps[i];
    maps.hid = hid ? *hid : act;
    maps.a16 = act16 ? *act16 : act;
    maps.hid16 = hid16 ? *hid16 : maps.hid;
    if (block_rows && (!act16 || (hid && !hid16))) return cudaErrorInvalidValue;
    maps.y = act;
    if (mode == kDown && !encode_rows_map(&maps.y, out, out_rows, d, 32)) return cudaErrorInvalidValue;
    TcArgs a{};
    a.block_expert = block_expert;
    a.meta = meta;
    a.loc = loc;
    a.out = out;
    a.f = f;
    a.d = d;
    a.err = err;
    a.sh = hid ? sh : SharedRows{};
    a.block_rows = block_rows;
    if (mode == kGateUp) {
        a.k_blocks = d / BK;
        a.n_tiles = f / 128;
    } else {
        a.k_blocks = f / BK;
        a.n_tiles = (d + BN - 1) / BN;
    }
    const int64_t tiles = nblk_max * a.n_tiles;
    const int grid = (int)(tiles < num_sms ? (tiles > 0 ? tiles : 1) : num_sms);
    if (mode == kGateUp)
        return contig ? launch_one<kGateUp, true>(maps, a, grid, s) : launch_one<kGateUp, false>(maps, a, grid, s);
    return contig ? launch_one<kDown, true>(maps, a, grid, s) : launch_one<kDown, false>(maps, a, grid, s);
}

#ifdef PMOE_GEMM_TRACE
extern "C" int pmoe_gemm_trace_read(int mode, unsigned long long* host, int n) {
    if (mode < 1 || mode > 2 || n > kTraceTiles * kTraceWords) return -1;
    return (int)cudaMemcpyFromSymbol(host, g_gemm_trace, sizeof(unsigned long long) * n,
                                     sizeof(unsigned long long) * kTraceTiles * kTraceWords * (mode - 1));
}
extern "C" int pmoe_gemm_trace_clear() {
    static unsigned long long zeros[2 * kTraceTiles * kTraceWords];
    return (int)cudaMemcpyToSymbol(g_gemm_trace, zeros, sizeof(zeros));
}
#endif

}  // namespace pmoe

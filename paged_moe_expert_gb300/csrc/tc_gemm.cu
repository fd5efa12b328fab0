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

#include "pmoe_internal.cuh"

namespace pmoe {

namespace {

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
constexpr int kSmemBytes = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

// Instruction descriptor of tcgen05.mma.kind::f16: D fp32, A and B bf16, both K-major,
// N = 256 (bits 17..22 hold N >> 3), M = 128 (bits 24..28 hold M >> 4).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

enum { kGateUp = 1, kDown = 2 };

struct TcArgs {
    const int32_t* block_expert;
    const int32_t* meta;
    const ExpertLoc* loc;
    void* out;          // h (bf16 [cap][f]) or y (fp32 [cap][d])
    int f, d;
    int k_blocks;       // K / 64
    int n_tiles;        // N tiles per sorted block
    int32_t* err;
};

struct TcMaps {
    CUtensorMap a;      // activations: X_sorted [cap][d] or h [cap][f]
    CUtensorMap w[3];   // weights of pool / load buffer 0 / load buffer 1
};

// ---- PTX wrappers ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after ~2 s (or when another role already gave up), raising the error.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* err) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > 2000000000ull) {
                *abort_flag = 1;
                raise_error(err, PMOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes in
// 8-row (1024-byte) groups.  Start address and strides are in 16-byte units; bits 46..47 hold
// the descriptor version (1), bits 61..63 the swizzle mode (2 = 128-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)1 << 16;                            // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                            // version
    d |= (uint64_t)2 << 61;                            // SWIZZLE_128B
    return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
        " [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    return (uint32_t)f32_to_bf16_bits(a) | ((uint32_t)f32_to_bf16_bits(b) << 16);
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

    const int nblocks = args.meta[kMetaNPadded] / BM;
    const int64_t ntiles = (int64_t)nblocks * args.n_tiles;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int pend_phase[STAGES];
            for (int s = 0; s < STAGES; ++s) pend_phase[s] = -1;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int mb = (int)(t / args.n_tiles), nt = (int)(t % args.n_tiles);
                ExpertLoc l0, l1;
                if (!tile_weights<kMode, kContig>(args, mb, l0, l1)) continue;
                const CUtensorMap* w0 = &maps.w[l0.map];
                const CUtensorMap* w1 = &maps.w[l1.map];
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
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    const uint32_t sa = sbase + stage * STAGE_BYTES;
                    tma_load_2d(sa, &maps.a, fb, kb * BK, mb * BM);
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
                const int mb = (int)(t / args.n_tiles);
                ExpertLoc l0, l1;
                if (!tile_weights<kMode, kContig>(args, mb, l0, l1)) continue;
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, args.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = sbase + stage * STAGE_BYTES;
                    const uint64_t adesc = smem_desc(sa);
                    const uint64_t bdesc = smem_desc(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // advance 16 elements (32 bytes) along K inside the swizzled row
                        mma_bf16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k),
                                 (kb | k) != 0 ? 1u : 0u);
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
        // ---------------- epilogue: warps 2..5 ----------------
        const int quad = warp & 3;                 // TMEM lanes 32*quad .. 32*quad+31
        const int row = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int mb = (int)(t / args.n_tiles), nt = (int)(t % args.n_tiles);
            ExpertLoc l0, l1;
            if (!tile_weights<kMode, kContig>(args, mb, l0, l1)) continue;
            if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.err)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
            const int64_t grow = (int64_t)mb * BM + row;
            if (kMode == kGateUp) {
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
                        const float a0 = g[2 * i] / (1.f + expf(-g[2 * i])) * u[2 * i];
                        const float a1 = g[2 * i + 1] / (1.f + expf(-g[2 * i + 1])) * u[2 * i + 1];
                        p[i] = pack_bf16(a0, a1);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(h + c0);
                    dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                    dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                }
            } else {
                float* y = static_cast<float*>(args.out) + grow * args.d;
                const int r0 = nt * BN;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    float v[16];
                    tmem_ld16(taddr + c0, v);
                    tmem_wait_ld();
                    if (r0 + c0 < args.d) {
                        float4* dst = reinterpret_cast<float4*>(y + r0 + c0);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// Row gather for the gate/up GEMM: X_sorted[r] = hidden[token of pair sorted_ids[r]], zero rows
// for pads; one warp per row.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ hidden,
                                                          const int32_t* __restrict__ sorted_ids,
                                                          const int32_t* __restrict__ meta, int T,
                                                          int k, int S, int d,
                                                          uint16_t* __restrict__ x) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= meta[kMetaNPadded]) return;
    const int NR = T * k, NP = T * (k + S);
    const int pair = sorted_ids[row];
    uint4* dst = reinterpret_cast<uint4*>(x + (int64_t)row * d);
    const int dv = d >> 3;
    if (pair < NP) {
        const int t = pair < NR ? pair / k : (pair - NR) % T;
        const uint4* src = reinterpret_cast<const uint4*>(hidden + (int64_t)t * d);
        for (int c = lane; c < dv; c += 32) dst[c] = src[c];
    } else {
        for (int c = lane; c < dv; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
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
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<kMode, kContig>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    tc_gemm_kernel<kMode, kContig><<<grid, kThreads, kSmemBytes, s>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace

// A bf16 row-major matrix [rows][cols] as a TMA map with 64 x 128 boxes and 128-byte swizzle.
bool encode_rows_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encoder();
    if (!fn || !base || rows <= 0 || cols <= 0 || (cols * 2) % 16 != 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gather(const uint16_t* hidden, const int32_t* sorted_ids, const int32_t* meta,
                          int T, int k, int S, int d, int64_t cap, uint16_t* x, cudaStream_t s) {
    const unsigned grid = (unsigned)((cap + 7) / 8);
    gather_rows_kernel<<<grid, 256, 0, s>>>(hidden, sorted_ids, meta, T, k, S, d, x);
    return cudaGetLastError();
}

cudaError_t launch_tc_gemm(int mode, bool contig, const CUtensorMap& act, const CUtensorMap* wmaps,
                           const int32_t* block_expert, const int32_t* meta, const ExpertLoc* loc,
                           void* out, int f, int d, int64_t nblk_max, int num_sms, int32_t* err,
                           cudaStream_t s) {
    TcMaps maps;
    maps.a = act;
    for (int i = 0; i < 3; ++i) maps.w[i] = wmaps[i];
    TcArgs a{};
    a.block_expert = block_expert;
    a.meta = meta;
    a.loc = loc;
    a.out = out;
    a.f = f;
    a.d = d;
    a.err = err;
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

}  // namespace pmoe

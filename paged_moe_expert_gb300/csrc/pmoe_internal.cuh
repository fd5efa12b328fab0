// Internal declarations shared by the CUDA translation units of libpmoe (not installed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pmoe.h"

namespace pmoe {

constexpr int kMaxExpertsTotal = 1024;  // E + S
constexpr int kMaxTopK = 16;
constexpr int kMaxPairsPerToken = 64;   // k + S
constexpr int kTcBlockM = 128;          // tensor-core path: rows per sorted block
constexpr int kTcPairBlockM = 256;      // CTA-pair tensor-core path: rows per sorted block
constexpr int kStreamMaxBlockM = 16;    // weight-streaming path: rows per sorted block (max)
constexpr int kStreamKChunk = 2048;     // weight-streaming down GEMM: K (= f) chunk per CTA
constexpr int kFusedMaxTokens = 32;     // fused decode kernel: tokens per call (MMA N <= 32)
constexpr int kFusedMaxGrid = 256;      // fused decode kernel: CTAs (one per SM)
constexpr int kSliceMaxTokens = 16;     // column-slice decode kernel: tokens per call
constexpr int kSliceMaxTiles = 12;      // column-slice decode kernel: 64-column tiles per CTA

// Where one expert matrix lives: map 0 = pool, 1 = load buffer 0, 2 = load buffer 1; `page` is
// the page index within that map (for a buffer, 3 * slot + matrix).  map < 0: invalid.
struct ExpertLoc {
    int32_t map;
    int32_t page;
};

// Byte offsets of the workspace regions for one call (all 256-byte aligned).
struct WsLayout {
    size_t ids, w, sorted, bexp, inv, meta, loc, part, units, unit_w2, ugroup, brows, x, h, y, total;
    size_t fp1, fh, fp2;   // fused decode kernel: gate/up partials, h, down partials
    size_t sp;             // column-slice decode kernel: per-CTA partials [kFusedMaxGrid][T][d] fp32
    int64_t np;          // T * (k + S) pairs
    int64_t cap;         // rows of sorted_ids / h / y / x
    int64_t nblk_max;    // upper bound on sorted blocks
    int block_m;
    int splits;          // down-GEMM K splits (partial y buffers)
};

// meta[] slots
enum { kMetaNPadded = 0, kMetaPairs = 1, kMetaSingles = 2, kMetaActive = 3, kMetaCount = 16 };

struct Plan {
    pmoe_layer_desc desc;
    const void* pool;
    int64_t num_pages;
    const void* buf[2];
    int32_t* d_error;    // device error word
    unsigned long long* d_arrive;   // arrival counter of the column-slice decode kernel
    uint32_t* d_flags;   // grid-barrier words of the fused decode kernel (one per CTA)
    unsigned long long* d_ucnt;   // its gate/up tile counters, (E+S)*f/64 of them
    uint32_t* d_hflag;            // its gate/up tile ready words, (E+S)*f/64 of them
    size_t words_bytes;           // bytes of the plan's device words (error word onwards)
    int device;
    int path;            // pmoe_path
    bool have_tmaps;
    cudaEvent_t prof_ev[16];   // measurement hook (pmoe_plan_set_profile_events)
    int n_prof;
    int last_path, last_kernels, last_launches;  // what the last forward ran
    int last_T, last_block_m;                    // its token count and sorted block size
    int num_sms;
    // column-slice decode kernel, per token count 1..kSliceMaxTokens (set at plan creation):
    // whether every routing fits it, its g0 and the most 64-column tiles a CTA can get
    int8_t slice_fits[kSliceMaxTokens + 1];
    int slice_g0[kSliceMaxTokens + 1], slice_tiles[kSliceMaxTokens + 1];
    CUtensorMap tm_rows_d[3];  // pool / buf0 / buf1 viewed as [pages * f, d]   (W1, W3 pages)
    CUtensorMap tm_rows_d64[3];  // the same views with 64-row boxes (stacked gate/up tiles)
    CUtensorMap tm_rows_f[3];  // pool / buf0 / buf1 viewed as [pages * d, f]   (W2 pages)
};

// Sets the text pmoe_last_error() returns and passes the status through.
pmoe_status record_failure(pmoe_status s, const char* msg);

// Host checks shared by every entry point that takes a layer descriptor: sizes in range
// (desc_ok) and a shape the kernels cover (shape_supported: d % 64, f % 128, d <= 16384,
// f <= 65536).
bool desc_ok(const pmoe_layer_desc* D);
bool shape_supported(const pmoe_layer_desc* D);

// Device helpers ----------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&b);
}

// SiLU(g) * u = g / (1 + e^-g) * u with the hardware exponential and reciprocal: no
// data-dependent slow path (the pad rows of a sorted block may hold any bits, and the IEEE
// divide's slow path on their overflowing values cost a gate/up epilogue three times its time);
// the error is a few fp32 ulps, far below the bf16 rounding of h.  For g -> -inf the divisor
// overflows and the quotient is 0, the limit of SiLU.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.f + __expf(-g)) * u;
}

__device__ __forceinline__ void raise_error(int32_t* err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// Streaming 16-byte load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Programmatic dependent launch: every kernel of the library waits for the previous grid to
// finish and publish its memory (wait) before it reads or writes global memory that grid
// touches, and only then lets the next kernel in the stream start (launch_dependents).  So the
// next kernel's launch and prologue overlap this kernel's work, and a kernel may read what the
// kernel two launches back wrote before its own wait.  A kernel launched without the attribute
// returns from the wait at once.
__device__ __forceinline__ void pdl_allow_next() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prev() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Raise a kernel's dynamic shared-memory limit to `bytes`.  The attribute belongs to the current
// device's context, so it is set once per device: `done` keeps one bit per device ordinal
// (ordinals >= 64 set it on every call).  Racing first calls set the same value.
inline cudaError_t raise_smem_limit(const void* kernel, int bytes,
                                    std::atomic<unsigned long long>* done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
    if (bit && (done->load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done->fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Launch with the programmatic-stream-serialisation attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Host-side launchers (defined in the .cu files) -------------------------------------------

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                         float* w, cudaStream_t s);

struct ResolveArgs {
    const int32_t* page_table;  // [E+S][3]
    const int32_t* buf_slot;    // [E]
    int64_t num_pages;
    int32_t slots_per_buffer;
    int32_t have_buf0, have_buf1;
    int32_t contiguous;         // 1: expert e's matrix j is pool page 3e + j, tables unused
    ExpertLoc* loc;             // [E+S][3] out
    int32_t* err;
    // optional work units over the sorted blocks (NULL: not written): for each expert, its blocks
    // taken two at a time, then its odd last block; units[i] = {(first block << 1) | single,
    // expert, packed location of W1, of W3} and unit_w2[i] = packed location of W2 (pack_loc);
    // count in meta[kMetaPairs], single-block units in meta[kMetaSingles]
    int4* units;
    int32_t* unit_w2;
    // optional with units: for each unit, {first unit, number of units} of its expert (an
    // expert's units are consecutive), so a GEMM can order its tiles by expert
    int2* unit_group;
    // optional (NULL: not written): valid rows of each sorted block, 1..block_m (the last block of
    // an expert holds its remainder, the others are full)
    int32_t* block_rows;
};

// An ExpertLoc in one word, (map << 29) | page, or -1 for none (pages of a pool or a buffer are
// fewer than 2^29: a page holds at least 64 x 128 bf16).
__host__ __device__ __forceinline__ int32_t pack_loc(ExpertLoc L) {
    return L.map < 0 ? -1 : (int32_t)(((uint32_t)L.map << 29) | (uint32_t)L.page);
}
__host__ __device__ __forceinline__ ExpertLoc unpack_loc(int32_t v) {
    return v < 0 ? ExpertLoc{-1, -1} : ExpertLoc{v >> 29, v & ((1 << 29) - 1)};
}

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int S, int block_m,
                         int32_t* sorted_ids, int32_t* block_expert, int32_t* inv,
                         int32_t* meta, const ResolveArgs* resolve, cudaStream_t s);

// Sort + pad over several CTAs when there are many pairs (two launches; `part` is scratch of
// align_part_bytes()); falls back to the single-CTA kernel for few pairs.
int align_ctas(int64_t NR, int ES);
size_t align_part_bytes();
cudaError_t launch_align_multi(const int32_t* ids, int T, int k, int E, int S, int block_m,
                               int32_t* part, int32_t* sorted_ids, int32_t* block_expert,
                               int32_t* inv, int32_t* meta, const ResolveArgs* resolve,
                               cudaStream_t s);

// Small batches: routing + sort/pad/resolve + row gather (x may be NULL: no gather) in one CTA.
cudaError_t launch_prep_small(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                              float* w, int S, int block_m, int32_t* sorted_ids,
                              int32_t* block_expert, int32_t* inv, int32_t* meta,
                              const ResolveArgs& rs, const uint16_t* hidden, int d, uint16_t* x,
                              cudaStream_t s);
// X[inv[i]] = hidden[token of pair i] for all T*(k+S) pairs (pad rows untouched).
cudaError_t launch_gather_pairs(const uint16_t* hidden, const int32_t* inv, int T, int k, int S,
                                int d, uint16_t* x, cudaStream_t s);

struct LayerPtrs {
    const uint16_t* map_base[3];  // pool, buf0, buf1 (bf16 elements)
    int d, f, E, k, S, T;
};

cudaError_t launch_stream_gemm1(const LayerPtrs& L, const uint16_t* hidden,
                                const int32_t* sorted_ids, const int32_t* block_expert,
                                const int32_t* meta, const ExpertLoc* loc, int block_m,
                                int64_t nblk_max, uint16_t* h, cudaStream_t s);
cudaError_t launch_stream_gemm2(const LayerPtrs& L, const int32_t* sorted_ids,
                                const int32_t* block_expert, const int32_t* meta,
                                const ExpertLoc* loc, int block_m, int64_t nblk_max, int splits,
                                int64_t cap, const uint16_t* h, float* y, cudaStream_t s);
// y_bf16: y holds bf16 rows (no K split); else fp32 rows, `splits` partials `cap` rows apart
cudaError_t launch_combine(const void* y, bool y_bf16, int splits, int64_t cap, const float* w,
                           const int32_t* inv, int T, int d, int k, int S, uint16_t* out,
                           cudaStream_t s);

// The blocks of the shared-expert chunks hold every token in order (chunk s, sorted row
// start_s + t is token t), and those chunks are the last experts of the sorted order.  With
// `direct` set the gate/up GEMMs load those rows from hidden itself, so the row gather copies
// routed pairs only.
struct SharedRows {
    int direct;   // 1: shared-chunk blocks read hidden
    int E, S;     // routed experts, shared chunks
    int rows;     // sorted rows of one shared chunk: T rounded up to the block size
};

// Row of hidden that sorted row `srow` of expert e (>= E) holds, given the padded row count.
__device__ __forceinline__ int shared_token_row(const SharedRows& sh, int e, int srow, int npad) {
    return srow - (npad - (sh.S - (e - sh.E)) * sh.rows);
}

// Tensor-core path (tc_gemm.cu)
bool encode_rows_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                     int box_rows = 128);
// mode 1: gate/up GEMM + SiLU-and-mul -> h (bf16); mode 2: down GEMM -> y (bf16, out_rows rows)
cudaError_t launch_tc_gemm(int mode, bool contig, const CUtensorMap& act, const CUtensorMap* wmaps,
                           const int32_t* block_expert, const int32_t* meta, const ExpertLoc* loc,
                           void* out, int64_t out_rows, int f, int d, int64_t nblk_max, int num_sms,
                           int32_t* err, cudaStream_t s, const CUtensorMap* hid = nullptr,
                           SharedRows sh = SharedRows{}, const int32_t* block_rows = nullptr,
                           const CUtensorMap* act16 = nullptr, const CUtensorMap* hid16 = nullptr);

// CTA-pair tensor-core path (tc_gemm2sm.cu): the work units of `units`/`unit_w2` (count
// meta[kMetaPairs], written by the sort): a pair of consecutive 128-row blocks of one expert, or
// an expert's odd last block, with the expert's weight locations;
// mode 1 gate/up -> h, 2 down -> y (bf16, out_rows rows).  act/act64, hid/hid64: the token rows
// with 128- and 64-row boxes; wmaps64: gate/up weight views with 64-row boxes.  shared_units:
// how many of the last units belong to shared chunks (spread among the routed units in the work
// order).
cudaError_t launch_tc_gemm2sm(int mode, bool contig, const CUtensorMap& act, const CUtensorMap& act64,
                              const CUtensorMap* wmaps, const CUtensorMap* wmaps64,
                              const int4* units, const int32_t* unit_w2, const int2* unit_group,
                              const int32_t* meta, void* out, int64_t out_rows, int f, int d,
                              int64_t units_max,
                              int num_sms, int32_t* err, cudaStream_t s,
                              const CUtensorMap* hid = nullptr, const CUtensorMap* hid64 = nullptr,
                              SharedRows sh = SharedRows{}, int shared_units = 0);

// Fused decode kernel (tc_fused.cu): routing, both projections and the combine of T <= 32
// tokens in one persistent launch of `grid` CTAs (one per SM); bn = 16 or 32 >= T.  The
// column-slice decode kernel (tc_slice.cu, T <= 16) takes the same arguments: p2 holds its
// per-CTA partials [grid][T][d] fp32, g0 the CTAs whose first tile (a shared-chunk tile) is
// streamed before routing, arrive its barrier counter, and p1, h, flags, ucnt, hflag, p1_base1
// are unused (the fused kernel does not use arrive).
struct FusedArgs {
    const float* logits;        // [T][E]
    const int32_t* page_table;  // [E+S][3]
    const int32_t* buf_slot;    // [E]
    float* p1;                  // gate/up partials: [pieces][bn][128] fp32
    uint16_t* h;                // [A_max * bn][f] bf16
    float* p2;                  // down partials: [pieces][bn][128] fp32
    uint16_t* out;              // [T][d] bf16
    uint32_t* flags;            // grid-barrier words, one per CTA (plan-owned)
    unsigned long long* arrive; // column-slice kernel: CTAs arrived, +grid per call (plan-owned)
    unsigned long long* ucnt;   // per gate/up tile: (epoch << 32 | pieces done) (plan-owned)
    uint32_t* hflag;            // per gate/up tile: epoch once its h is written (plan-owned)
    int32_t* err;
    // CTA 0's routing and active-slot table, written to the workspace where the other paths keep
    // their routing state (read back by pmoe_plan_routing_view): ids [T][k], weights [T][k],
    // the expert of each active slot [A], and A in meta[kMetaActive]
    int32_t* ids_out;
    float* w_out;
    int32_t* active_out;
    int32_t* meta_out;
    int64_t num_pages;
    int64_t p1_base1;           // first piece slot of the routed gate/up space
    int g0;                     // CTAs that share the shared chunks' gate/up (1..grid)
    int T, E, k, S, renorm, d, f;
    int slots_per_buffer, have_buf0, have_buf1, contig;
    int epl;                    // logits per lane in routing: 1, 2, 4, ..., 32 (E <= 32 * epl)
};
cudaError_t launch_fused_decode(const CUtensorMap& xmap, const CUtensorMap& hmap,
                                const CUtensorMap* w64, const CUtensorMap* wf, const FusedArgs& a,
                                int bn, int grid, cudaStream_t s);
cudaError_t launch_slice_decode(const CUtensorMap& xmap, const CUtensorMap* w64, const CUtensorMap* wf,
                                const FusedArgs& a, int grid, cudaStream_t s);

// Copy-in of absent routed experts (copy_in.cu): routes the T tokens, gives every routed expert
// with buf_slot == -2 a free slot of load buffer `buf` (buf_slot updated on the device), lists
// them in missed ([0] count, [1..] experts, [1+E..] slots) and copies each from
// host_experts[e] (device-readable, 3*f*d bf16) into its slot.  Uses the plan's words at bytes
// 256..388 (routed-expert bitmap and an arrival counter), which it leaves zeroed.
cudaError_t launch_copy_in(const Plan& P, const float* logits, int T, int32_t* buf_slot, int buf,
                           const void* const* host_experts, int32_t* missed, cudaStream_t s);

// Small-batch tensor-core path (tc_decode.cu): mode 1 gate/up -> h, mode 2 down -> y partials,
// mode 3 gate/up with 64+64-row stacked tiles (bn <= 32; weight maps with 64-row boxes).
cudaError_t launch_tc_swap(int mode, bool contig, int bn, const CUtensorMap& act,
                           const CUtensorMap* wmaps, const int32_t* sorted_ids, int T, int k,
                           int S, const int32_t* block_expert, const int32_t* meta,
                           const ExpertLoc* loc, void* out, int f, int d, int splits,
                           int64_t ystride, int64_t nblk_max, int num_sms, int32_t* err,
                           int early, cudaStream_t s, const CUtensorMap* hid = nullptr,
                           SharedRows sh = SharedRows{}, const int32_t* block_rows = nullptr);

}  // namespace pmoe

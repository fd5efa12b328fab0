// C ABI of libpmoe: plans, the paged and contiguous layer forward, the double-buffered
// prefetch, event waits and error reporting.  Every device step runs in this library's own
// kernels on the caller's stream; nothing here allocates on the forward path.
#include <stdio.h>
#include <string.h>

#include <chrono>
#include <new>
#include <string>
#include <thread>

#include "pmoe_internal.cuh"

namespace pmoe {

static thread_local std::string g_last_error;

static pmoe_status fail(pmoe_status s, const char* msg) {
    g_last_error = msg;
    return s;
}

pmoe_status record_failure(pmoe_status s, const char* msg) { return fail(s, msg); }

static pmoe_status cuda_fail(cudaError_t e, const char* where) {
    g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
    return PMOE_ERR_CUDA;
}

#define PMOE_CUDA(call, where)                      \
    do {                                            \
        cudaError_t e_ = (call);                    \
        if (e_ != cudaSuccess) return cuda_fail(e_, where); \
    } while (0)

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Device words a plan owns: the error word, (at 256 B) the copy-in's routed-expert bitmap and
// arrival counter, (at 512 B) the column-slice decode kernel's arrival counter (8 B), (at 1 KB)
// one barrier word per CTA, (at 2 KB) the fused decode kernel's gate/up tile counters (8 B) and
// ready words (4 B), one per tile of f/64 columns of every expert and shared chunk.
static size_t plan_words_bytes(const pmoe_layer_desc& D) {
    const size_t tiles = (size_t)(D.num_experts + D.num_shared_chunks) * (D.f / 64);
    return 2048 + 12 * tiles;
}

bool desc_ok(const pmoe_layer_desc* D) {
    if (!D) return false;
    if (D->d <= 0 || D->f <= 0 || D->num_experts <= 0 || D->top_k <= 0) return false;
    if (D->top_k > D->num_experts || D->top_k > kMaxTopK) return false;
    if (D->num_shared_chunks < 0 || D->slots_per_buffer < 0) return false;
    if (D->num_experts + D->num_shared_chunks > kMaxExpertsTotal) return false;
    if (D->top_k + D->num_shared_chunks > kMaxPairsPerToken) return false;
    return true;
}

bool shape_supported(const pmoe_layer_desc* D) {
    return D->d % 64 == 0 && D->f % 128 == 0 && D->d <= 16384 && D->f <= 65536;
}

// Rows per sorted block on the weight-streaming path: the smallest power of two covering the
// largest possible per-expert token count (T), at most 16, and small enough for the block's
// tokens to fit in shared memory.
static int stream_block_m(const pmoe_layer_desc& D, int64_t T) {
    int bm = 1;
    while (bm < T && bm < kStreamMaxBlockM) bm <<= 1;
    while (bm > 1 && (size_t)bm * D.d * 2 > 128 * 1024) bm >>= 1;
    return bm;
}

// The automatic path, by the routed tokens per expert T*k/E (measured crossovers on GB300): up to
// 24, and up to 320 tokens, the small-batch tensor-core kernels (tokens on the MMA's N side; the
// 512-expert Zipf-routed layer crosses to 128-token blocks between 256 and 384 tokens, 512 of them
// 194.8 -> 187.9 us, 1024 244.0 -> 229.6 us); above, the CTA-pair kernels
// from 64 on for layers of at most 128 experts, else the single-CTA 128-token-block kernels (with
// hundreds of small experts most experts end in an odd block, which costs a CTA pair as much as
// a pair of blocks).  Routing and sort + pad run as one single-CTA kernel up to 128 tokens.
constexpr int kSwapMaxTokensPerExpert = 24;
constexpr int kSwapMaxTokens = 320;
// The column-slice decode kernel up to 16 tokens while no routing leaves a CTA more than 10 MiB
// of weights to stream (its column tiles x 64 columns x d x 3 matrices x 2 bytes).  Measured on
// GB300 against the fused kernel, with the layers' own routings and with routings that spread
// the tokens over the most experts: ahead or level up to 16 tokens on the Qwen1.5- and
// Qwen3-Next-shaped layers (d = 2048: at most 10 and 9 tiles, 7.9 and 7.1 MiB per CTA; 16
// tokens 140 against 144 us and 72 against 78 us), and at 1 and 2 tokens on the Mixtral-shaped
// one (d = 4096, 9.4 MiB at 2 tokens); behind beyond that (3 and more Mixtral-shaped tokens, up
// to 12 tiles = 18.9 MiB, 8-9% behind), where the fused kernel's even k-block split keeps more
// bytes in flight per SM.
constexpr int kSliceAutoTokens = 16;
constexpr int64_t kSliceAutoBytes = (int64_t)10 << 20;
constexpr int kPairMinTokensPerExpert = 64;
constexpr int kPairMaxExperts = 128;
constexpr int kPrepSmallMaxTokens = 128;
// The one-CTA prep routes every token on one SM; its routing work grows with tokens x logits per
// lane x k.  Past this the routing kernel's many CTAs and a separate sort win (measured on GB300:
// the Qwen1.5-MoE-shaped layer at 128 tokens 22.4 us in the prep against 6.1 + 12.3 us, at 40
// and 64 tokens 1-2 us; 512 experts top-10 at 64 tokens took 36 us in the prep); the
// Mixtral-shaped layer stays in the prep up to 128 tokens.
constexpr int64_t kPrepSmallRouteWork = 256;

static bool use_prep_small(int T, int E, int k) {
    return T <= kPrepSmallMaxTokens && (int64_t)T * ((E + 31) / 32) * k <= kPrepSmallRouteWork;
}

static int stream_splits(const pmoe_layer_desc& D) {
    return (D.f + kStreamKChunk - 1) / kStreamKChunk;
}

// Small-batch tensor-core path: tokens per block (MMA N), K splits of the down projection and the
// row stride of its partial outputs.  BN covers the largest per-expert token count (T, reached by
// the shared chunks) up to 128; the down projection is split along K until there are about two
// tiles per SM (taking ~160 SMs so the workspace size does not depend on the device).
struct SwapParams {
    int bn, splits;
    int64_t ystride;
};
static SwapParams swap_params(const pmoe_layer_desc& D, int64_t T) {
    SwapParams p{};
    // tokens per block: T rounded up to a power of two, at most 64 up to 128 tokens (a block of
    // 128 token rows leaves room for only four 48 KB ring stages, and with few tokens per expert
    // the deeper ring of 40 KB stages streams faster: Qwen3-Next-shaped T=128 150 -> 143 us)
    // and 128 above
    int bn = 16;
    while (bn < T && bn < (T > 128 ? 128 : 64)) bn <<= 1;
    p.bn = bn;
    const int64_t ES = D.num_experts + D.num_shared_chunks;
    const int64_t np = T * (D.top_k + D.num_shared_chunks);
    const int64_t active = ES < np ? ES : np;
    p.ystride = np + active * (bn - 1);
    const int64_t kb = D.f / 64, wt = (D.d + 127) / 128;
    int64_t sp = (320 + active * wt - 1) / (active * wt > 0 ? active * wt : 1);
    if (sp < 1) sp = 1;
    if (sp > 8) sp = 8;
    if (sp > kb) sp = kb;
    const int64_t per = (kb + sp - 1) / sp;
    p.splits = (int)((kb + per - 1) / per);   // every split non-empty
    return p;
}

// Fused decode kernel sizes for T <= kFusedMaxTokens tokens: MMA N (16 or 32), active-expert
// slots (shared chunks first), and piece slots of the stream-K partial buffers (one per unit plus
// one per CTA boundary inside a unit, for at most kFusedMaxGrid CTAs per iteration space).
struct FusedShape {
    int bn;
    int64_t a_max, u1_shared, u1_routed_max, u2_max, p1_pieces, p2_pieces;
};
static FusedShape fused_shape(const pmoe_layer_desc& D, int64_t T) {
    FusedShape F{};
    F.bn = T <= 16 ? 16 : 32;
    const int64_t routed = T * D.top_k < D.num_experts ? T * D.top_k : D.num_experts;
    F.a_max = routed + D.num_shared_chunks;
    const int64_t f64 = D.f / 64, m2 = (D.d + 127) / 128;
    F.u1_shared = D.num_shared_chunks * f64;
    F.u1_routed_max = routed * f64;
    F.u2_max = F.a_max * m2;
    F.p1_pieces = F.u1_shared + F.u1_routed_max + 2 * kFusedMaxGrid;
    F.p2_pieces = F.u2_max + kFusedMaxGrid;
    return F;
}

// One layout that serves both kernel families for up to T tokens.
static WsLayout layout(const pmoe_layer_desc& D, int64_t T) {
    WsLayout W{};
    const int64_t ES = D.num_experts + D.num_shared_chunks;
    const int64_t k = D.top_k;
    W.np = T * (k + D.num_shared_chunks);
    // rows for any block size up to the pair path's 256
    const int64_t cap_tc = (W.np + ES * (kTcPairBlockM - 1) + kTcPairBlockM - 1) / kTcPairBlockM * kTcPairBlockM;
    const int64_t cap_st = W.np + ES * (kStreamMaxBlockM - 1);
    W.cap = cap_tc > cap_st ? cap_tc : cap_st;
    W.nblk_max = W.np + ES + 1;  // any block size >= 1
    W.splits = stream_splits(D);
    size_t o = 0;
    W.ids = o;    o = align256(o + sizeof(int32_t) * T * k);
    W.w = o;      o = align256(o + sizeof(float) * T * k);
    W.sorted = o; o = align256(o + sizeof(int32_t) * W.cap);
    W.bexp = o;   o = align256(o + sizeof(int32_t) * W.nblk_max);
    W.inv = o;    o = align256(o + sizeof(int32_t) * (W.np > 0 ? W.np : 1));
    W.meta = o;   o = align256(o + sizeof(int32_t) * kMetaCount);
    W.loc = o;    o = align256(o + sizeof(ExpertLoc) * ES * 3);
    W.part = o;   o = align256(o + align_part_bytes());
    W.units = o;  o = align256(o + sizeof(int4) * W.nblk_max);
    W.unit_w2 = o; o = align256(o + sizeof(int32_t) * W.nblk_max);
    W.ugroup = o; o = align256(o + sizeof(int2) * W.nblk_max);
    W.brows = o;  o = align256(o + sizeof(int32_t) * W.nblk_max);
    W.x = o;      o = align256(o + 2 * (size_t)cap_tc * D.d);
    W.h = o;      o = align256(o + 2 * (size_t)W.cap * D.f);
    const size_t y_tc = sizeof(float) * (size_t)cap_tc * D.d;
    const size_t y_st = sizeof(float) * (size_t)W.splits * cap_st * D.d;
    const SwapParams sw = swap_params(D, T);
    const size_t y_sw = sizeof(float) * (size_t)sw.splits * sw.ystride * D.d;
    size_t y_max = y_tc > y_st ? y_tc : y_st;
    if (y_sw > y_max) y_max = y_sw;
    W.y = o;      o = align256(o + y_max);
    W.total = o;
    // fused decode kernel (T <= kFusedMaxTokens): partials and h, over the regions above
    W.fp1 = W.fh = W.fp2 = 0;
    if (T <= kFusedMaxTokens) {
        const FusedShape F = fused_shape(D, T);
        size_t q = W.x;
        W.fp1 = q; q = align256(q + sizeof(float) * (size_t)F.p1_pieces * F.bn * 128);
        W.fh = q;  q = align256(q + 2 * (size_t)F.a_max * F.bn * D.f);
        W.fp2 = q; q = align256(q + sizeof(float) * (size_t)F.p2_pieces * F.bn * 128);
        if (q > W.total) W.total = q;
    }
    // column-slice decode kernel (T <= kSliceMaxTokens): one fp32 partial of the output per CTA
    W.sp = 0;
    if (T <= kSliceMaxTokens) {
        W.sp = W.x;
        const size_t q = align256(W.sp + sizeof(float) * (size_t)kFusedMaxGrid * T * D.d);
        if (q > W.total) W.total = q;
    }
    return W;
}

// The column-slice decode kernel over `grid` CTAs: whether every routing of T tokens leaves at
// most kSliceMaxTiles 64-column tiles per CTA, and g0, the CTAs whose first tile is a shared-chunk
// tile under every routing (tile c of CTA c < G' for G' = ceil(NT / ceil(NT / grid)), NT the
// tiles of the active experts), which may stream it before routing.
static bool slice_fit(const pmoe_layer_desc& D, int64_t T, int grid, int* g0, int* tiles_max) {
    if (T < 1 || T > kSliceMaxTokens || grid < 1) return false;
    const int64_t f64 = D.f / 64, E = D.num_experts, S = D.num_shared_chunks;
    const int64_t ar_lo = D.top_k < E ? D.top_k : E;
    const int64_t ar_hi = T * D.top_k < E ? T * D.top_k : E;
    int64_t gmin = grid;
    for (int64_t ar = ar_lo; ar <= ar_hi; ++ar) {
        const int64_t nt = (S + ar) * f64;
        const int64_t tpc = (nt + grid - 1) / grid;
        if (tpc > kSliceMaxTiles) return false;
        const int64_t gw = (nt + tpc - 1) / tpc;
        if (gw < gmin) gmin = gw;
    }
    const int64_t shared_tiles = S * f64;
    *g0 = (int)(shared_tiles < gmin ? shared_tiles : gmin);
    *tiles_max = (int)(((S + ar_hi) * f64 + grid - 1) / grid);
    return true;
}

// Records the plan's i-th profiling event, if the measurement hook is set.
static cudaError_t mark(const Plan* P, int i, cudaStream_t s) {
    return (i < P->n_prof && P->prof_ev[i]) ? cudaEventRecord(P->prof_ev[i], s) : cudaSuccess;
}

template <typename T>
static T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

static pmoe_status forward_impl(Plan* P, const void* hidden, int32_t T, const float* logits,
                                int32_t top_k, const int32_t* page_table, const int32_t* buf_slot,
                                void* out, void* ws, size_t ws_bytes, cudaStream_t stream,
                                bool contig) {
    if (!P) return fail(PMOE_ERR_INVALID_ARG, "plan is NULL");
    const pmoe_layer_desc& D = P->desc;
    if (T < 0) return fail(PMOE_ERR_INVALID_ARG, "T < 0");
    if (top_k != D.top_k) return fail(PMOE_ERR_INVALID_ARG, "top_k differs from the plan's");
    if (T == 0) return PMOE_OK;
    if (!hidden || !logits || !out || !ws) return fail(PMOE_ERR_INVALID_ARG, "NULL pointer");
    if (!contig && (!page_table || (D.num_experts > 0 && !buf_slot)))
        return fail(PMOE_ERR_INVALID_ARG, "NULL page_table or buf_slot");
    if (((uintptr_t)ws & 255) || ((uintptr_t)hidden & 15) || ((uintptr_t)out & 15))
        return fail(PMOE_ERR_INVALID_ARG, "misaligned workspace (256 B) or hidden/out (16 B)");
    if ((int64_t)T * (D.top_k + D.num_shared_chunks) > (int64_t)1 << 30)
        return fail(PMOE_ERR_INVALID_ARG, "too many tokens");
    const WsLayout W = layout(D, T);
    if (ws_bytes < W.total) return fail(PMOE_ERR_WORKSPACE, "workspace too small");

    int path = P->path;
    if (path == PMOE_PATH_FUSED && T > kFusedMaxTokens)
        return fail(PMOE_ERR_UNSUPPORTED, "the fused decode kernel takes at most 32 tokens");
    const int dgrid = P->num_sms < kFusedMaxGrid ? P->num_sms : kFusedMaxGrid;   // decode kernels
    int slice_g0 = 0, slice_tiles = 0;
    bool slice_ok = false;
    if (T >= 1 && T <= kSliceMaxTokens) {   // worked out at plan creation
        slice_ok = P->slice_fits[T] != 0;
        slice_g0 = P->slice_g0[T];
        slice_tiles = P->slice_tiles[T];
    }
    if (path == PMOE_PATH_SLICE && !slice_ok)
        return fail(PMOE_ERR_UNSUPPORTED,
                    "the column-slice decode kernel takes at most 16 tokens and 12 column tiles per SM");
    if (path == PMOE_PATH_AUTO) {
        const int64_t routed = (int64_t)T * D.top_k;   // routed tokens; per expert: routed / E
        // the fused decode kernel up to 32 tokens for layers of at most 128 experts and up to 16
        // tokens otherwise (measured on GB300: with hundreds of small experts at 17..32 tokens
        // the small-batch kernels stream a little faster)
        const int fused_max = D.num_experts <= 128 ? kFusedMaxTokens : 16;
        const bool slice_auto = slice_ok && T <= kSliceAutoTokens &&
                                (int64_t)slice_tiles * 64 * D.d * 3 * 2 <= kSliceAutoBytes;
        path = slice_auto ? PMOE_PATH_SLICE
             : T <= fused_max ? PMOE_PATH_FUSED
             : (routed <= (int64_t)kSwapMaxTokensPerExpert * D.num_experts && T <= kSwapMaxTokens)
                 ? PMOE_PATH_TC_DECODE
             : (routed >= (int64_t)kPairMinTokensPerExpert * D.num_experts &&
                D.num_experts <= kPairMaxExperts) ? PMOE_PATH_TC2
             : PMOE_PATH_TC;
    }
    const bool tc_family = path == PMOE_PATH_TC || path == PMOE_PATH_TC_DECODE || path == PMOE_PATH_TC2 ||
                           path == PMOE_PATH_FUSED || path == PMOE_PATH_SLICE;
    if (tc_family && !P->have_tmaps)
        return fail(PMOE_ERR_UNSUPPORTED, "tensor maps unavailable for this plan");

    int32_t* ids = at<int32_t>(ws, W.ids);
    float* w = at<float>(ws, W.w);
    int32_t* sorted = at<int32_t>(ws, W.sorted);
    int32_t* bexp = at<int32_t>(ws, W.bexp);
    int32_t* inv = at<int32_t>(ws, W.inv);
    int32_t* meta = at<int32_t>(ws, W.meta);
    ExpertLoc* loc = at<ExpertLoc>(ws, W.loc);
    uint16_t* x = at<uint16_t>(ws, W.x);
    uint16_t* h = at<uint16_t>(ws, W.h);
    float* y = at<float>(ws, W.y);

    CUtensorMap xmap, hmap;
    const int64_t ES = D.num_experts + D.num_shared_chunks;
    const int64_t cap_tc = (W.np + ES * (kTcPairBlockM - 1) + kTcPairBlockM - 1) / kTcPairBlockM * kTcPairBlockM;
    const SwapParams sw = swap_params(D, T);
    if (path == PMOE_PATH_TC || path == PMOE_PATH_TC2) {
        if (!encode_rows_map(&xmap, x, cap_tc, D.d, kTcBlockM) ||
            !encode_rows_map(&hmap, h, cap_tc, D.f, kTcBlockM))
            return fail(PMOE_ERR_CUDA, "tensor map encoding failed");
    } else if (path == PMOE_PATH_TC_DECODE) {
        if (!encode_rows_map(&xmap, x, cap_tc, D.d, sw.bn) || !encode_rows_map(&hmap, h, cap_tc, D.f, sw.bn))
            return fail(PMOE_ERR_CUDA, "tensor map encoding failed");
    }

    if (path == PMOE_PATH_SLICE) {
        // routing, gate/up + SiLU-and-mul, down and the combine in one persistent launch, each CTA
        // on whole columns of the intermediate dimension
        CUtensorMap sx;
        if (!encode_rows_map(&sx, hidden, T, D.d, 16)) return fail(PMOE_ERR_CUDA, "tensor map encoding failed");
        FusedArgs fa{};
        fa.logits = logits;
        fa.page_table = page_table;
        fa.buf_slot = buf_slot;
        fa.p2 = at<float>(ws, W.sp);
        fa.out = static_cast<uint16_t*>(out);
        fa.arrive = P->d_arrive;
        fa.err = P->d_error;
        fa.ids_out = ids;
        fa.w_out = w;
        fa.active_out = sorted;
        fa.meta_out = meta;
        fa.num_pages = P->num_pages;
        fa.g0 = slice_g0;
        fa.T = T;
        fa.E = D.num_experts;
        fa.k = D.top_k;
        fa.S = D.num_shared_chunks;
        fa.renorm = D.renormalize;
        fa.d = D.d;
        fa.f = D.f;
        fa.slots_per_buffer = D.slots_per_buffer;
        fa.have_buf0 = P->buf[0] != nullptr;
        fa.have_buf1 = P->buf[1] != nullptr;
        fa.contig = contig ? 1 : 0;
        fa.epl = 1;
        while (32 * fa.epl < D.num_experts) fa.epl <<= 1;
        PMOE_CUDA(mark(P, 0, stream), "profile event");
        PMOE_CUDA(launch_slice_decode(sx, P->tm_rows_d64, P->tm_rows_f, fa, dgrid, stream), "slice decode");
        PMOE_CUDA(mark(P, 1, stream), "profile event");
        P->last_path = path;
        P->last_kernels = 1;
        P->last_launches = 1;
        P->last_T = T;
        P->last_block_m = 0;
        return PMOE_OK;
    }

    if (path == PMOE_PATH_FUSED) {
        // routing, gate/up + SiLU-and-mul, down and the combine in one persistent launch
        const FusedShape F = fused_shape(D, T);
        const int grid = dgrid;
        CUtensorMap fx, fh;
        if (!encode_rows_map(&fx, hidden, T, D.d, F.bn) ||
            !encode_rows_map(&fh, at<uint16_t>(ws, W.fh), F.a_max * F.bn, D.f, F.bn))
            return fail(PMOE_ERR_CUDA, "tensor map encoding failed");
        FusedArgs fa{};
        fa.logits = logits;
        fa.page_table = page_table;
        fa.buf_slot = buf_slot;
        fa.p1 = at<float>(ws, W.fp1);
        fa.h = at<uint16_t>(ws, W.fh);
        fa.p2 = at<float>(ws, W.fp2);
        fa.out = static_cast<uint16_t*>(out);
        fa.flags = P->d_flags;
        fa.ucnt = P->d_ucnt;
        fa.hflag = P->d_hflag;
        fa.err = P->d_error;
        fa.ids_out = ids;
        fa.w_out = w;
        fa.active_out = sorted;
        fa.meta_out = meta;
        fa.num_pages = P->num_pages;
        fa.p1_base1 = F.u1_shared + grid;
        // the shared chunks' gate/up (streamed before routing is known) goes to the first g0
        // CTAs, with pieces of at least 8 k-blocks each
        {
            const int64_t i0 = (int64_t)D.num_shared_chunks * (D.f / 64) * (D.d / 64);
            const int64_t g0 = i0 / 8;
            fa.g0 = (int)(g0 < 1 ? 1 : (g0 > grid ? grid : g0));
        }
        fa.T = T;
        fa.E = D.num_experts;
        fa.k = D.top_k;
        fa.S = D.num_shared_chunks;
        fa.renorm = D.renormalize;
        fa.d = D.d;
        fa.f = D.f;
        fa.slots_per_buffer = D.slots_per_buffer;
        fa.have_buf0 = P->buf[0] != nullptr;
        fa.have_buf1 = P->buf[1] != nullptr;
        fa.contig = contig ? 1 : 0;
        fa.epl = 1;
        while (32 * fa.epl < D.num_experts) fa.epl <<= 1;
        PMOE_CUDA(mark(P, 0, stream), "profile event");
        PMOE_CUDA(launch_fused_decode(fx, fh, P->tm_rows_d64, P->tm_rows_f, fa, F.bn, grid, stream),
                  "fused decode");
        PMOE_CUDA(mark(P, 1, stream), "profile event");
        P->last_path = path;
        P->last_kernels = 1;
        P->last_launches = 1;
        P->last_T = T;
        P->last_block_m = 0;
        return PMOE_OK;
    }

    ResolveArgs rs{};
    rs.page_table = page_table;
    rs.buf_slot = buf_slot;
    rs.num_pages = P->num_pages;
    rs.slots_per_buffer = D.slots_per_buffer;
    rs.have_buf0 = P->buf[0] != nullptr;
    rs.have_buf1 = P->buf[1] != nullptr;
    rs.contiguous = contig ? 1 : 0;
    rs.loc = loc;
    rs.err = P->d_error;

    const int bm = (path == PMOE_PATH_TC || path == PMOE_PATH_TC2) ? kTcBlockM
                 : path == PMOE_PATH_TC_DECODE ? sw.bn : stream_block_m(D, T);
    int4* units = at<int4>(ws, W.units);
    int32_t* unit_w2 = at<int32_t>(ws, W.unit_w2);
    if (path == PMOE_PATH_TC2) {
        rs.units = units;
        rs.unit_w2 = unit_w2;
        rs.unit_group = at<int2>(ws, W.ugroup);
    }
    int32_t* brows = at<int32_t>(ws, W.brows);
    if (path == PMOE_PATH_TC || path == PMOE_PATH_TC_DECODE) rs.block_rows = brows;
    const uint16_t* hid = static_cast<const uint16_t*>(hidden);
    int ev = 0;
    // the single-CTA prep also copies the rows when they are few (at most 64 KB)
    const bool prep = use_prep_small(T, D.num_experts, D.top_k);
    const bool gather_in_prep = prep && tc_family && W.np * D.d * 2 <= 64 * 1024;
    if (prep) {
        // one CTA: routing, sort + pad + page resolution
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_prep_small(logits, T, D.num_experts, D.top_k, D.renormalize, ids, w,
                                    D.num_shared_chunks, bm, sorted, bexp, inv, meta, rs, hid, D.d,
                                    gather_in_prep ? x : nullptr, stream), "prep");
    } else {
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_route(logits, T, D.num_experts, D.top_k, D.renormalize, ids, w, stream), "route");
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_align_multi(ids, T, D.top_k, D.num_experts, D.num_shared_chunks, bm,
                                     at<int32_t>(ws, W.part), sorted, bexp, inv, meta, &rs, stream),
                  "align");
    }
    // With a separate row gather, the gate/up GEMMs read the shared chunks' rows (every token, in
    // order) from hidden itself and the gather copies routed pairs only.
    SharedRows sh{};
    CUtensorMap hidmap;
    if (tc_family && !gather_in_prep) {
        sh.direct = 1;
        sh.E = D.num_experts;
        sh.S = D.num_shared_chunks;
        sh.rows = (int)((T + bm - 1) / bm * bm);
        if (!encode_rows_map(&hidmap, hidden, T, D.d, path == PMOE_PATH_TC_DECODE ? sw.bn : kTcBlockM))
            return fail(PMOE_ERR_CUDA, "tensor map encoding failed");
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_gather_pairs(hid, inv, T, D.top_k, 0, D.d, x, stream), "gather");
    }
    const CUtensorMap* hidp = sh.direct ? &hidmap : nullptr;
    const int64_t nblk = (W.np + bm - 1) / bm + (ES < W.np ? ES : W.np);
    int64_t ystride;
    int splits;
    if (path == PMOE_PATH_TC) {
        // blocks mostly padding (few tokens per expert) load only their rows, 16 at a time
        CUtensorMap x16, h16, hid16;
        if (!encode_rows_map(&x16, x, cap_tc, D.d, 16) || !encode_rows_map(&h16, h, cap_tc, D.f, 16) ||
            (sh.direct && !encode_rows_map(&hid16, hidden, T, D.d, 16)))
            return fail(PMOE_ERR_CUDA, "tensor map encoding failed");
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_tc_gemm(1, contig, xmap, P->tm_rows_d, bexp, meta, loc, h, cap_tc, D.f, D.d,
                                 nblk, P->num_sms, P->d_error, stream, hidp, sh, brows, &x16,
                                 sh.direct ? &hid16 : nullptr),
                  "gate/up gemm");
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_tc_gemm(2, contig, hmap, P->tm_rows_f, bexp, meta, loc, y, cap_tc, D.f, D.d,
                                 nblk, P->num_sms, P->d_error, stream, nullptr, SharedRows{}, brows,
                                 &h16, nullptr), "down gemm");
        ystride = cap_tc;
        splits = 1;
    } else if (path == PMOE_PATH_TC2) {
        // 256-row pairs of blocks and each expert's odd last block, all on CTA pairs in one
        // launch per GEMM; the shared chunks' units are the last ones of the list
        const int shared_units = (int)(D.num_shared_chunks * (((T + kTcBlockM - 1) / kTcBlockM + 1) / 2));
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        CUtensorMap x64, h64, hid64;
        if (!encode_rows_map(&x64, x, cap_tc, D.d, 64) || !encode_rows_map(&h64, h, cap_tc, D.f, 64) ||
            (sh.direct && !encode_rows_map(&hid64, hidden, T, D.d, 64)))
            return fail(PMOE_ERR_CUDA, "tensor map encoding failed");
        const int2* ugroup = at<int2>(ws, W.ugroup);
        PMOE_CUDA(launch_tc_gemm2sm(1, contig, xmap, x64, P->tm_rows_d, P->tm_rows_d64, units, unit_w2,
                                    ugroup, meta, h, cap_tc, D.f, D.d, nblk, P->num_sms, P->d_error,
                                    stream, hidp, sh.direct ? &hid64 : nullptr, sh, shared_units),
                  "gate/up gemm");
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_tc_gemm2sm(2, contig, hmap, h64, P->tm_rows_f, P->tm_rows_f, units, unit_w2,
                                    ugroup, meta, y, cap_tc, D.f, D.d, nblk, P->num_sms, P->d_error, stream,
                                    nullptr, nullptr, SharedRows{}, shared_units), "down gemm");
        ystride = cap_tc;
        splits = 1;
    } else if (path == PMOE_PATH_TC_DECODE) {
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        // few-token blocks: half-size (stacked) tiles once the full-size ones outnumber the SMs,
        // so the persistent CTAs finish together; below that, full tiles (less epilogue work)
        const int64_t act_est = (ES < W.np ? ES : W.np);
        const bool stacked = sw.bn <= 32 && act_est * (D.f / 128) > P->num_sms;
        PMOE_CUDA(launch_tc_swap(stacked ? 3 : 1, contig, sw.bn, xmap,
                                 stacked ? P->tm_rows_d64 : P->tm_rows_d, sorted, T, D.top_k,
                                 D.num_shared_chunks, bexp, meta, loc, h, D.f, D.d, 1, 0, nblk,
                                 P->num_sms, P->d_error, gather_in_prep ? 0 : 1, stream, hidp, sh, brows),
                  "gate/up gemm");
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_tc_swap(2, contig, sw.bn, hmap, P->tm_rows_f, sorted, T, D.top_k,
                                 D.num_shared_chunks, bexp, meta, loc, y, D.f, D.d, sw.splits,
                                 sw.ystride, nblk, P->num_sms, P->d_error, 1, stream, nullptr,
                                 SharedRows{}, brows), "down gemm");
        ystride = sw.ystride;
        splits = sw.splits;
    } else {
        LayerPtrs L{};
        L.map_base[0] = static_cast<const uint16_t*>(P->pool);
        L.map_base[1] = static_cast<const uint16_t*>(P->buf[0]);
        L.map_base[2] = static_cast<const uint16_t*>(P->buf[1]);
        L.d = D.d; L.f = D.f; L.E = D.num_experts; L.k = D.top_k; L.S = D.num_shared_chunks; L.T = T;
        ystride = W.np + ES * (bm - 1);
        splits = W.splits;
        const ExpertLoc* lp = contig ? nullptr : loc;
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_stream_gemm1(L, hid, sorted, bexp, meta, lp, bm, nblk, h, stream), "gemm1");
        PMOE_CUDA(mark(P, ev++, stream), "profile event");
        PMOE_CUDA(launch_stream_gemm2(L, sorted, bexp, meta, lp, bm, nblk, splits, ystride, h, y,
                                      stream), "gemm2");
    }
    PMOE_CUDA(mark(P, ev++, stream), "profile event");
    const bool y_bf16 = path == PMOE_PATH_TC || path == PMOE_PATH_TC2;   // bf16 y rows, no K split
    PMOE_CUDA(launch_combine(y, y_bf16, splits, ystride, w, inv, T, D.d, D.top_k, D.num_shared_chunks,
                             static_cast<uint16_t*>(out), stream), "combine");
    PMOE_CUDA(mark(P, ev++, stream), "profile event");
    P->last_path = path;
    P->last_T = T;
    P->last_block_m = bm;
    P->last_kernels = ev - 1;
    P->last_launches = ev - 1 + (!prep && align_ctas(W.np - (int64_t)T * D.num_shared_chunks, D.num_experts + D.num_shared_chunks) > 1 ? 1 : 0);
    return PMOE_OK;
}

}  // namespace pmoe

using namespace pmoe;

extern "C" {

const char* pmoe_status_string(pmoe_status s) {
    switch (s) {
        case PMOE_OK: return "ok";
        case PMOE_ERR_INVALID_ARG: return "invalid argument";
        case PMOE_ERR_PAGE_OOB: return "page index out of range";
        case PMOE_ERR_SLOT_OOB: return "load-buffer slot out of range";
        case PMOE_ERR_UNSUPPORTED: return "unsupported shape or path";
        case PMOE_ERR_CUDA: return "CUDA error";
        case PMOE_ERR_TIMEOUT: return "timeout";
        case PMOE_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

const char* pmoe_last_error(void) { return g_last_error.c_str(); }

pmoe_status pmoe_plan_create(const pmoe_layer_desc* desc, const void* page_pool, int64_t num_pages,
                             const void* load_buf0, const void* load_buf1, pmoe_plan_t* out) {
    if (!out) return fail(PMOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!desc_ok(desc)) return fail(PMOE_ERR_INVALID_ARG, "bad layer descriptor");
    if (!shape_supported(desc)) return fail(PMOE_ERR_UNSUPPORTED, "d must be a multiple of 64 and f of 128");
    if (!page_pool || num_pages <= 0) return fail(PMOE_ERR_INVALID_ARG, "empty page pool");
    if (((uintptr_t)page_pool & 15) || ((uintptr_t)load_buf0 & 15) || ((uintptr_t)load_buf1 & 15))
        return fail(PMOE_ERR_INVALID_ARG, "pool and buffers must be 16-byte aligned");
    Plan* P = new (std::nothrow) Plan();
    if (!P) return fail(PMOE_ERR_INVALID_ARG, "out of host memory");
    P->desc = *desc;
    P->pool = page_pool;
    P->num_pages = num_pages;
    P->buf[0] = load_buf0;
    P->buf[1] = load_buf1;
    P->path = PMOE_PATH_AUTO;
    cudaError_t e = cudaGetDevice(&P->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, P->device);
    if (e == cudaSuccess) {
        // the column-slice kernel's fit depends only on the layer, T and the grid
        const int dgrid = P->num_sms < kFusedMaxGrid ? P->num_sms : kFusedMaxGrid;
        for (int t = 1; t <= kSliceMaxTokens; ++t)
            P->slice_fits[t] = slice_fit(*desc, t, dgrid, &P->slice_g0[t], &P->slice_tiles[t]) ? 1 : 0;
    }
    // one allocation of device words: the error word, the fused kernel's barrier words and tiles
    P->words_bytes = plan_words_bytes(*desc);
    if (e == cudaSuccess) e = cudaMalloc(&P->d_error, P->words_bytes);
    if (e == cudaSuccess) e = cudaMemset(P->d_error, 0, P->words_bytes);
    if (e == cudaSuccess) {
        char* base = reinterpret_cast<char*>(P->d_error);
        const size_t tiles = (size_t)(desc->num_experts + desc->num_shared_chunks) * (desc->f / 64);
        P->d_arrive = reinterpret_cast<unsigned long long*>(base + 512);
        P->d_flags = reinterpret_cast<uint32_t*>(base + 1024);
        P->d_ucnt = reinterpret_cast<unsigned long long*>(base + 2048);
        P->d_hflag = reinterpret_cast<uint32_t*>(base + 2048 + 8 * tiles);
    }
    if (e != cudaSuccess) {
        if (P->d_error) cudaFree(P->d_error);
        delete P;
        return cuda_fail(e, "plan_create");
    }
    // TMA views of the pool and the buffers: rows [pages*f, d] for gate/up pages, rows
    // [pages*d, f] for down pages; a buffer slot s holds its matrices as pages 3s, 3s+1, 3s+2.
    const int64_t f = desc->f, d = desc->d;
    const int64_t bpages = 3 * (int64_t)desc->slots_per_buffer;
    bool ok = encode_rows_map(&P->tm_rows_d[0], page_pool, num_pages * f, d) &&
              encode_rows_map(&P->tm_rows_d64[0], page_pool, num_pages * f, d, 64) &&
              encode_rows_map(&P->tm_rows_f[0], page_pool, num_pages * d, f);
    for (int b = 0; b < 2 && ok; ++b) {
        if (P->buf[b] && bpages > 0) {
            ok = encode_rows_map(&P->tm_rows_d[1 + b], P->buf[b], bpages * f, d) &&
                 encode_rows_map(&P->tm_rows_d64[1 + b], P->buf[b], bpages * f, d, 64) &&
                 encode_rows_map(&P->tm_rows_f[1 + b], P->buf[b], bpages * d, f);
        } else {
            P->tm_rows_d[1 + b] = P->tm_rows_d[0];   // never addressed: no slot maps here
            P->tm_rows_d64[1 + b] = P->tm_rows_d64[0];
            P->tm_rows_f[1 + b] = P->tm_rows_f[0];
        }
    }
    P->have_tmaps = ok;
    *out = reinterpret_cast<pmoe_plan_t>(P);
    return PMOE_OK;
}

pmoe_status pmoe_plan_destroy(pmoe_plan_t plan) {
    if (!plan) return PMOE_OK;
    Plan* P = reinterpret_cast<Plan*>(plan);
    cudaError_t e = P->d_error ? cudaFree(P->d_error) : cudaSuccess;
    delete P;
    return e == cudaSuccess ? PMOE_OK : cuda_fail(e, "plan_destroy");
}

pmoe_status pmoe_plan_set_path(pmoe_plan_t plan, int32_t path) {
    if (!plan || path < PMOE_PATH_AUTO || path > PMOE_PATH_SLICE)
        return fail(PMOE_ERR_INVALID_ARG, "bad plan or path");
    reinterpret_cast<Plan*>(plan)->path = path;
    return PMOE_OK;
}

pmoe_status pmoe_plan_last_run(pmoe_plan_t plan, int32_t* path, int32_t* n_steps,
                               int32_t* n_launches) {
    Plan* P = reinterpret_cast<Plan*>(plan);
    if (!P || !path || !n_steps || !n_launches) return fail(PMOE_ERR_INVALID_ARG, "NULL argument");
    *path = P->last_path;
    *n_steps = P->last_kernels;
    *n_launches = P->last_launches;
    return PMOE_OK;
}

pmoe_status pmoe_plan_set_profile_events(pmoe_plan_t plan, const pmoe_event_t* events, int32_t n) {
    Plan* P = reinterpret_cast<Plan*>(plan);
    if (!P || n < 0 || n > 16 || (n > 0 && !events)) return fail(PMOE_ERR_INVALID_ARG, "bad profile events");
    for (int i = 0; i < n; ++i) P->prof_ev[i] = (cudaEvent_t)events[i];
    P->n_prof = n;
    return PMOE_OK;
}

pmoe_status pmoe_plan_routing_view(pmoe_plan_t plan, int32_t T, pmoe_routing_view* out) {
    Plan* P = reinterpret_cast<Plan*>(plan);
    if (!P || !out) return fail(PMOE_ERR_INVALID_ARG, "NULL plan or view");
    if (P->last_T <= 0 || T != P->last_T)
        return fail(PMOE_ERR_INVALID_ARG, "T differs from the token count of the plan's last forward call");
    const WsLayout W = layout(P->desc, T);
    pmoe_routing_view v;
    v.path = P->last_path;
    v.tokens = T;
    v.block_m = P->last_block_m;
    v.top_k = P->desc.top_k;
    v.ids = (int64_t)W.ids;
    v.weights = (int64_t)W.w;
    v.meta = (int64_t)W.meta;
    v.sorted_ids = v.block_expert = v.inv = v.block_rows = v.units = v.active = -1;
    if (v.path == PMOE_PATH_FUSED || v.path == PMOE_PATH_SLICE) {
        v.active = (int64_t)W.sorted;
    } else {
        v.sorted_ids = (int64_t)W.sorted;
        v.block_expert = (int64_t)W.bexp;
        v.inv = (int64_t)W.inv;
        if (v.path == PMOE_PATH_TC || v.path == PMOE_PATH_TC_DECODE) v.block_rows = (int64_t)W.brows;
        if (v.path == PMOE_PATH_TC2) v.units = (int64_t)W.units;
    }
    *out = v;
    return PMOE_OK;
}

size_t pmoe_workspace_size(const pmoe_layer_desc* desc, int32_t max_tokens) {
    if (!desc_ok(desc) || max_tokens < 0) return 0;
    // every region grows with T inside the ranges the decode kernels serve, but those kernels'
    // scratch exists only up to their own token limits, so a call of up to 16 or 32 tokens can
    // need more than a larger one: take the largest of the three
    size_t m = layout(*desc, max_tokens).total;
    const int32_t lim[2] = {kSliceMaxTokens, kFusedMaxTokens};
    for (int i = 0; i < 2; ++i) {
        const size_t b = layout(*desc, max_tokens < lim[i] ? max_tokens : lim[i]).total;
        if (b > m) m = b;
    }
    return m;
}

pmoe_status moe_paged_forward(pmoe_plan_t plan, const void* hidden, int32_t T,
                              const float* router_logits, int32_t top_k, const int32_t* page_table,
                              const int32_t* buf_slot, void* out, void* workspace,
                              size_t workspace_bytes, pmoe_stream_t stream) {
    return forward_impl(reinterpret_cast<Plan*>(plan), hidden, T, router_logits, top_k, page_table,
                        buf_slot, out, workspace, workspace_bytes, (cudaStream_t)stream, false);
}

pmoe_status moe_contig_forward(pmoe_plan_t plan, const void* hidden, int32_t T,
                               const float* router_logits, int32_t top_k, void* out,
                               void* workspace, size_t workspace_bytes, pmoe_stream_t stream) {
    Plan* P = reinterpret_cast<Plan*>(plan);
    if (P && P->num_pages < 3 * (int64_t)(P->desc.num_experts + P->desc.num_shared_chunks))
        return fail(PMOE_ERR_INVALID_ARG, "contiguous plan needs 3*(E+S) pages");
    return forward_impl(P, hidden, T, router_logits, top_k, nullptr, nullptr, out, workspace,
                        workspace_bytes, (cudaStream_t)stream, true);
}

pmoe_status pmoe_prefetch_async(pmoe_plan_t plan, int32_t buf, int32_t n,
                                const void* const* host_experts, const int32_t* slots,
                                pmoe_stream_t copy_stream, pmoe_event_t buf_free,
                                pmoe_event_t copy_done) {
    Plan* P = reinterpret_cast<Plan*>(plan);
    if (!P) return fail(PMOE_ERR_INVALID_ARG, "plan is NULL");
    if (buf != 0 && buf != 1) return fail(PMOE_ERR_INVALID_ARG, "buf must be 0 or 1");
    if (!P->buf[buf]) return fail(PMOE_ERR_INVALID_ARG, "plan has no such load buffer");
    const int S = P->desc.slots_per_buffer;
    if (n < 0 || n > S) return fail(PMOE_ERR_INVALID_ARG, "n exceeds expert_offload_limit");
    if (n > 0 && (!host_experts || !slots)) return fail(PMOE_ERR_INVALID_ARG, "NULL host arrays");
    for (int i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= S) return fail(PMOE_ERR_SLOT_OOB, "slot out of range");
        if (!host_experts[i]) return fail(PMOE_ERR_INVALID_ARG, "NULL host expert");
        for (int j = 0; j < i; ++j)
            if (slots[j] == slots[i]) return fail(PMOE_ERR_INVALID_ARG, "duplicate slot");
    }
    cudaStream_t cs = (cudaStream_t)copy_stream;
    if (buf_free) PMOE_CUDA(cudaStreamWaitEvent(cs, (cudaEvent_t)buf_free, 0), "wait buf_free");
    const size_t bytes = (size_t)3 * P->desc.f * P->desc.d * 2;
    char* base = static_cast<char*>(const_cast<void*>(P->buf[buf]));
    for (int i = 0; i < n; ++i)
        PMOE_CUDA(cudaMemcpyAsync(base + (size_t)slots[i] * bytes, host_experts[i], bytes,
                                  cudaMemcpyHostToDevice, cs), "prefetch copy");
    if (copy_done) PMOE_CUDA(cudaEventRecord((cudaEvent_t)copy_done, cs), "record copy_done");
    return PMOE_OK;
}

pmoe_status pmoe_fill_pages_async(pmoe_plan_t plan, int32_t n, const void* const* host_experts,
                                  const int32_t* pages, pmoe_stream_t copy_stream,
                                  pmoe_event_t after, pmoe_event_t copy_done) {
    Plan* P = reinterpret_cast<Plan*>(plan);
    if (!P) return fail(PMOE_ERR_INVALID_ARG, "plan is NULL");
    if (n < 0) return fail(PMOE_ERR_INVALID_ARG, "n < 0");
    if (n > 0 && (!host_experts || !pages)) return fail(PMOE_ERR_INVALID_ARG, "NULL host arrays");
    for (int i = 0; i < n; ++i)
        if (!host_experts[i]) return fail(PMOE_ERR_INVALID_ARG, "NULL host expert");
    for (int i = 0; i < 3 * n; ++i) {
        if (pages[i] < 0 || pages[i] >= P->num_pages)
            return fail(PMOE_ERR_PAGE_OOB, "page out of range");
        for (int j = 0; j < i; ++j)
            if (pages[j] == pages[i]) return fail(PMOE_ERR_INVALID_ARG, "duplicate page");
    }
    cudaStream_t cs = (cudaStream_t)copy_stream;
    if (after) PMOE_CUDA(cudaStreamWaitEvent(cs, (cudaEvent_t)after, 0), "wait after");
    const size_t page_bytes = (size_t)P->desc.f * P->desc.d * 2;
    char* pool = static_cast<char*>(const_cast<void*>(P->pool));
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < 3; ++j)
            PMOE_CUDA(cudaMemcpyAsync(pool + (size_t)pages[3 * i + j] * page_bytes,
                                      static_cast<const char*>(host_experts[i]) + j * page_bytes,
                                      page_bytes, cudaMemcpyHostToDevice, cs),
                      "fill page copy");
    if (copy_done) PMOE_CUDA(cudaEventRecord((cudaEvent_t)copy_done, cs), "record copy_done");
    return PMOE_OK;
}

pmoe_status pmoe_copy_in_missing(pmoe_plan_t plan, const float* router_logits, int32_t T,
                                 int32_t* buf_slot, int32_t buf, const void* const* host_experts,
                                 int32_t* missed, pmoe_stream_t stream) {
    Plan* P = reinterpret_cast<Plan*>(plan);
    if (!P) return fail(PMOE_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0) return fail(PMOE_ERR_INVALID_ARG, "T < 0");
    if (!buf_slot || !host_experts || !missed || (T > 0 && !router_logits))
        return fail(PMOE_ERR_INVALID_ARG, "NULL pointer");
    if (buf != 0 && buf != 1) return fail(PMOE_ERR_INVALID_ARG, "buf must be 0 or 1");
    if (!P->buf[buf] || P->desc.slots_per_buffer <= 0)
        return fail(PMOE_ERR_INVALID_ARG, "plan has no such load buffer");
    if (P->desc.slots_per_buffer > 65536) return fail(PMOE_ERR_UNSUPPORTED, "more than 65536 slots per buffer");
    if ((int64_t)T * P->desc.top_k > (int64_t)1 << 30) return fail(PMOE_ERR_INVALID_ARG, "too many tokens");
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        PMOE_CUDA(cudaMemsetAsync(missed, 0, sizeof(int32_t), s), "copy-in count");
        return PMOE_OK;
    }
    PMOE_CUDA(launch_copy_in(*P, router_logits, T, buf_slot, buf, host_experts, missed, s), "copy-in");
    return PMOE_OK;
}

pmoe_status pmoe_device_pointers(int32_t n, const void* const* host, void** device) {
    if (n < 0 || (n > 0 && (!host || !device))) return fail(PMOE_ERR_INVALID_ARG, "bad arguments");
    for (int i = 0; i < n; ++i) {
        if (!host[i]) {
            device[i] = nullptr;
            continue;
        }
        void* d = nullptr;
        const cudaError_t e = cudaHostGetDevicePointer(&d, const_cast<void*>(host[i]), 0);
        if (e != cudaSuccess) {
            cudaGetLastError();   // not a sticky error: clear it
            return fail(PMOE_ERR_INVALID_ARG, "a pointer has no device address (not pinned host memory)");
        }
        if ((uintptr_t)d & 15) return fail(PMOE_ERR_INVALID_ARG, "a pointer is not 16-byte aligned");
        device[i] = d;
    }
    return PMOE_OK;
}

pmoe_status pmoe_wait_event(pmoe_event_t ev, int32_t timeout_ms) {
    if (!ev) return fail(PMOE_ERR_INVALID_ARG, "event is NULL");
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaEventQuery((cudaEvent_t)ev);
        if (e == cudaSuccess) return PMOE_OK;
        if (e != cudaErrorNotReady) return cuda_fail(e, "event query");
        const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                            std::chrono::steady_clock::now() - t0).count();
        if (ms >= timeout_ms) return fail(PMOE_ERR_TIMEOUT, "event not complete before timeout");
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

pmoe_status pmoe_get_device_error(pmoe_plan_t plan, int32_t clear, int32_t* code,
                                  pmoe_stream_t stream) {
    Plan* P = reinterpret_cast<Plan*>(plan);
    if (!P || !code) return fail(PMOE_ERR_INVALID_ARG, "NULL plan or code");
    cudaStream_t s = (cudaStream_t)stream;
    int32_t v = 0;
    PMOE_CUDA(cudaMemcpyAsync(&v, P->d_error, sizeof v, cudaMemcpyDeviceToHost, s), "read error word");
    PMOE_CUDA(cudaStreamSynchronize(s), "sync");
    if (clear) {
        // also resets the decode kernels' barrier words, arrival counter and tile words, which a
        // kernel that timed out may leave behind
        PMOE_CUDA(cudaMemsetAsync(P->d_error, 0, P->words_bytes, s), "clear error word");
        PMOE_CUDA(cudaStreamSynchronize(s), "sync");
    }
    *code = v;
    return PMOE_OK;
}

pmoe_status pmoe_route(const float* router_logits, int32_t T, int32_t E, int32_t top_k,
                       int32_t renormalize, int32_t* ids, float* weights, pmoe_stream_t stream) {
    if (T < 0 || E <= 0 || E > kMaxExpertsTotal || top_k <= 0 || top_k > E || top_k > kMaxTopK)
        return fail(PMOE_ERR_INVALID_ARG, "bad routing sizes");
    if (T > 0 && (!router_logits || !ids || !weights)) return fail(PMOE_ERR_INVALID_ARG, "NULL pointer");
    PMOE_CUDA(launch_route(router_logits, T, E, top_k, renormalize, ids, weights, (cudaStream_t)stream), "route");
    return PMOE_OK;
}

size_t pmoe_align_scratch_size(void) { return align_part_bytes(); }

pmoe_status pmoe_align(const int32_t* ids, int32_t T, int32_t top_k, int32_t E, int32_t S,
                       int32_t block_m, int32_t* sorted_ids, int32_t* block_expert, int32_t* inv,
                       int32_t* n_padded, void* scratch, pmoe_stream_t stream) {
    if (T < 0 || top_k <= 0 || E <= 0 || S < 0 || E + S > kMaxExpertsTotal)
        return fail(PMOE_ERR_INVALID_ARG, "bad align sizes");
    if (block_m < 1 || block_m > 256 || (block_m & (block_m - 1)))
        return fail(PMOE_ERR_INVALID_ARG, "block_m must be a power of two <= 256");
    if (!sorted_ids || !block_expert || !n_padded || (T > 0 && (!ids || !inv)))
        return fail(PMOE_ERR_INVALID_ARG, "NULL pointer");
    if ((int64_t)T * (top_k + S) > (int64_t)1 << 30) return fail(PMOE_ERR_INVALID_ARG, "too many pairs");
    if (scratch)
        PMOE_CUDA(launch_align_multi(ids, T, top_k, E, S, block_m, static_cast<int32_t*>(scratch),
                                     sorted_ids, block_expert, inv, n_padded, nullptr,
                                     (cudaStream_t)stream), "align");
    else
        PMOE_CUDA(launch_align(ids, T, top_k, E, S, block_m, sorted_ids, block_expert, inv, n_padded,
                               nullptr, (cudaStream_t)stream), "align");
    return PMOE_OK;
}

}  // extern "C"

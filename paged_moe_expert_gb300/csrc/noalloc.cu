// A forward entry point that allocates nothing: the decode-size (weight-streaming) layer
// forward with its scratch in a fixed, file-scope device array.
//
// Some callers cannot allocate device memory at the time they run the layer: inference-server
// plugins and embedded runtimes that are handed a fixed device-memory budget at start-up and may
// not call cudaMalloc afterwards, or latency-critical loops where cudaMalloc would block until
// in-flight device work finishes.  They cannot create a plan either (a plan owns a small device
// allocation), so this entry point takes the pool, the buffers and the tables directly, like
// moe_paged_forward, and keeps every intermediate (routing ids and weights, the sorted pair
// list, the block map, the page locations, h and the down-projection partials) in the array
// below.  It runs the same kernels as moe_paged_forward's weight-streaming path.
#include <mutex>

#include "pmoe_internal.cuh"

namespace pmoe {

namespace {

// 16 MiB of scratch; every GPU that loads this library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
static void* g_scratch_addr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  The array's name in host code is
// only a host-side stand-in, so the address is looked up once per device with that device
// current, and cached.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

struct NoAllocLayout {
    size_t ids, w, sorted, bexp, inv, meta, loc, h, y, total;
    int64_t np, cap, nblk;
    int bm, splits;
};

// Compact layout of the weight-streaming path for exactly T tokens.
NoAllocLayout noalloc_layout(const pmoe_layer_desc& D, int64_t T) {
    NoAllocLayout L{};
    const int64_t ES = D.num_experts + D.num_shared_chunks;
    L.np = T * (D.top_k + D.num_shared_chunks);
    int bm = 1;
    while (bm < T && bm < kStreamMaxBlockM) bm <<= 1;
    while (bm > 1 && (size_t)bm * D.d * 2 > 128 * 1024) bm >>= 1;
    L.bm = bm;
    const int64_t active = ES < L.np ? ES : L.np;  // experts that can own a block
    L.cap = L.np + active * (bm - 1);
    L.nblk = (L.np + bm - 1) / bm + active;
    L.splits = (D.f + kStreamKChunk - 1) / kStreamKChunk;
    size_t o = 0;
    L.ids = o;    o = up256(o + sizeof(int32_t) * T * D.top_k);
    L.w = o;      o = up256(o + sizeof(float) * T * D.top_k);
    L.sorted = o; o = up256(o + sizeof(int32_t) * L.cap);
    L.bexp = o;   o = up256(o + sizeof(int32_t) * (L.nblk + 1));
    L.inv = o;    o = up256(o + sizeof(int32_t) * (L.np > 0 ? L.np : 1));
    L.meta = o;   o = up256(o + sizeof(int32_t) * kMetaCount);
    L.loc = o;    o = up256(o + sizeof(ExpertLoc) * ES * 3);
    L.h = o;      o = up256(o + 2 * (size_t)L.cap * D.f);
    L.y = o;      o = up256(o + sizeof(float) * (size_t)L.splits * L.cap * D.d);
    L.total = o;
    return L;
}

}  // namespace

}  // namespace pmoe

using namespace pmoe;

extern "C" pmoe_status moe_paged_forward_noalloc(
    const pmoe_layer_desc* desc, const void* page_pool, int64_t num_pages, const void* load_buf0,
    const void* load_buf1, const void* hidden, int32_t T, const float* router_logits,
    int32_t top_k, const int32_t* page_table, const int32_t* buf_slot, void* out,
    int32_t* device_error, pmoe_stream_t stream) {
    if (!desc_ok(desc)) return record_failure(PMOE_ERR_INVALID_ARG, "bad layer descriptor");
    if (!shape_supported(desc))
        return record_failure(PMOE_ERR_UNSUPPORTED, "d must be a multiple of 64 (<= 16384) and f of 128 (<= 65536)");
    if (T < 0 || top_k != desc->top_k) return record_failure(PMOE_ERR_INVALID_ARG, "bad T or top_k");
    if (T == 0) return PMOE_OK;
    if (!page_pool || num_pages <= 0 || !hidden || !router_logits || !page_table || !buf_slot || !out)
        return record_failure(PMOE_ERR_INVALID_ARG, "NULL pointer");
    if (!device_error)
        return record_failure(PMOE_ERR_INVALID_ARG, "device_error is NULL: table errors would go unreported");
    if (((uintptr_t)hidden & 15) || ((uintptr_t)out & 15) || ((uintptr_t)page_pool & 15) ||
        ((uintptr_t)load_buf0 & 15) || ((uintptr_t)load_buf1 & 15))
        return record_failure(PMOE_ERR_INVALID_ARG,
                              "hidden, out, the pool and the load buffers must be 16-byte aligned");
    if ((int64_t)T * (desc->top_k + desc->num_shared_chunks) > (int64_t)1 << 24)
        return record_failure(PMOE_ERR_WORKSPACE, "too many tokens for the fixed scratch");
    const NoAllocLayout W = noalloc_layout(*desc, T);
    if (W.total > kNoAllocScratchBytes)
        return record_failure(PMOE_ERR_WORKSPACE, "layer and token count exceed the fixed scratch");

    void* base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess) return record_failure(PMOE_ERR_CUDA, "scratch address lookup failed");
    char* ws = static_cast<char*>(base);
    cudaStream_t s = (cudaStream_t)stream;
    int32_t* err = device_error;
    int32_t* ids = reinterpret_cast<int32_t*>(ws + W.ids);
    float* w = reinterpret_cast<float*>(ws + W.w);
    int32_t* sorted = reinterpret_cast<int32_t*>(ws + W.sorted);
    int32_t* bexp = reinterpret_cast<int32_t*>(ws + W.bexp);
    int32_t* inv = reinterpret_cast<int32_t*>(ws + W.inv);
    int32_t* meta = reinterpret_cast<int32_t*>(ws + W.meta);
    ExpertLoc* loc = reinterpret_cast<ExpertLoc*>(ws + W.loc);
    uint16_t* h = reinterpret_cast<uint16_t*>(ws + W.h);
    float* y = reinterpret_cast<float*>(ws + W.y);

    // The scratch keeps the previous call's contents; everything below is written before it is
    // read.
    const pmoe_layer_desc& D = *desc;
    ResolveArgs rs{};
    rs.page_table = page_table;
    rs.buf_slot = buf_slot;
    rs.num_pages = num_pages;
    rs.slots_per_buffer = D.slots_per_buffer;
    rs.have_buf0 = load_buf0 != nullptr;
    rs.have_buf1 = load_buf1 != nullptr;
    rs.contiguous = 0;
    rs.loc = loc;
    rs.err = err;
    LayerPtrs L{};
    L.map_base[0] = static_cast<const uint16_t*>(page_pool);
    L.map_base[1] = static_cast<const uint16_t*>(load_buf0);
    L.map_base[2] = static_cast<const uint16_t*>(load_buf1);
    L.d = D.d; L.f = D.f; L.E = D.num_experts; L.k = D.top_k; L.S = D.num_shared_chunks; L.T = T;

    if ((e = launch_route(router_logits, T, D.num_experts, D.top_k, D.renormalize, ids, w, s)) != cudaSuccess ||
        (e = launch_align(ids, T, D.top_k, D.num_experts, D.num_shared_chunks, W.bm, sorted, bexp,
                          inv, meta, &rs, s)) != cudaSuccess ||
        (e = launch_stream_gemm1(L, static_cast<const uint16_t*>(hidden), sorted, bexp, meta, loc,
                                 W.bm, W.nblk, h, s)) != cudaSuccess ||
        (e = launch_stream_gemm2(L, sorted, bexp, meta, loc, W.bm, W.nblk, W.splits, W.cap, h, y,
                                 s)) != cudaSuccess ||
        (e = launch_combine(y, false, W.splits, W.cap, w, inv, T, D.d, D.top_k, D.num_shared_chunks,
                            static_cast<uint16_t*>(out), s)) != cudaSuccess)
        return record_failure(PMOE_ERR_CUDA, "kernel launch failed");
    return PMOE_OK;
}

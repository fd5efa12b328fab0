// Copy-in of routed experts that were not prefetched.
//
// Rimuru (paper-daily.com/en, "The pipeline: what happens in one scheduling round"): the GPU-side
// manager merges the experts it predicts a layer will need into that layer's prefetch queue, but
// the layer's actual routing decides; an expert the routing picks that is neither cached in the
// pool nor in the load buffer has to be copied in before the layer computes.  Here that step runs
// on the device, on the compute stream, right before the layer's forward call, so it needs no
// host round trip (and stays inside a captured CUDA graph):
//
//   scan  CTAs route the tokens (the forward's own warp routine, so the same experts) and OR the
//         routed experts into a bitmap in plan memory; the last CTA to arrive takes every routed
//         expert marked absent (buf_slot = -2) in ascending id, gives each the next free slot of
//         load buffer `buf` (a slot no expert's buf_slot points at), writes the new buf_slot
//         entry and the list of copies, and clears the bitmap for the next call;
//   copy  every CTA streams its share of those experts' W1 | W3 | W2 from mapped pinned host
//         memory (NVLink-C2C) into their slots with 16-byte loads and stores.
//
// Neither kernel lets the next kernel start early, so the forward that follows sees the new
// table entries and the copied bytes before it reads either.
#include "pmoe_internal.cuh"
#include "route_common.cuh"

namespace pmoe {

namespace {

constexpr int kScanWarps = 4;
constexpr int kCopyThreads = 256;

// Plan words used here (after the error word, before the fused kernel's barrier words).
constexpr size_t kBitmapOffset = 256;   // uint32 [kMaxExpertsTotal / 32]: routed experts
constexpr size_t kCounterOffset = 384;  // uint32: CTAs of the running scan that have finished

template <int EPL>
__global__ void __launch_bounds__(kScanWarps * 32) copy_in_scan_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ buf_slot, int buf,
    int slots, const void* const* __restrict__ host_experts, uint32_t* bitmap, uint32_t* counter,
    int32_t* __restrict__ missed, int32_t* __restrict__ err) {
    __shared__ int32_t ids_s[kScanWarps][kMaxTopK];
    __shared__ float w_s[kScanWarps][kMaxTopK];
    __shared__ int last_s;
    // last CTA only: used[ceil(slots/32)] slots of buffer `buf` in use, absent[E] the absent
    // routed experts in ascending id, freeslot[E] the free slots in ascending order
    extern __shared__ uint32_t dyn[];
    pdl_wait_prev();   // logits and tables may come from the previous kernel; no early trigger
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kScanWarps + warp;
    if (t < T) {
        route_token<EPL>(logits + (int64_t)t * E, E, k, 0, lane, ids_s[warp], w_s[warp]);
        __syncwarp();
        if (lane < k) {
            const int e = ids_s[warp][lane];
            atomicOr(&bitmap[e >> 5], 1u << (e & 31));
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();   // this CTA's bits before its arrival
        last_s = atomicAdd(counter, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last_s) return;
    __threadfence();       // every CTA's bits are visible from here on

    const int nw = (slots + 31) / 32;
    uint32_t* used = dyn;
    int32_t* absent = reinterpret_cast<int32_t*>(dyn + nw);
    int32_t* freeslot = absent + E;
    for (int i = threadIdx.x; i < nw; i += blockDim.x) used[i] = 0u;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int r = buf_slot[e] - buf * slots;
        if (r >= 0 && r < slots) atomicOr(&used[r >> 5], 1u << (r & 31));
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t lt = (1u << lane) - 1u;
        int na = 0;   // absent routed experts, ascending id
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const bool a = e < E && (__ldcg(&bitmap[e0 >> 5]) >> lane & 1u) && buf_slot[e] == -2;
            const uint32_t bal = __ballot_sync(0xffffffffu, a);
            if (a) absent[na + __popc(bal & lt)] = e;
            na += __popc(bal);
        }
        int nf = 0;   // the first na free slots, ascending
        for (int s0 = 0; s0 < slots && nf < na; s0 += 32) {
            const int sl = s0 + lane;
            const bool f = sl < slots && !(used[s0 >> 5] >> lane & 1u);
            const uint32_t bal = __ballot_sync(0xffffffffu, f);
            const int pos = nf + __popc(bal & lt);
            if (f && pos < na) freeslot[pos] = sl;
            nf += __popc(bal);
        }
        nf = nf < na ? nf : na;
        __syncwarp();
        int m = 0;    // experts that get a slot: the i-th absent expert takes the i-th free slot
        for (int i0 = 0; i0 < na; i0 += 32) {
            const int i = i0 + lane;
            bool ok = false;
            int e = -1, sl = -1;
            if (i < na) {
                e = absent[i];
                if (i >= nf) {
                    raise_error(err, PMOE_ERR_SLOT_OOB);      // no free slot left: stays absent
                } else if (!host_experts[e]) {
                    raise_error(err, PMOE_ERR_INVALID_ARG);   // no host copy to bring in
                } else {
                    ok = true;
                    sl = freeslot[i];
                    buf_slot[e] = buf * slots + sl;
                }
            }
            const uint32_t bal = __ballot_sync(0xffffffffu, ok);
            if (ok) {
                const int pos = m + __popc(bal & lt);
                missed[1 + pos] = e;
                missed[1 + E + pos] = sl;
            }
            m += __popc(bal);
        }
        if (lane == 0) missed[0] = m;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < (E + 31) / 32; i += blockDim.x) bitmap[i] = 0u;
    if (threadIdx.x == 0) *counter = 0u;
}

// Every CTA copies one contiguous share of the concatenated experts (whole 16 KB pieces), so
// the expert and its source and destination change only at the few expert boundaries inside a
// share; each thread keeps U 16-byte loads of host memory in flight before storing them.
__global__ void __launch_bounds__(kCopyThreads) copy_in_kernel(
    const int32_t* __restrict__ missed, int E, const void* const* __restrict__ host_experts,
    uint4* __restrict__ buf_base, int64_t slot_vecs) {
    pdl_wait_prev();   // the scan's list; no early trigger: the forward reads these bytes next
    constexpr int U = 8;
    constexpr int64_t kPiece = 1024;   // 16-byte vectors
    const int n = missed[0];
    const int64_t total = (int64_t)n * slot_vecs;
    const int64_t per = ((total + gridDim.x - 1) / gridDim.x + kPiece - 1) / kPiece * kPiece;
    const int64_t beg = (int64_t)blockIdx.x * per;
    const int64_t end = beg + per < total ? beg + per : total;
    for (int64_t base = beg; base < end;) {
        const int q = (int)(base / slot_vecs);
        const int64_t off0 = base - (int64_t)q * slot_vecs;
        const int64_t len = (end - base < slot_vecs - off0) ? end - base : slot_vecs - off0;
        const uint4* src = static_cast<const uint4*>(host_experts[missed[1 + q]]) + off0;
        uint4* dst = buf_base + (int64_t)missed[1 + E + q] * slot_vecs + off0;
        for (int64_t i0 = threadIdx.x; i0 < len; i0 += (int64_t)U * kCopyThreads) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + (int64_t)u * kCopyThreads;
                if (i < len) v[u] = src[i];
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + (int64_t)u * kCopyThreads;
                if (i < len) dst[i] = v[u];
            }
        }
        base += len;
    }
}

}  // namespace

cudaError_t launch_copy_in(const Plan& P, const float* logits, int T, int32_t* buf_slot, int buf,
                           const void* const* host_experts, int32_t* missed, cudaStream_t s) {
    const pmoe_layer_desc& D = P.desc;
    const int E = D.num_experts, k = D.top_k, slots = D.slots_per_buffer;
    char* words = reinterpret_cast<char*>(P.d_error);
    uint32_t* bitmap = reinterpret_cast<uint32_t*>(words + kBitmapOffset);
    uint32_t* counter = reinterpret_cast<uint32_t*>(words + kCounterOffset);
    const dim3 grid((unsigned)((T + kScanWarps - 1) / kScanWarps)), block(kScanWarps * 32);
    const size_t smem = sizeof(uint32_t) * ((size_t)(slots + 31) / 32 + 2 * (size_t)E);
    cudaError_t e;
#define SCAN(EPL) launch_pdl(copy_in_scan_kernel<EPL>, grid, block, smem, s, logits, T, E, k, buf_slot, buf, \
                             slots, host_experts, bitmap, counter, missed, P.d_error)
    if (E <= 32) e = SCAN(1);
    else if (E <= 64) e = SCAN(2);
    else if (E <= 128) e = SCAN(4);
    else if (E <= 256) e = SCAN(8);
    else if (E <= 512) e = SCAN(16);
    else e = SCAN(32);
#undef SCAN
    if (e != cudaSuccess) return e;
    const int64_t slot_vecs = (int64_t)3 * D.f * D.d * 2 / 16;
    // a few waves of 16-byte loads in flight per SM: host memory answers slowly
    const unsigned copy_grid = (unsigned)(4 * (P.num_sms > 0 ? P.num_sms : 148));
    return launch_pdl(copy_in_kernel, dim3(copy_grid), dim3(kCopyThreads), 0, s, (const int32_t*)missed,
                      E, host_experts, static_cast<uint4*>(const_cast<void*>(P.buf[buf])), slot_vecs);
}

}  // namespace pmoe

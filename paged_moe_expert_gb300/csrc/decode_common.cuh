// Device building blocks shared by the persistent decode kernels (tc_fused.cu, tc_slice.cu): page
// resolution, the grid barrier, the named barriers of the routing/epilogue warp group and a
// group-wide prefix scan.
#pragma once

#include "tc_common.cuh"

namespace pmoe {
namespace dec {
namespace {

using namespace tc;

constexpr int kGroupThreads = 256;             // warps 2..9 of a decode kernel: routing, epilogues, combine
constexpr int kGroupWarps = kGroupThreads / 32;

// Where matrix j of expert e lives: (map, page).  Shared chunks (e >= E) are pool pages.  A page
// or slot out of range raises the error and reads pool page 0 instead (the output is undefined
// then, but every role of every CTA still runs the same schedule).
__device__ __forceinline__ int2 resolve(const FusedArgs& a, int e, int j) {
    if (a.contig) return make_int2(0, 3 * e + j);
    const int bs = e < a.E ? a.buf_slot[e] : -1;
    if (bs >= 0) {
        const int b = a.slots_per_buffer > 0 ? bs / a.slots_per_buffer : 2;
        const bool have = (b == 0 && a.have_buf0) || (b == 1 && a.have_buf1);
        if (b < 2 && have) return make_int2(1 + b, 3 * (bs % a.slots_per_buffer) + j);
        raise_error(a.err, PMOE_ERR_SLOT_OOB);
        return make_int2(0, 0);
    }
    if (bs != -1) {
        raise_error(a.err, PMOE_ERR_SLOT_OOB);
        return make_int2(0, 0);
    }
    const int p = a.page_table[e * 3 + j];
    if (p >= 0 && p < a.num_pages) return make_int2(0, p);
    raise_error(a.err, PMOE_ERR_PAGE_OOB);
    return make_int2(0, 0);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier over the G resident CTAs, run by one whole warp per CTA after the CTA synchronised
// its writes (bar.sync orders them before lane 0's release store, which publishes them gpu-wide:
// a release is cumulative).  Every CTA owns one word; it publishes `target` there, then the warp
// polls all G words (a few cache lines, one load per lane) until each has reached `target`, and
// an acquire fence orders what the CTA reads next after the other CTAs' writes.  The words only
// count up (one step per call), so they are equal between calls and each call continues from
// their value at its start.  Bounded: gives up after ~2 s (or when the CTA already aborted),
// raising PMOE_ERR_TIMEOUT.
__device__ bool grid_barrier(uint32_t* flags, int G, int cta, uint32_t target, int lane,
                             volatile int* abort_flag, int32_t* err) {
    if (lane == 0)
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flags + cta), "r"(target) : "memory");
    __syncwarp();
    const uint64_t t0 = globaltimer();
    const volatile uint32_t* vf = flags;
    for (uint32_t it = 1;; ++it) {
        bool mine = true;
        for (int c = lane; c < G; c += 32)
            if ((int32_t)(vf[c] - target) < 0) mine = false;
        if (__all_sync(0xffffffffu, mine)) break;
        if ((it & 15u) == 0) {
            const bool stop = *abort_flag || globaltimer() - t0 > 2000000000ull;
            if (__any_sync(0xffffffffu, stop)) {
                if (lane == 0 && !*abort_flag) {
                    *abort_flag = 1;
                    raise_error(err, PMOE_ERR_TIMEOUT);
                }
                return false;
            }
        }
    }
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    return true;
}

__device__ __forceinline__ void group_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kGroupThreads) : "memory"); }
// the four epilogue warps (2..5)
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Inclusive prefix (sum or max) over the 256 threads of the group, one value per thread.
template <bool kMax>
__device__ __forceinline__ int32_t group_scan(int32_t v, int lane, int gw, int32_t* wtot) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v = kMax ? max(v, y) : v + y;
    }
    if (lane == 31) wtot[gw] = v;
    group_bar();
    int32_t base = kMax ? INT32_MIN : 0;
    for (int w = 0; w < gw; ++w) base = kMax ? max(base, wtot[w]) : base + wtot[w];
    group_bar();   // wtot may be reused after this
    return kMax ? max(base, v) : base + v;
}

}  // namespace
}  // namespace dec
}  // namespace pmoe

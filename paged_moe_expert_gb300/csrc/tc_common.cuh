// tcgen05 / TMA / mbarrier building blocks shared by the tensor-core kernels (sm_103a).
#pragma once

#include "pmoe_internal.cuh"

namespace pmoe {
namespace tc {

// Instruction descriptor of tcgen05.mma.kind::f16 with fp32 accumulation and bf16 A and B,
// both K-major: bits 4..5 D format (1 = f32), 7..9 A format (1 = bf16), 10..12 B format
// (1 = bf16), 17..22 N >> 3, 24..28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

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

// The same load with an L2 cache policy (createpolicy), e.g. evict-first for data read once.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int c0, int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- tensor stores from shared memory (epilogues) ----

// 2D tiled TMA store of a shared-memory box, tracked by this thread's bulk async-groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most the most recent bulk group of this thread still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Waits until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Makes this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
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

__device__ __forceinline__ void st_shared_v4u(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Epilogue of an fp32 accumulator to bf16: this warp's 32 TMEM lanes (32 output rows) x 64
// columns from TMEM column address `taddr` are rounded to bf16 into a 4 KB shared-memory box in
// the 128-byte swizzled layout (row r's 16-byte chunk j at chunk j ^ (r mod 8): the warp's stores
// hit every bank once per four wavefronts) and stored to y[row0 .. row0+31][col0 .. col0+63] by
// one TMA store issued by lane 0.  `box` must be 1024-byte aligned and the caller must alternate
// two boxes: before writing one, lane 0 waits until only its latest store (from the other box)
// may still be reading shared memory.
__device__ __forceinline__ void store_rows_bf16x64(const CUtensorMap* ymap, uint32_t box, uint32_t taddr,
                                                   int lane, int col0, int row0) {
    if (lane == 0) bulk_wait_read_1();
    __syncwarp();
    const uint32_t rb = box + (uint32_t)lane * 128u;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float a[16], b[16];
        tmem_ld16(taddr + 32u * half, a);
        tmem_ld16(taddr + 32u * half + 16u, b);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            st_shared_v4u(rb + ((uint32_t)((4 * half + j) ^ (lane & 7)) << 4), pack_bf16(a[8 * j], a[8 * j + 1]),
                          pack_bf16(a[8 * j + 2], a[8 * j + 3]), pack_bf16(a[8 * j + 4], a[8 * j + 5]),
                          pack_bf16(a[8 * j + 6], a[8 * j + 7]));
            st_shared_v4u(rb + ((uint32_t)((4 * half + 2 + j) ^ (lane & 7)) << 4),
                          pack_bf16(b[8 * j], b[8 * j + 1]), pack_bf16(b[8 * j + 2], b[8 * j + 3]),
                          pack_bf16(b[8 * j + 4], b[8 * j + 5]), pack_bf16(b[8 * j + 6], b[8 * j + 7]));
        }
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(ymap, box, col0, row0);
        bulk_commit();
    }
}

}  // namespace tc
}  // namespace pmoe

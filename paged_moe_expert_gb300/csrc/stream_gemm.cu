// Weight-streaming paged expert GEMMs for decode-sized batches, and the weighted combine.
//
// At a few tokens per expert the layer is bound by reading each active expert's three pages
// once.  These kernels stream weight rows with 16-byte non-allocating loads, keep the block's
// tokens in shared memory, and reduce each (row, token) dot product across a warp in a fixed
// order.  The page lookup follows Rimuru's address rule (paper-daily.com/en, "Expert weights
// are scattered across pages. How does the kernel read them?"):
//     addr_e(n, t) = B_P + p_e(n) * f * d + (n mod f) * d + t
// -- the page (or buffer slot) of expert e's matrix is resolved once per CTA, then rows are read
// at fixed strides inside the page.  Gate (W1) and up (W3) rows come from two different pages
// and are never concatenated in memory.
#include <math.h>

#include "pmoe_internal.cuh"

namespace pmoe {

namespace {

constexpr int kThreads = 256;      // 8 warps
constexpr int kRows1 = 16;         // gate/up rows (of f) per CTA
constexpr int kRows2 = 16;         // down rows (of d) per CTA
constexpr int kUnroll = 4;         // 16-byte chunks in flight per lane and matrix

__device__ __forceinline__ float dot8(const uint4& w, const uint4& x) {
    float s = bf16_lo(w.x) * bf16_lo(x.x);
    s = fmaf(bf16_hi(w.x), bf16_hi(x.x), s);
    s = fmaf(bf16_lo(w.y), bf16_lo(x.y), s);
    s = fmaf(bf16_hi(w.y), bf16_hi(x.y), s);
    s = fmaf(bf16_lo(w.z), bf16_lo(x.z), s);
    s = fmaf(bf16_hi(w.z), bf16_hi(x.z), s);
    s = fmaf(bf16_lo(w.w), bf16_lo(x.w), s);
    s = fmaf(bf16_hi(w.w), bf16_hi(x.w), s);
    return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Token index of a pair (routed pair t*k + j, shared pair T*k + s*T + t).
__device__ __forceinline__ int pair_token(int pair, int T, int k) {
    const int NR = T * k;
    return pair < NR ? pair / k : (pair - NR) % T;
}

// Rows of block b that hold a pair (the rest are pads at the tail).
template <int MT>
__device__ __forceinline__ int block_rows(const int32_t* sorted_ids, int b, int NP) {
    int c = 0;
#pragma unroll
    for (int r = 0; r < MT; ++r) c += sorted_ids[b * MT + r] < NP ? 1 : 0;
    return c;
}

// Base of a map without indexing the parameter array dynamically (that would spill it).
__device__ __forceinline__ const uint16_t* map_ptr(const LayerPtrs& L, int map) {
    return map == 0 ? L.map_base[0] : (map == 1 ? L.map_base[1] : L.map_base[2]);
}

__device__ __forceinline__ ExpertLoc resolve(const ExpertLoc* loc, int e, int j, bool contig) {
    if (contig) return ExpertLoc{0, 3 * e + j};
    return loc[e * 3 + j];
}

// h[b*MT + m][n] = bf16( silu(W1_e[n] . x_m) * (W3_e[n] . x_m) ) for the block's real rows m.
template <int MT, bool kContig>
__global__ void __launch_bounds__(kThreads) stream_gemm1_kernel(
    LayerPtrs L, const uint16_t* __restrict__ hidden, const int32_t* __restrict__ sorted_ids,
    const int32_t* __restrict__ block_expert, const int32_t* __restrict__ meta,
    const ExpertLoc* __restrict__ loc, uint16_t* __restrict__ h) {
    extern __shared__ uint4 xs[];  // [MT][d/8]
    pdl_wait_prev();
    pdl_allow_next();
    const int b = blockIdx.y;
    if (b * MT >= meta[kMetaNPadded]) return;
    const int d = L.d, f = L.f, dv = d >> 3;
    const int NP = L.T * (L.k + L.S);
    const int e = block_expert[b];
    const ExpertLoc l1 = resolve(loc, e, 0, kContig), l3 = resolve(loc, e, 1, kContig);
    if (l1.map < 0 || l3.map < 0) return;  // invalid page: reported by the resolve step
    const int m_real = block_rows<MT>(sorted_ids, b, NP);

    for (int idx = threadIdx.x; idx < MT * dv; idx += kThreads) {
        const int r = idx / dv, c = idx - r * dv;
        const int pair = sorted_ids[b * MT + r];
        uint4 v = make_uint4(0, 0, 0, 0);
        if (pair < NP) v = reinterpret_cast<const uint4*>(hidden + (int64_t)pair_token(pair, L.T, L.k) * d)[c];
        xs[idx] = v;
    }
    __syncthreads();

    // p_e(n) for n < f is the W1 page, for n >= f the W3 page; (n mod f) is the row inside it.
    const uint16_t* w1 = map_ptr(L, l1.map) + (int64_t)l1.page * f * d;
    const uint16_t* w3 = map_ptr(L, l3.map) + (int64_t)l3.page * f * d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kRowsPerWarp = kRows1 / (kThreads / 32);
#pragma unroll 1
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int n = blockIdx.x * kRows1 + warp * kRowsPerWarp + rr;
        const uint4* r1 = reinterpret_cast<const uint4*>(w1 + (int64_t)n * d);
        const uint4* r3 = reinterpret_cast<const uint4*>(w3 + (int64_t)n * d);
        float g[MT], u[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) g[m] = u[m] = 0.f;
        for (int c0 = lane; c0 < dv; c0 += 32 * kUnroll) {
            uint4 a[kUnroll], bq[kUnroll];
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int c = c0 + 32 * q;
                if (c < dv) {
                    a[q] = ld_stream_v4(r1 + c);
                    bq[q] = ld_stream_v4(r3 + c);
                }
            }
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int c = c0 + 32 * q;
                if (c < dv) {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m < m_real) {
                            const uint4 x = xs[m * dv + c];
                            g[m] += dot8(a[q], x);
                            u[m] += dot8(bq[q], x);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < m_real) {
                const float gs = warp_sum(g[m]);
                const float us = warp_sum(u[m]);
                if (lane == m % 32) {
                    const float a = silu_mul(gs, us);
                    h[(int64_t)(b * MT + m) * f + n] = f32_to_bf16_bits(a);
                }
            }
        }
    }
}

// y[split][b*MT + m][r] = W2_e[r][k0:k0+kc] . h[b*MT + m][k0:k0+kc] for the block's real rows.
template <int MT, bool kContig>
__global__ void __launch_bounds__(kThreads) stream_gemm2_kernel(
    LayerPtrs L, const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ block_expert,
    const int32_t* __restrict__ meta, const ExpertLoc* __restrict__ loc,
    const uint16_t* __restrict__ h, float* __restrict__ y, int64_t ystride) {
    extern __shared__ uint4 hs[];  // [MT][kc/8]
    pdl_wait_prev();
    pdl_allow_next();
    const int b = blockIdx.y;
    if (b * MT >= meta[kMetaNPadded]) return;
    const int d = L.d, f = L.f;
    const int NP = L.T * (L.k + L.S);
    const int e = block_expert[b];
    const ExpertLoc l2 = resolve(loc, e, 2, kContig);
    if (l2.map < 0) return;
    const int m_real = block_rows<MT>(sorted_ids, b, NP);
    const int k0 = blockIdx.z * kStreamKChunk;
    const int kc = min(kStreamKChunk, f - k0);
    const int kv = kc >> 3;

    for (int idx = threadIdx.x; idx < m_real * kv; idx += kThreads) {
        const int r = idx / kv, c = idx - r * kv;
        hs[idx] = reinterpret_cast<const uint4*>(h + (int64_t)(b * MT + r) * f + k0)[c];
    }
    __syncthreads();

    const uint16_t* w2 = map_ptr(L, l2.map) + (int64_t)l2.page * f * d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kRowsPerWarp = kRows2 / (kThreads / 32);
    float* yb = y + (int64_t)blockIdx.z * ystride * d;
#pragma unroll 1
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = blockIdx.x * kRows2 + warp * kRowsPerWarp + rr;
        const uint4* wr = reinterpret_cast<const uint4*>(w2 + (int64_t)r * f + k0);
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        for (int c0 = lane; c0 < kv; c0 += 32 * kUnroll) {
            uint4 a[kUnroll];
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int c = c0 + 32 * q;
                if (c < kv) a[q] = ld_stream_v4(wr + c);
            }
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int c = c0 + 32 * q;
                if (c < kv) {
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < m_real) acc[m] += dot8(a[q], hs[m * kv + c]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < m_real) {
                const float s = warp_sum(acc[m]);
                if (lane == m % 32) yb[(int64_t)(b * MT + m) * d + r] = s;
            }
        }
    }
}

template <typename K>
cudaError_t allow_smem(K kernel, std::atomic<unsigned long long>* done) {
    return raise_smem_limit(reinterpret_cast<const void*>(kernel), 200 * 1024, done);
}

template <int MT, bool C>
cudaError_t gemm1_mt(const LayerPtrs& L, const uint16_t* hidden, const int32_t* sorted_ids,
                     const int32_t* block_expert, const int32_t* meta, const ExpertLoc* loc,
                     int64_t nblk_max, uint16_t* h, cudaStream_t s) {
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = allow_smem(stream_gemm1_kernel<MT, C>, &attr);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(L.f / kRows1), (unsigned)nblk_max);
    const size_t smem = (size_t)MT * L.d * 2;
    return launch_pdl(stream_gemm1_kernel<MT, C>, grid, dim3(kThreads), smem, s, L, hidden, sorted_ids,
                      block_expert, meta, loc, h);
}

template <int MT, bool C>
cudaError_t gemm2_mt(const LayerPtrs& L, const int32_t* sorted_ids, const int32_t* block_expert,
                     const int32_t* meta, const ExpertLoc* loc, int64_t nblk_max, int splits,
                     int64_t ystride, const uint16_t* h, float* y, cudaStream_t s) {
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = allow_smem(stream_gemm2_kernel<MT, C>, &attr);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(L.d / kRows2), (unsigned)nblk_max, (unsigned)splits);
    const size_t smem = (size_t)MT * (L.f < kStreamKChunk ? L.f : kStreamKChunk) * 2;
    return launch_pdl(stream_gemm2_kernel<MT, C>, grid, dim3(kThreads), smem, s, L, sorted_ids,
                      block_expert, meta, loc, h, y, ystride);
}

// contiguous addressing is selected by loc == nullptr
#define PMOE_MT_SWITCH(MTV, CALL_T, CALL_F) \
    switch (MTV) {                          \
        case 1: return contig ? CALL_T(1) : CALL_F(1);   \
        case 2: return contig ? CALL_T(2) : CALL_F(2);   \
        case 4: return contig ? CALL_T(4) : CALL_F(4);   \
        case 8: return contig ? CALL_T(8) : CALL_F(8);   \
        case 16: return contig ? CALL_T(16) : CALL_F(16); \
        default: return cudaErrorInvalidValue;           \
    }

}  // namespace

cudaError_t launch_stream_gemm1(const LayerPtrs& L, const uint16_t* hidden,
                                const int32_t* sorted_ids, const int32_t* block_expert,
                                const int32_t* meta, const ExpertLoc* loc, int block_m,
                                int64_t nblk_max, uint16_t* h, cudaStream_t s) {
    const bool contig = loc == nullptr;
#define G1T(M) gemm1_mt<M, true>(L, hidden, sorted_ids, block_expert, meta, loc, nblk_max, h, s)
#define G1F(M) gemm1_mt<M, false>(L, hidden, sorted_ids, block_expert, meta, loc, nblk_max, h, s)
    PMOE_MT_SWITCH(block_m, G1T, G1F)
#undef G1T
#undef G1F
}

cudaError_t launch_stream_gemm2(const LayerPtrs& L, const int32_t* sorted_ids,
                                const int32_t* block_expert, const int32_t* meta,
                                const ExpertLoc* loc, int block_m, int64_t nblk_max, int splits,
                                int64_t ystride, const uint16_t* h, float* y, cudaStream_t s) {
    const bool contig = loc == nullptr;
#define G2T(M) gemm2_mt<M, true>(L, sorted_ids, block_expert, meta, loc, nblk_max, splits, ystride, h, y, s)
#define G2F(M) gemm2_mt<M, false>(L, sorted_ids, block_expert, meta, loc, nblk_max, splits, ystride, h, y, s)
    PMOE_MT_SWITCH(block_m, G2T, G2F)
#undef G2T
#undef G2F
}

// ---------------------------------------------------------------------------------------------
// Combine: out[t] = bf16( sum_j w[t,j] * y[inv[t*k+j]] + sum_s y[inv[T*k + s*T + t]] ), with
// each y a bf16 row (the 128-token-block and CTA-pair paths) or the fp32 sum of its K-split
// partials (the small-batch and weight-streaming paths); the order of every sum is fixed (pairs
// in order j, then shared chunks s, each a fused multiply-add with weight 1 for the shared
// ones), so the output
// does not depend on where the experts live or on scheduling.  A thread owns four columns of one
// token and issues the loads of up to eight pairs before it adds any of them.
// ---------------------------------------------------------------------------------------------
constexpr int kCombineThreads = 64;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const float* __restrict__ y, int splits, int64_t ystride, const float* __restrict__ w,
    const int32_t* __restrict__ inv, int T, int d, int k, int S, uint16_t* __restrict__ out) {
    pdl_wait_prev();
    pdl_allow_next();
    const int t = blockIdx.y;
    const int c = blockIdx.x * kCombineThreads + threadIdx.x;   // float4 column
    const int P = k + S;
    const int64_t NR = (int64_t)T * k;
    __shared__ int64_t s_row[64];
    __shared__ float s_w[64];
    for (int p = threadIdx.x; p < P; p += kCombineThreads) {
        s_row[p] = p < k ? inv[(int64_t)t * k + p] : inv[NR + (int64_t)(p - k) * T + t];
        s_w[p] = p < k ? w[(int64_t)t * k + p] : 1.f;
    }
    __syncthreads();
    if (c >= (d >> 2)) return;
    const float4* y4 = reinterpret_cast<const float4*>(y);
    const int64_t dq = d >> 2;
    const int64_t split_q = ystride * dq;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < P; p0 += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p0 + i < P) v[i] = __ldg(y4 + s_row[p0 + i] * dq + c);
        }
        for (int sp = 1; sp < splits; ++sp) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (p0 + i < P) {
                    const float4 u = __ldg(y4 + sp * split_q + s_row[p0 + i] * dq + c);
                    v[i].x += u.x; v[i].y += u.y; v[i].z += u.z; v[i].w += u.w;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (p0 + i < P) {
                const float wp = s_w[p0 + i];
                acc.x = fmaf(wp, v[i].x, acc.x);
                acc.y = fmaf(wp, v[i].y, acc.y);
                acc.z = fmaf(wp, v[i].z, acc.z);
                acc.w = fmaf(wp, v[i].w, acc.w);
            }
        }
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(acc.x) | ((uint32_t)f32_to_bf16_bits(acc.y) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(acc.z) | ((uint32_t)f32_to_bf16_bits(acc.w) << 16);
    reinterpret_cast<uint2*>(out + (int64_t)t * d)[c] = o;
}

// The same sum over bf16 y rows (the 128-token-block and CTA-pair paths, no K split): a thread owns
// CPT groups of eight columns, c, c + G, ... (G: the token's threads), one 16-byte load per pair
// row and group, eight loads in flight per thread: with few pairs per token (top-2) a thread takes
// four groups, so each round trip to memory carries as many bytes as with eight pairs.  Each
// column is summed over the pairs in order, whatever CPT is.
template <int CPT>
__global__ void __launch_bounds__(kCombineThreads) combine_bf16_kernel(
    const uint16_t* __restrict__ y, const float* __restrict__ w, const int32_t* __restrict__ inv,
    int T, int d, int k, int S, uint16_t* __restrict__ out) {
    constexpr int PB = 8 / CPT;   // pairs per batch of loads
    pdl_wait_prev();
    pdl_allow_next();
    const int t = blockIdx.y;
    const int c = blockIdx.x * kCombineThreads + threadIdx.x;   // first group of 8 columns
    const int G = gridDim.x * kCombineThreads;
    const int P = k + S;
    const int64_t NR = (int64_t)T * k;
    __shared__ int64_t s_row[64];
    __shared__ float s_w[64];
    for (int p = threadIdx.x; p < P; p += kCombineThreads) {
        s_row[p] = p < k ? inv[(int64_t)t * k + p] : inv[NR + (int64_t)(p - k) * T + t];
        s_w[p] = p < k ? w[(int64_t)t * k + p] : 1.f;
    }
    __syncthreads();
    const int d8 = d >> 3;
    if (c >= d8) return;
    const uint4* y8 = reinterpret_cast<const uint4*>(y);
    float acc[CPT][8];
#pragma unroll
    for (int j = 0; j < CPT; ++j)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[j][q] = 0.f;
    for (int p0 = 0; p0 < P; p0 += PB) {
        uint4 v[PB][CPT];
#pragma unroll
        for (int i = 0; i < PB; ++i)
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                v[i][j] = make_uint4(0u, 0u, 0u, 0u);
                if (p0 + i < P && c + j * G < d8) v[i][j] = __ldg(y8 + s_row[p0 + i] * d8 + c + j * G);
            }
#pragma unroll
        for (int i = 0; i < PB; ++i) {
            if (p0 + i < P) {
                const float wp = s_w[p0 + i];
#pragma unroll
                for (int j = 0; j < CPT; ++j) {
                    acc[j][0] = fmaf(wp, bf16_lo(v[i][j].x), acc[j][0]);
                    acc[j][1] = fmaf(wp, bf16_hi(v[i][j].x), acc[j][1]);
                    acc[j][2] = fmaf(wp, bf16_lo(v[i][j].y), acc[j][2]);
                    acc[j][3] = fmaf(wp, bf16_hi(v[i][j].y), acc[j][3]);
                    acc[j][4] = fmaf(wp, bf16_lo(v[i][j].z), acc[j][4]);
                    acc[j][5] = fmaf(wp, bf16_hi(v[i][j].z), acc[j][5]);
                    acc[j][6] = fmaf(wp, bf16_lo(v[i][j].w), acc[j][6]);
                    acc[j][7] = fmaf(wp, bf16_hi(v[i][j].w), acc[j][7]);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        if (c + j * G >= d8) break;
        uint4 o;
        o.x = (uint32_t)f32_to_bf16_bits(acc[j][0]) | ((uint32_t)f32_to_bf16_bits(acc[j][1]) << 16);
        o.y = (uint32_t)f32_to_bf16_bits(acc[j][2]) | ((uint32_t)f32_to_bf16_bits(acc[j][3]) << 16);
        o.z = (uint32_t)f32_to_bf16_bits(acc[j][4]) | ((uint32_t)f32_to_bf16_bits(acc[j][5]) << 16);
        o.w = (uint32_t)f32_to_bf16_bits(acc[j][6]) | ((uint32_t)f32_to_bf16_bits(acc[j][7]) << 16);
        reinterpret_cast<uint4*>(out + (int64_t)t * d)[c + j * G] = o;
    }
}

cudaError_t launch_combine(const void* y, bool y_bf16, int splits, int64_t ystride, const float* w,
                           const int32_t* inv, int T, int d, int k, int S, uint16_t* out,
                           cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (y_bf16) {
        const int P = k + S;
        const int cpt = P <= 2 ? 4 : P <= 4 ? 2 : 1;   // groups of 8 columns per thread
        const int threads = (d / 8 + cpt - 1) / cpt;
        const dim3 grid((unsigned)((threads + kCombineThreads - 1) / kCombineThreads), (unsigned)T);
        const uint16_t* yb = static_cast<const uint16_t*>(y);
        if (cpt == 4)
            return launch_pdl(combine_bf16_kernel<4>, grid, dim3(kCombineThreads), 0, s, yb, w, inv, T, d, k, S, out);
        if (cpt == 2)
            return launch_pdl(combine_bf16_kernel<2>, grid, dim3(kCombineThreads), 0, s, yb, w, inv, T, d, k, S, out);
        return launch_pdl(combine_bf16_kernel<1>, grid, dim3(kCombineThreads), 0, s, yb, w, inv, T, d, k, S, out);
    }
    const dim3 grid((unsigned)((d / 4 + kCombineThreads - 1) / kCombineThreads), (unsigned)T);
    return launch_pdl(combine_kernel, grid, dim3(kCombineThreads), 0, s, static_cast<const float*>(y),
                      splits, ystride, w, inv, T, d, k, S, out);
}

}  // namespace pmoe

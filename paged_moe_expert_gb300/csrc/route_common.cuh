// Top-k softmax routing of one token by one warp, shared by every kernel that routes (the routing
// kernel, the small-batch sort kernel and the fused decode kernel), so all of them select the same
// experts bit for bit.
#pragma once

#include <math.h>

#include "pmoe_internal.cuh"

namespace pmoe {

// ---------------------------------------------------------------------------------------------
// Routing: one warp per token.  Lane l holds logits l, l+32, l+64, ... (coalesced loads) as
// order-preserving 32-bit keys (-0 counted as +0, so equal values tie).  Each of the k rounds
// takes the warp maximum of the lanes' best keys with one redux, then the lowest expert id among
// the lanes holding it with a second, so the order is (value desc, id asc) exactly; only the
// winning lane rescans its EPL keys.  Softmax over all E with the top-1 value as the max, or, with
// renormalisation, e^(v - max) of the k chosen over their own sum (the same weights: the sum over
// all E cancels, so it is not formed).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Best untaken (key, slot) over a lane's keys: highest key, lowest slot among equal keys.  Key 0
// marks a missing expert (every real value has a key above 0).
template <int EPL>
__device__ __forceinline__ void lane_best(const uint32_t (&key)[EPL], uint32_t taken, uint32_t& bk,
                                          int& bi) {
    bk = 0u;
    bi = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const uint32_t ki = (taken >> i & 1u) ? 0u : key[i];
        if (ki > bk) {
            bk = ki;
            bi = i;
        }
    }
}

template <int EPL>
__device__ __forceinline__ void route_token(const float* __restrict__ lg, int E, int k, int renorm,
                                            int lane, int32_t* __restrict__ ids_out,
                                            float* __restrict__ w_out) {
    uint32_t key[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? order_key(lg[e]) : 0u;
    }
    uint32_t taken = 0u, bk;
    int bi;
    lane_best<EPL>(key, taken, bk, bi);
    // lane j keeps the j-th selection
    int my_id = 0;
    uint32_t my_key = 0u, top = 0u;
    for (int j = 0; j < k; ++j) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t cand = bk == m ? (uint32_t)(lane + 32 * bi) : 0xffffffffu;
        const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
        if (j == 0) top = m;
        if (lane == j) {
            my_id = (int)win;
            my_key = m;
        }
        if ((int)(win & 31u) == lane) {
            taken |= 1u << bi;
            lane_best<EPL>(key, taken, bk, bi);
        }
    }
    const float mx = key_value(top);
    const float ej = lane < k ? expf(key_value(my_key) - mx) : 0.f;
    float den = 0.f;
    if (renorm) {
        // renormalised over the k chosen experts, the softmax's sum over all E cancels:
        // w_j = e^(v_j - max) / sum over the chosen of e^(v_i - max)
        den = ej;
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (key[i] != 0u) den += expf(key_value(key[i]) - mx);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane < k) {
        ids_out[lane] = my_id;
        w_out[lane] = ej / den;
    }
}

// Two tokens by one warp, their k rounds interleaved so that the two tokens' reductions are in
// flight together (the rounds are latency-bound): the same selection and weights as route_token
// for each of them.
template <int EPL>
__device__ __forceinline__ void route_token_pair(const float* __restrict__ lg0, const float* __restrict__ lg1,
                                                 int E, int k, int renorm, int lane,
                                                 int32_t* __restrict__ ids0, float* __restrict__ w0,
                                                 int32_t* __restrict__ ids1, float* __restrict__ w1) {
    const float* lg[2] = {lg0, lg1};
    uint32_t key[2][EPL];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            key[n][i] = e < E ? order_key(lg[n][e]) : 0u;
        }
    uint32_t taken[2] = {0u, 0u}, bk[2];
    int bi[2];
#pragma unroll
    for (int n = 0; n < 2; ++n) lane_best<EPL>(key[n], 0u, bk[n], bi[n]);
    int my_id[2] = {0, 0};
    uint32_t my_key[2] = {0u, 0u}, top[2] = {0u, 0u};
    for (int j = 0; j < k; ++j) {
        uint32_t m[2], win[2];
#pragma unroll
        for (int n = 0; n < 2; ++n) m[n] = __reduce_max_sync(0xffffffffu, bk[n]);
#pragma unroll
        for (int n = 0; n < 2; ++n)
            win[n] = __reduce_min_sync(0xffffffffu, bk[n] == m[n] ? (uint32_t)(lane + 32 * bi[n]) : 0xffffffffu);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            if (j == 0) top[n] = m[n];
            if (lane == j) {
                my_id[n] = (int)win[n];
                my_key[n] = m[n];
            }
            if ((int)(win[n] & 31u) == lane) {
                taken[n] |= 1u << bi[n];
                lane_best<EPL>(key[n], taken[n], bk[n], bi[n]);
            }
        }
    }
    int32_t* ids[2] = {ids0, ids1};
    float* wo[2] = {w0, w1};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        const float mx = key_value(top[n]);
        const float ej = lane < k ? expf(key_value(my_key[n]) - mx) : 0.f;
        float den = 0.f;
        if (renorm) {
            den = ej;
        } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (key[n][i] != 0u) den += expf(key_value(key[n][i]) - mx);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (lane < k) {
            ids[n][lane] = my_id[n];
            wo[n][lane] = ej / den;
        }
    }
}

}  // namespace pmoe

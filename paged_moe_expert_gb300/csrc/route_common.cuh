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

}  // namespace pmoe

// topk.cuh -- warp-level top-k of the router logits (shared by the routing
// kernel and the fused layer kernel, so both select identically).
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "A 40B MoE that activates 2.5B parameters": sigmoid top-6 routing.  The
// selection is taken on the fp32 logits (sigmoid is monotone), larger logit
// first, a tie going to the lower expert index.
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving key: larger logit first, then smaller expert index.
// -0.0 is folded into +0.0 (they compare equal as values); NaN sorts last.
__device__ __forceinline__ unsigned long long rank_key(float v, int e)
{
    uint32_t u;
    if (v != v) {
        u = 0u;
    } else {
        v = v + 0.0f;
        u = __float_as_uint(v);
        u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFu - (uint32_t)e);
}

__device__ __forceinline__ int key_expert(unsigned long long k) { return 0xFFFF - (int)(k & 0xFFFFu); }

__device__ __forceinline__ void cas_desc(unsigned long long &a, unsigned long long &b)
{
    unsigned long long hi = a > b ? a : b;
    unsigned long long lo = a > b ? b : a;
    a = hi;
    b = lo;
}

// Sort 8 keys in descending order (Batcher's odd-even merge network, 19 CAS).
__device__ __forceinline__ void sort8_desc(unsigned long long k[8])
{
    cas_desc(k[0], k[1]); cas_desc(k[2], k[3]); cas_desc(k[4], k[5]); cas_desc(k[6], k[7]);
    cas_desc(k[0], k[2]); cas_desc(k[1], k[3]); cas_desc(k[4], k[6]); cas_desc(k[5], k[7]);
    cas_desc(k[1], k[2]); cas_desc(k[5], k[6]);
    cas_desc(k[0], k[4]); cas_desc(k[1], k[5]); cas_desc(k[2], k[6]); cas_desc(k[3], k[7]);
    cas_desc(k[2], k[4]); cas_desc(k[3], k[5]);
    cas_desc(k[1], k[2]); cas_desc(k[3], k[4]); cas_desc(k[5], k[6]);
}

// Sort a bitonic sequence of 8 keys into descending order (12 CAS).
__device__ __forceinline__ void bitonic8_desc(unsigned long long k[8])
{
    cas_desc(k[0], k[4]); cas_desc(k[1], k[5]); cas_desc(k[2], k[6]); cas_desc(k[3], k[7]);
    cas_desc(k[0], k[2]); cas_desc(k[1], k[3]); cas_desc(k[4], k[6]); cas_desc(k[5], k[7]);
    cas_desc(k[0], k[1]); cas_desc(k[2], k[3]); cas_desc(k[4], k[5]); cas_desc(k[6], k[7]);
}

// Top-8 of E = 256 keys held 8 per lane; every lane ends with the sorted top 8.
__device__ __forceinline__ void warp_top8(unsigned long long k[8])
{
    sort8_desc(k);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        unsigned long long p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            p[i] = __shfl_xor_sync(0xFFFFFFFFu, k[i], off);
        // top 8 of two descending lists = elementwise max against the reversed
        // partner list, which is bitonic
#pragma unroll
        for (int i = 0; i < 8; ++i)
            k[i] = k[i] > p[7 - i] ? k[i] : p[7 - i];
        bitonic8_desc(k);
    }
}

// Top-k of one token's E = 256 fp32 logits by one warp: returns in lanes
// 0..TOPK-1 the selected expert (best first) and its renormalised sigmoid
// weight, and reports whether a logit was not finite.
__device__ __forceinline__ void warp_route_token(const float *logits_row, int lane, int &ex, float &wt,
                                                 bool &nonfinite)
{
    unsigned long long k[8];
    bool bad = false;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int ee = lane + 32 * m;
        const float v = __ldcg(logits_row + ee);
        bad |= !isfinite(v);
        k[m] = rank_key(v, ee);
    }
    nonfinite = __any_sync(0xFFFFFFFFu, bad);
    warp_top8(k);
    float s = 0.0f, sum = 0.0f;
    ex = 0;
#pragma unroll
    for (int i = 0; i < TOPK; ++i) {
        const int ei = key_expert(k[i]);
        const float v = __ldcg(logits_row + ei);
        const float si = 1.0f / (1.0f + expf(-v));
        sum += si;
        if (lane == i) { s = si; ex = ei; }
    }
    wt = s / sum;
}

}  // namespace moe

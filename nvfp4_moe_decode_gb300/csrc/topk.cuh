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

// The logit a key was built from (exact; NaN keys give a NaN).
__device__ __forceinline__ float key_logit(unsigned long long key)
{
    const uint32_t u = (uint32_t)(key >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
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
    // TOPK rounds of a warp-wide argmax (keys are unique: index in the low bits)
    float s = 0.0f, sum = 0.0f;
    ex = 0;
#pragma unroll 1
    for (int i = 0; i < TOPK; ++i) {
        unsigned long long best = k[0];
#pragma unroll
        for (int m = 1; m < 8; ++m)
            best = k[m] > best ? k[m] : best;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
            best = o > best ? o : best;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m)
            if (k[m] == best)
                k[m] = 0ull;
        const float si = 1.0f / (1.0f + expf(-key_logit(best)));
        sum += si;
        if (lane == i) {
            s = si;
            ex = key_expert(best);
        }
    }
    wt = s / sum;
}

}  // namespace moe

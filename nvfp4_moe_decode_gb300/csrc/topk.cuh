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

// Descending compare-exchange of two keys.
__device__ __forceinline__ void cx_desc(unsigned long long &a, unsigned long long &b)
{
    const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
    a = hi;
    b = lo;
}

// Top-k of one token's E = 256 fp32 logits by one warp: lane l holds the
// logits of experts l + 32 m (m = 0..7).  Returns in lanes 0..TOPK-1 the
// selected expert (best first) and its renormalised sigmoid weight, and
// reports whether a logit was not finite.  Each lane first sorts its eight
// keys (a 19-comparator odd-even merge network); then every round two
// warp-wide max reductions (redux.sync, on the high then the low 32 bits of
// the lanes' best remaining keys) find the best remaining key, which is
// unique, and its owner drops it from the head of its list.
// SINK: lanes j < n_sink also hold the logit of expert sink j (a shared
// expert that joins the normalisation but is never selected; TML Inkling
// page, section "MoE"): its sigmoid is added to the denominator after the
// selected ones (sink order), and swt of lane j receives its weight.
template <bool SINK>
__device__ __forceinline__ void warp_route_values_t(const float v[8], int lane, int &ex, float &wt, bool &nonfinite,
                                                    float sink_v, int n_sink, float &swt)
{
    unsigned long long k[8];
    bool bad = false;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        bad |= !isfinite(v[m]);
        k[m] = rank_key(v[m], lane + 32 * m);
    }
    if (SINK && lane < n_sink)
        bad |= !isfinite(sink_v);
    nonfinite = __any_sync(0xFFFFFFFFu, bad);
    cx_desc(k[0], k[2]); cx_desc(k[1], k[3]); cx_desc(k[4], k[6]); cx_desc(k[5], k[7]);
    cx_desc(k[0], k[4]); cx_desc(k[1], k[5]); cx_desc(k[2], k[6]); cx_desc(k[3], k[7]);
    cx_desc(k[0], k[1]); cx_desc(k[2], k[3]); cx_desc(k[4], k[5]); cx_desc(k[6], k[7]);
    cx_desc(k[2], k[4]); cx_desc(k[3], k[5]);
    cx_desc(k[1], k[4]); cx_desc(k[3], k[6]);
    cx_desc(k[1], k[2]); cx_desc(k[3], k[4]); cx_desc(k[5], k[6]);
    // Round i: the largest high word (the logit) over the lanes' best keys;
    // when one lane holds it, that lane wins without a second reduction (a
    // tie on the logit takes the larger low word: the lower expert index).
    // The winners' keys reach lanes 0..5 after the rounds.
    unsigned long long chosen = 0ull;   // lane i < TOPK: the i-th best key
    int winner[TOPK];
    unsigned long long won[TOPK];       // on the winner lane of round i: its key
#pragma unroll
    for (int i = 0; i < TOPK; ++i) {
        const unsigned long long mine = k[0];
        const uint32_t mh = (uint32_t)(mine >> 32);
        const uint32_t hi = __reduce_max_sync(0xFFFFFFFFu, mh);
        uint32_t cand = __ballot_sync(0xFFFFFFFFu, mh == hi);
        if (cand & (cand - 1)) {
            const uint32_t lo = __reduce_max_sync(0xFFFFFFFFu, mh == hi ? (uint32_t)mine : 0u);
            cand = __ballot_sync(0xFFFFFFFFu, mh == hi && (uint32_t)mine == lo);
        }
        winner[i] = __ffs(cand) - 1;
        if (lane == winner[i]) {
            won[i] = mine;
#pragma unroll
            for (int m = 0; m < 7; ++m)
                k[m] = k[m + 1];
            k[7] = 0ull;
        }
    }
#pragma unroll
    for (int i = 0; i < TOPK; ++i) {
        const unsigned long long w = __shfl_sync(0xFFFFFFFFu, won[i], winner[i]);
        if (lane == i)
            chosen = w;
    }
    // sigmoid of each chosen logit on its own lane, the sum in selection order
    const float s = 1.0f / (1.0f + expf(-key_logit(chosen)));
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < TOPK; ++i)
        sum += __shfl_sync(0xFFFFFFFFu, s, i);
    float ss = 0.0f;
    if (SINK) {
        ss = lane < n_sink ? 1.0f / (1.0f + expf(-sink_v)) : 0.0f;
        for (int j = 0; j < n_sink; ++j)
            sum += __shfl_sync(0xFFFFFFFFu, ss, j);
    }
    ex = lane < TOPK ? key_expert(chosen) : 0;
    wt = lane < TOPK ? s / sum : 0.0f;
    swt = SINK && lane < n_sink ? ss / sum : 0.0f;
}

__device__ __forceinline__ void warp_route_values(const float v[8], int lane, int &ex, float &wt, bool &nonfinite)
{
    float unused;
    warp_route_values_t<false>(v, lane, ex, wt, nonfinite, 0.0f, 0, unused);
}

// The same, reading the token's logits row from global memory (L2).
__device__ __forceinline__ void warp_route_token(const float *logits_row, int lane, int &ex, float &wt,
                                                 bool &nonfinite)
{
    float v[8];
#pragma unroll
    for (int m = 0; m < 8; ++m)
        v[m] = __ldcg(logits_row + lane + 32 * m);
    warp_route_values(v, lane, ex, wt, nonfinite);
}

// Router partial sums of the 16 compute warps of a CTA (2 experts x 8 warps,
// each lane a sequential chain of 8 exact bf16 x bf16 products per token)
// reduced to logits through shared memory: 16 threads per (expert, token)
// add 16 partials each as a balanced tree, then one thread adds those 16 as
// a balanced tree.  Summation depth 7 + 4 + 4 = 15.
struct RouterRed {
    float p[2][MAXT][256];
    float q[2][MAXT][16];
};

__device__ __forceinline__ float tree16(const float *v)
{
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a[i] = v[2 * i] + v[2 * i + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = a[2 * i] + a[2 * i + 1];
    return (a[0] + a[1]) + (a[2] + a[3]);
}

// tid: 0..511 (warp w: expert w / 8, column slice w % 8).  Afterwards threads
// tid < 2 * MAXT with t = tid % MAXT < T return true with the logit of
// (expert e0 + tid / MAXT, token t) in *logit.
__device__ __forceinline__ bool router_reduce(const float acc[MAXT], int tid, int T, RouterRed &r, int bar_id,
                                              float *logit)
{
    const int e = tid >> 8, i = tid & 255;
#pragma unroll
    for (int t = 0; t < MAXT; ++t)
        if (t < T)
            r.p[e][t][i] = acc[t];
    asm volatile("bar.sync %0, 512;" ::"r"(bar_id) : "memory");
    if (tid < 2 * MAXT * 16) {
        const int ee = tid / (MAXT * 16), t = (tid / 16) % MAXT, g = tid % 16;
        if (t < T)
            r.q[ee][t][g] = tree16(&r.p[ee][t][16 * g]);
    }
    asm volatile("bar.sync %0, 512;" ::"r"(bar_id) : "memory");
    if (tid < 2 * MAXT) {
        const int ee = tid / MAXT, t = tid % MAXT;
        if (t < T) {
            *logit = tree16(r.q[ee][t]);
            return true;
        }
    }
    return false;
}

}  // namespace moe

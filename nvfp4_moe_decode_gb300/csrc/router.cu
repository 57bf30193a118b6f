// router.cu -- K1: router GEMV + sigmoid top-k + renormalise + expert union.
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "A 40B MoE that activates 2.5B parameters": 256 experts, sigmoid top-6
// routing plus a shared expert.  Section "From 1,096 kernels to 346": the
// routing is fused into the router GEMV, and every kernel uses programmatic
// dependent launch so that it loads its weights while its predecessor runs.
//
// Grid: E/2 CTAs of 256 threads.  CTA c computes the logits of experts 2c and
// 2c+1 for all T tokens: warps 0-3 take expert 2c, warps 4-7 expert 2c+1, one
// quarter of the hidden dimension each.  A lane multiplies 16 bf16 pairs
// (exact products in fp32) in k order, the warp adds its 32 lane sums by a
// 5-level butterfly, and warp 0/4 adds the four quarter sums in order: every
// logit is an fp32 sum of exact products of depth 16 + 5 + 3 = 24.
//
// The CTA that arrives last (arrival counter in the workspace) selects the
// top-k of each token on the fp32 logits (one warp per token), computes the
// renormalised sigmoid weights, and builds the slot table that the expert
// kernels read: the shared expert(s) first, then the distinct selected
// experts in ascending order, each with the routing weight of every token
// (0 where the token did not select it).
#include "kernels.cuh"
#include "topk.cuh"

namespace moe {

__global__ void __launch_bounds__(256) router_topk_kernel(RouterArgs a)
{
    const WsLayout L = ws_layout();
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(a.ws + L.ctrl);
    float *logits = reinterpret_cast<float *>(a.ws + L.logits);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 2 + (warp >> 2);
    const int kq = warp & 3;

    // Router weights do not depend on the preceding kernel: load them first.
    uint4 wv[2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
        wv[m] = ldg_nc_v4(a.wr + (size_t)e * H + 512 * kq + 256 * m + 8 * lane);

    griddep_wait();      // x may be written by the preceding kernel
    griddep_launch();    // the expert kernel may start its prologue now

    __shared__ float part[8][MAXT];
    __shared__ int is_last;

    // all tokens at once: the x loads are independent, so they are issued
    // together; each token keeps its own sequential chain of 16 products
    uint4 xv[MAXT][2];
#pragma unroll
    for (int t = 0; t < MAXT; ++t)
        if (t < a.T) {
#pragma unroll
            for (int m = 0; m < 2; ++m)
                xv[t][m] = ldg_nc_v4(a.x + (size_t)t * H + 512 * kq + 256 * m + 8 * lane);
        }
    float acc[MAXT];
#pragma unroll
    for (int t = 0; t < MAXT; ++t) {
        acc[t] = 0.0f;
        if (t < a.T) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const uint32_t xs[4] = {xv[t][m].x, xv[t][m].y, xv[t][m].z, xv[t][m].w};
                const uint32_t ws[4] = {wv[m].x, wv[m].y, wv[m].z, wv[m].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[t] = fmaf(bf16_bits_to_float(xs[q] & 0xFFFFu), bf16_bits_to_float(ws[q] & 0xFFFFu), acc[t]);
                    acc[t] = fmaf(bf16_bits_to_float(xs[q] >> 16), bf16_bits_to_float(ws[q] >> 16), acc[t]);
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
        for (int t = 0; t < MAXT; ++t)
            if (t < a.T)
                acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], off);
    if (lane == 0) {
#pragma unroll
        for (int t = 0; t < MAXT; ++t)
            if (t < a.T)
                part[warp][t] = acc[t];
    }
    __syncthreads();
    if ((warp & 3) == 0 && lane < a.T) {
        const int t = lane;
        float v = ((part[warp][t] + part[warp + 1][t]) + part[warp + 2][t]) + part[warp + 3][t];
        logits[t * E + e] = v;
        if (a.user_logits)
            a.user_logits[(size_t)t * E + e] = v;
        __threadfence();   // publish before this CTA's arrival is counted
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t prev = atomicAdd(&ctrl[1], 1u);
        is_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last)
        return;
    __threadfence();

    // ---- last CTA: top-k per token, weights, slot table ----
    __shared__ int32_t sel[MAXT][TOPK];
    __shared__ float selw[MAXT][TOPK];
    int32_t *topk_idx = reinterpret_cast<int32_t *>(a.ws + L.topk_idx);
    float *topk_w = reinterpret_cast<float *>(a.ws + L.topk_w);
    SlotTable *st = reinterpret_cast<SlotTable *>(a.ws + L.slots);

    if (warp < a.T) {
        const int t = warp;
        int ex;
        float wi;
        bool bad;
        warp_route_token(logits + t * E, lane, ex, wi, bad);
        if (bad && lane == 0)
            atomicOr(&ctrl[0], FLAG_NONFINITE);
        if (lane < TOPK) {
            sel[t][lane] = ex;
            selw[t][lane] = wi;
            topk_idx[t * TOPK + lane] = ex;
            topk_w[t * TOPK + lane] = wi;
            if (a.user_idx) a.user_idx[t * TOPK + lane] = ex;
            if (a.user_w) a.user_w[t * TOPK + lane] = wi;
        }
    }
    __syncthreads();

    // Slot table: shared expert(s), then the sorted union of selected experts.
    __shared__ uint32_t bitmap[E / 32];
    __shared__ int32_t prefix[E / 32];
    if (threadIdx.x < E / 32)
        bitmap[threadIdx.x] = 0u;
    __syncthreads();
    if (threadIdx.x < a.T * TOPK) {
        const int ei = sel[threadIdx.x / TOPK][threadIdx.x % TOPK];
        atomicOr(&bitmap[ei >> 5], 1u << (ei & 31));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int i = 0; i < E / 32; ++i) {
            prefix[i] = run;
            run += __popc(bitmap[i]);
        }
        st->n_shared = a.n_shared;
        st->n_slots = a.n_shared + run;
    }
    __syncthreads();
    // expert ids of the routed slots
    if (threadIdx.x < E) {
        const int ei = threadIdx.x;
        const uint32_t bits = bitmap[ei >> 5];
        if (bits & (1u << (ei & 31))) {
            const int slot = a.n_shared + prefix[ei >> 5] + __popc(bits & ((1u << (ei & 31)) - 1u));
            st->expert[slot] = ei;
        }
    }
    // per-slot token weights: clear every slot, then fill
    for (int i = threadIdx.x; i < MAX_SLOTS * MAXT; i += blockDim.x)
        st->wts[i / MAXT][i % MAXT] = 0.0f;
    if (threadIdx.x < a.n_shared)
        st->expert[threadIdx.x] = -1 - (int)threadIdx.x;
    __syncthreads();
    if (threadIdx.x < a.n_shared * MAXT) {
        const int s = threadIdx.x / MAXT, t = threadIdx.x % MAXT;
        st->wts[s][t] = (t < a.T) ? 1.0f : 0.0f;
    }
    if (threadIdx.x < a.T * TOPK) {
        const int t = threadIdx.x / TOPK, i = threadIdx.x % TOPK;
        const int ei = sel[t][i];
        const uint32_t bits = bitmap[ei >> 5];
        const int slot = a.n_shared + prefix[ei >> 5] + __popc(bits & ((1u << (ei & 31)) - 1u));
        st->wts[slot][t] = selw[t][i];
    }
    if (threadIdx.x == 0)
        ctrl[1] = 0u;   // re-arm the arrival counter for the next call
}

cudaError_t launch_router(const RouterArgs &a, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(E / 2);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, router_topk_kernel, a);
}

}  // namespace moe

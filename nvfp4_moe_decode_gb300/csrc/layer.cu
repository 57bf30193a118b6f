// layer.cu -- the small-batch NVFP4 MoE layer as one persistent kernel.
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "A 40B MoE that activates 2.5B parameters": 256 routed experts with sigmoid
// top-6 routing plus one shared expert, NVFP4 weights run weight-only with
// BF16 activations.  Section "From 1,096 kernels to 346": router and expert
// GEMVs that read only the selected experts' weights, routing and the expert
// combine fused into the GEMV kernels, programmatic dependent launch so that
// a kernel loads weights while its predecessor finishes.
//
// One CTA per SM, 16 warps in 4 groups of 4.  Phases:
//  1. before waiting on the preceding kernel: router CTAs load their slice of
//     the router weights; group 0 of the first 64 CTAs starts the bulk copies
//     of one band of the shared expert (it needs no routing);
//  2. router: CTAs 0..127 (warps 8..15) compute the fp32 logits of two experts
//     each and publish them; warps 0..7 turn x into f16 mma fragments;
//  3. every CTA waits for all logits, takes the top-6 of each token (one warp
//     per token, identical in every CTA) and builds the slot table: the shared
//     expert, then the distinct selected experts in ascending order, each with
//     its per-token routing weight;
//  4. a work queue (one atomic counter) hands each group units:
//       gate/up unit (slot, band):  the 4 warps take one K quarter each of a
//         16-row band of W13 (8 gate + 8 up rows); SiLU*up -> h (bf16) with a
//         per-(slot, token) running max of |h|;
//       down unit (slot, 4 bands):  waits until the slot's 64 gate/up bands are
//         done, loads the slot's h, rescales it to f16 fragments, and each warp
//         computes one 16-row band of W2 h, times the routing weight;
//     gate/up units come first in the queue, so a down unit only ever waits
//     on units that running warps already hold;
//  5. the last down partial of each band adds all partials in slot order
//     (deterministic) and writes out (bf16).
// Every warp streams its units' weights through a private 3-stage ring of
// shared-memory buffers filled by cp.async.bulk; waits are bounded and report
// MOE_FLAG_WAIT_TIMEOUT instead of hanging.
#include "kernels.cuh"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int FW = 16;                 // warps per CTA
constexpr int FT = FW * 32;            // threads per CTA
constexpr int NG = 4;                  // unit groups per CTA
constexpr int GW = 4;                  // warps per group
constexpr int RING = 3;                // stages per warp
constexpr int STG = 2 * SC_BYTES;      // 2304 bytes: two super-chunks
constexpr int ROUTER_CTAS = E / 2;     // 128 CTAs x 2 experts
constexpr int UNITS_AHEAD = 3;         // unit-id ring per group
constexpr int H_BYTES = MAXT * I * 2;  // one slot's h (bf16), 8 KB at T = 8

struct FSmem {
    uint8_t ring[FW][RING][STG];
    uint2 xfrag[(H / 16) * 32];        // compact: entry (step, l) at step * 4T + l
    uint8_t hbuf[NG][2][H_BYTES];      // raw h, rescaled in place into fragments
    float4 red[2][NG][GW - 1][32];     // gate/up K-part partials (double-buffered)
    uint64_t full[FW][RING];
    uint64_t hbar[NG][2];
    int unit[NG][UNITS_AHEAD];
    int hissued[NG][2];
    float rpart[8][MAXT];
    int32_t sel[MAXT][TOPK];
    float selw[MAXT][TOPK];
    uint32_t bitmap[E / 32];
    int32_t prefix[E / 32];
    int n_slots;
    int32_t slot_expert[MAX_SLOTS];
    float wts[MAX_SLOTS][MAXT];
    int xshift[MAXT];
    int route_ok;
};

__device__ __forceinline__ float pow2i(int k) { return __int_as_float((127 + k) << 23); }

__device__ __forceinline__ int act_shift(float maxabs)
{
    int sh = ACT_EXP - exponent_of(maxabs);
    return sh < -100 ? -100 : (sh > 100 ? 100 : sh);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded spin until *p >= target.  Returns false (and flags) on timeout.
__device__ __forceinline__ bool spin_until(const uint32_t *p, uint32_t target, uint32_t *flag)
{
    for (uint32_t it = 0; it < SPIN_LIMIT; ++it) {
        if (ld_acquire(p) >= target)
            return true;
        __nanosleep(64);
    }
    atomicOr(flag, FLAG_TIMEOUT);
    return false;
}

__device__ __forceinline__ void ffma2(float &a0, float &a1, float s, float d0, float d1)
{
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %2};\n\tmov.b64 y, {%3, %4};\n\t"
        "mov.b64 z, {%0, %1};\n\tfma.rn.f32x2 z, x, y, z;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "+f"(a0), "+f"(a1) : "f"(s), "f"(d0), "f"(d1));
}

__device__ __forceinline__ void decode4(uint32_t w, uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(w));
}

// Two consecutive super-chunks of one band (one stage) times the B fragments
// from k16 step `step0`; blanes = 4T lanes carry tokens.
__device__ __forceinline__ void mma_stage(const uint8_t *stage, const uint2 *bfrag, int blanes, int step0,
                                          int lane, float acc[4])
{
    const int g = lane >> 2;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint8_t *base = stage + q * SC_BYTES;
        const uint4 sc = *reinterpret_cast<const uint4 *>(base + 1024 + g * 16);
        const uint32_t sws[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint4 cw = *reinterpret_cast<const uint4 *>(base + half * 512 + lane * 16);
            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int step = step0 + q * 8 + half * 4 + s;
                const uint2 b = (lane < blanes) ? bfrag[step * blanes + lane] : make_uint2(0u, 0u);
                uint32_t a0, a1, a2, a3;
                decode4(words[s], a0, a1, a2, a3);
                float d[4];
                mma_f16_16816(d, a0, a1, a2, a3, b.x, b.y);
                const int sb = half * 4 + s;
                const uint32_t sw = sws[sb >> 1];
                const float2 sf = e4m3x2_to_float2((sb & 1) ? (sw >> 16) : (sw & 0xFFFFu));
                ffma2(acc[0], acc[1], sf.x, d[0], d[1]);
                ffma2(acc[2], acc[3], sf.y, d[2], d[3]);
            }
        }
    }
}

struct Unit {
    bool down;   // down unit (else gate/up)
    int slot;
    int idx;     // band (gate/up) or band group (down)
};

}  // namespace

__global__ void __launch_bounds__(FT, 1) moe_layer_kernel(LayerArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    FSmem &sm = *reinterpret_cast<FSmem *>(smem_raw);

    const WsLayout L = ws_layout();
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(a.ws + L.ctrl);
    uint32_t *flag = ctrl;
    uint32_t *slot_cnt = reinterpret_cast<uint32_t *>(a.ws + L.slot_cnt);
    uint32_t *hmax = reinterpret_cast<uint32_t *>(a.ws + L.hmax);
    uint32_t *band_cnt = reinterpret_cast<uint32_t *>(a.ws + L.band_cnt);
    float *logits = reinterpret_cast<float *>(a.ws + L.logits);
    __nv_bfloat16 *hglob = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.h);
    float *partials = reinterpret_cast<float *>(a.ws + L.partials);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = warp / GW, wq = warp % GW;
    const bool leader = (wq == 0);
    const int T = a.T;
    const int blanes = 4 * T;

    if (lane == 0) {
        for (int s = 0; s < RING; ++s)
            mbar_init(&sm.full[warp][s], 1);
        if (leader) {
            mbar_init(&sm.hbar[grp][0], 1);
            mbar_init(&sm.hbar[grp][1], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // ---- unit decoding (valid once the slot table is known, or for the
    // shared expert, whose slot 0 needs no routing) ----
    auto w13_src = [&](int slot, int band) -> const uint8_t * {
        const uint8_t *base = (slot < a.n_shared) ? a.s_w13 + (size_t)slot * W13_BYTES
                                                  : a.r_w13 + (size_t)sm.slot_expert[slot] * W13_BYTES;
        return base + (size_t)band * W13_BAND_BYTES;
    };
    auto w2_src = [&](int slot, int band) -> const uint8_t * {
        const uint8_t *base = (slot < a.n_shared) ? a.s_w2 + (size_t)slot * W2_BYTES
                                                  : a.r_w2 + (size_t)sm.slot_expert[slot] * W2_BYTES;
        return base + (size_t)band * W2_BAND_BYTES;
    };
    // stage i of this warp's stream: unit i/2, part i%2
    auto issue_stage = [&](int i, const Unit &u) {
        if (lane != 0)
            return;
        const uint8_t *src;
        if (!u.down)
            src = w13_src(u.slot, u.idx) + (size_t)(4 * wq + 2 * (i & 1)) * SC_BYTES;
        else
            src = w2_src(u.slot, 4 * u.idx + wq) + (size_t)(2 * (i & 1)) * SC_BYTES;
        uint64_t *bar = &sm.full[warp][i % RING];
        mbar_arrive_expect_tx(bar, STG);
        bulk_g2s(sm.ring[warp][i % RING], src, STG, bar);
    };

    // ---- phase 1: work that needs nothing from the preceding kernel ----
    const bool static_shared = (a.n_shared > 0) && grp == 0 && blockIdx.x < W13_BANDS;
    if (static_shared) {
        const Unit u0{false, 0, (int)blockIdx.x};
        issue_stage(0, u0);
        issue_stage(1, u0);
    }
    const bool router_warp = blockIdx.x < ROUTER_CTAS && warp >= 8;
    const int r_e = blockIdx.x * 2 + ((warp - 8) >> 2);
    const int r_kq = (warp - 8) & 3;
    uint4 wv[2];
    if (router_warp) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
            wv[m] = ldg_nc_v4(a.wr + (size_t)r_e * H + 512 * r_kq + 256 * m + 8 * lane);
    }

    griddep_wait();      // x is written by the preceding kernel
    griddep_launch();    // the next kernel may start its own phase 1

    // ---- phase 2: router logits (warps 8..15) | activation fragments (0..7) ----
    if (router_warp) {
        uint4 xv[MAXT][2];
#pragma unroll
        for (int t = 0; t < MAXT; ++t)
            if (t < T) {
#pragma unroll
                for (int m = 0; m < 2; ++m)
                    xv[t][m] = ldg_nc_v4(a.x + (size_t)t * H + 512 * r_kq + 256 * m + 8 * lane);
            }
        float acc[MAXT];
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
            acc[t] = 0.0f;
            if (t < T) {
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
                if (t < T)
                    acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], off);
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < MAXT; ++t)
                if (t < T)
                    sm.rpart[warp - 8][t] = acc[t];
        }
        named_barrier_sync(5, 256);
        if ((warp == 8 || warp == 12) && lane < T) {
            const int t = lane, w0 = warp - 8;
            const float v = ((sm.rpart[w0][t] + sm.rpart[w0 + 1][t]) + sm.rpart[w0 + 2][t]) + sm.rpart[w0 + 3][t];
            logits[t * E + r_e] = v;
            __threadfence();
        }
        named_barrier_sync(5, 256);
        if (warp == 8 && lane == 0)
            atomicAdd(&ctrl[2], 1u);   // after the fence above: the logits are published
    } else if (warp < 8) {
        if (warp < T) {
            const uint4 *row = reinterpret_cast<const uint4 *>(a.x + (size_t)warp * H);
            float m = 0.f;
#pragma unroll
            for (int i = 0; i < H / 256; ++i) {
                const uint4 v = __ldg(row + lane + 32 * i);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[q] << 16)), fabsf(__uint_as_float(w4[q] & 0xFFFF0000u))));
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
            if (lane == 0)
                sm.xshift[warp] = act_shift(m);
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < (H / 16) * blanes; idx += FT) {
        const int step = idx / blanes, l = idx % blanes, g = l >> 2, c = l & 3;
        const float p = pow2i(sm.xshift[g]);
        const uint32_t *xr = reinterpret_cast<const uint32_t *>(a.x + (size_t)g * H + 16 * step);
        uint2 v;
        v.x = bf16x2_to_f16x2_scaled(__ldg(xr + c), p);
        v.y = bf16x2_to_f16x2_scaled(__ldg(xr + 4 + c), p);
        sm.xfrag[idx] = v;
    }

    // ---- phase 3: routing (every CTA, identically) ----
    if (threadIdx.x == 0)
        sm.route_ok = spin_until(&ctrl[2], (uint32_t)ROUTER_CTAS, flag) ? 1 : 0;
    __syncthreads();
    if (warp < T) {
        int ex;
        float wt;
        bool bad;
        warp_route_token(logits + warp * E, lane, ex, wt, bad);
        if (lane < TOPK) {
            sm.sel[warp][lane] = ex;
            sm.selw[warp][lane] = wt;
        }
        if (blockIdx.x == 0) {
            if (bad && lane == 0)
                atomicOr(flag, FLAG_NONFINITE);
            if (lane < TOPK) {
                reinterpret_cast<int32_t *>(a.ws + L.topk_idx)[warp * TOPK + lane] = ex;
                reinterpret_cast<float *>(a.ws + L.topk_w)[warp * TOPK + lane] = wt;
            }
        }
    }
    if (threadIdx.x < E / 32)
        sm.bitmap[threadIdx.x] = 0u;
    for (int i = threadIdx.x; i < MAX_SLOTS * MAXT; i += FT)
        sm.wts[i / MAXT][i % MAXT] = 0.0f;
    __syncthreads();
    if (threadIdx.x < T * TOPK) {
        const int ei = sm.sel[threadIdx.x / TOPK][threadIdx.x % TOPK];
        atomicOr(&sm.bitmap[ei >> 5], 1u << (ei & 31));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int i = 0; i < E / 32; ++i) {
            sm.prefix[i] = run;
            run += __popc(sm.bitmap[i]);
        }
        sm.n_slots = a.n_shared + run;
    }
    __syncthreads();
    if (threadIdx.x < E) {
        const int ei = threadIdx.x;
        const uint32_t bits = sm.bitmap[ei >> 5];
        if (bits & (1u << (ei & 31)))
            sm.slot_expert[a.n_shared + sm.prefix[ei >> 5] + __popc(bits & ((1u << (ei & 31)) - 1u))] = ei;
    }
    if (threadIdx.x < a.n_shared) {
        sm.slot_expert[threadIdx.x] = -1 - (int)threadIdx.x;
        for (int t = 0; t < T; ++t)
            sm.wts[threadIdx.x][t] = 1.0f;
    }
    __syncthreads();
    if (threadIdx.x < T * TOPK) {
        const int t = threadIdx.x / TOPK, i = threadIdx.x % TOPK;
        const int ei = sm.sel[t][i];
        const uint32_t bits = sm.bitmap[ei >> 5];
        sm.wts[a.n_shared + sm.prefix[ei >> 5] + __popc(bits & ((1u << (ei & 31)) - 1u))][t] = sm.selw[t][i];
    }
    __syncthreads();
    const int n_slots = sm.n_slots;
    if (blockIdx.x == 0) {
        SlotTable *st = reinterpret_cast<SlotTable *>(a.ws + L.slots);
        if (threadIdx.x == 0) {
            st->n_slots = n_slots;
            st->n_shared = a.n_shared;
        }
        if (threadIdx.x < MAX_SLOTS)
            st->expert[threadIdx.x] = threadIdx.x < n_slots ? sm.slot_expert[threadIdx.x] : 0;
        for (int i = threadIdx.x; i < MAX_SLOTS * MAXT; i += FT)
            st->wts[i / MAXT][i % MAXT] = sm.wts[i / MAXT][i % MAXT];
    }

    // ---- phase 4: the unit queue ----
    const int n_routed_slots = n_slots - a.n_shared;
    const int gu_total = n_slots * W13_BANDS;                       // unit ids [0, gu_total): gate/up
    const int q_gu = n_routed_slots * W13_BANDS;                    // routed gate/up units in the queue
    const int q_total = q_gu + n_slots * (W2_BANDS / GW);           // + down units
    const int end_id = gu_total + n_slots * (W2_BANDS / GW);
    auto fetch = [&]() -> int {
        const uint32_t q = atomicAdd(&ctrl[3], 1u);
        if ((int)q < q_gu)
            return a.n_shared * W13_BANDS + (int)q;
        if ((int)q < q_total)
            return gu_total + ((int)q - q_gu);
        return end_id;
    };
    auto decode = [&](int id) -> Unit {
        if (id < gu_total)
            return Unit{false, id / W13_BANDS, id % W13_BANDS};
        const int d = id - gu_total;
        return Unit{true, d / (W2_BANDS / GW), d % (W2_BANDS / GW)};
    };
    // h of a down unit: raw bf16 [T][I] of the slot into hbuf[grp][b]
    auto issue_h = [&](int slot, int b) {
        uint64_t *bar = &sm.hbar[grp][b];
        const uint32_t bytes = (uint32_t)(T * I * 2);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(sm.hbuf[grp][b], hglob + (size_t)slot * MAXT * I, bytes, bar);
    };
    auto slot_ready = [&](int slot) { return ld_acquire(&slot_cnt[slot]) >= (uint32_t)W13_BANDS; };

    if (leader && lane == 0) {
        sm.unit[grp][0] = static_shared ? (int)blockIdx.x : fetch();
        sm.unit[grp][1] = fetch();
        sm.unit[grp][2] = fetch();
        sm.hissued[grp][0] = sm.hissued[grp][1] = 0;
        for (int k = 0; k < 2; ++k) {
            const int id = sm.unit[grp][k];
            if (id < end_id) {
                const Unit u = decode(id);
                if (u.down && slot_ready(u.slot)) {
                    issue_h(u.slot, k);
                    sm.hissued[grp][k] = 1;
                }
            }
        }
    }
    named_barrier_sync(1 + grp, GW * 32);
    {
        const int id0 = sm.unit[grp][0];
        if (!static_shared && id0 < end_id) {
            issue_stage(0, decode(id0));
            issue_stage(1, decode(id0));
        }
    }

    int hcnt[2] = {0, 0};
    float acc[4];
    for (int k = 0;; ++k) {
        const int id = sm.unit[grp][k % UNITS_AHEAD];
        if (id >= end_id)
            break;
        const Unit u = decode(id);
        const int id_next = sm.unit[grp][(k + 1) % UNITS_AHEAD];
        const bool has_next = id_next < end_id;
        const Unit un = has_next ? decode(id_next) : Unit{false, 0, 0};
        if (has_next)
            issue_stage(2 * k + 2, un);

        const uint2 *bfrag = sm.xfrag;
        int step0 = 32 * wq;   // gate/up: this warp's K quarter
        if (u.down) {
            const int b = k & 1;
            if (leader && lane == 0 && !sm.hissued[grp][b]) {
                spin_until(&slot_cnt[u.slot], (uint32_t)W13_BANDS, flag);
                issue_h(u.slot, b);
                sm.hissued[grp][b] = 1;
            }
            mbar_wait_bounded(&sm.hbar[grp][b], hcnt[b] & 1, flag);
            hcnt[b]++;
            // rescale h (bf16 [T][I]) in place into f16 fragments [step][4T]
            uint32_t *hb = reinterpret_cast<uint32_t *>(sm.hbuf[grp][b]);
            const int nent = (I / 16) * blanes;            // <= 1024
            uint32_t src[2][8];
            int shv[MAXT];
#pragma unroll
            for (int t = 0; t < MAXT; ++t)
                shv[t] = (t < T) ? act_shift(__uint_as_float(__ldcg(&hmax[u.slot * MAXT + t]))) : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = (wq * 32 + lane) + j * (GW * 32);
                src[0][j] = src[1][j] = 0u;
                if (e < nent) {
                    const int step = e / blanes, l = e % blanes, g = l >> 2, c = l & 3;
                    src[0][j] = hb[(g * I + 16 * step) / 2 + c];
                    src[1][j] = hb[(g * I + 16 * step + 8) / 2 + c];
                }
            }
            named_barrier_sync(1 + grp, GW * 32);
            uint2 *hf = reinterpret_cast<uint2 *>(sm.hbuf[grp][b]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = (wq * 32 + lane) + j * (GW * 32);
                if (e < nent) {
                    const int g = (e % blanes) >> 2;
                    int sh = 0;
#pragma unroll
                    for (int t = 0; t < MAXT; ++t)
                        if (t == g) sh = shv[t];
                    const float p = pow2i(sh);
                    hf[e] = make_uint2(bf16x2_to_f16x2_scaled(src[0][j], p), bf16x2_to_f16x2_scaled(src[1][j], p));
                }
            }
            named_barrier_sync(1 + grp, GW * 32);
            bfrag = hf;
            step0 = 0;
        }

        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        // stage 2k
        mbar_wait_bounded(&sm.full[warp][(2 * k) % RING], ((2 * k) / RING) & 1, flag);
        mma_stage(sm.ring[warp][(2 * k) % RING], bfrag, blanes, step0, lane, acc);
        __syncwarp();
        if (has_next)
            issue_stage(2 * k + 3, un);
        // stage 2k + 1
        mbar_wait_bounded(&sm.full[warp][(2 * k + 1) % RING], ((2 * k + 1) / RING) & 1, flag);
        mma_stage(sm.ring[warp][(2 * k + 1) % RING], bfrag, blanes, step0 + 16, lane, acc);
        __syncwarp();

        const int g = lane >> 2, c = lane & 3;
        if (!u.down) {
            // K parts -> warp 0 of the group; SiLU*up; h; running max of |h|
            if (wq != 0)
                sm.red[k & 1][grp][wq - 1][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            named_barrier_sync(1 + grp, GW * 32);
            if (wq == 0) {
#pragma unroll
                for (int j = 0; j < GW - 1; ++j) {
                    const float4 r = sm.red[k & 1][grp][j][lane];
                    acc[0] += r.x; acc[1] += r.y; acc[2] += r.z; acc[3] += r.w;
                }
                const float ts = (u.slot < a.n_shared) ? __ldg(a.s_ts13 + u.slot)
                                                       : __ldg(a.r_ts13 + sm.slot_expert[u.slot]);
                float hm[2];
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int t = 2 * c + tt;
                    hm[tt] = 0.f;
                    if (t < T) {
                        const float f = ts * pow2i(-sm.xshift[t]);
                        const float gv = acc[tt] * f, uv = acc[2 + tt] * f;
                        const __nv_bfloat16 hv = __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
                        hglob[((size_t)u.slot * MAXT + t) * I + u.idx * 8 + g] = hv;
                        hm[tt] = fabsf(__bfloat162float(hv));
                    }
                }
#pragma unroll
                for (int off = 4; off <= 16; off <<= 1) {
                    hm[0] = fmaxf(hm[0], __shfl_xor_sync(0xFFFFFFFFu, hm[0], off));
                    hm[1] = fmaxf(hm[1], __shfl_xor_sync(0xFFFFFFFFu, hm[1], off));
                }
                if (g == 0) {
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt)
                        if (2 * c + tt < T)
                            atomicMax(&hmax[u.slot * MAXT + 2 * c + tt], __float_as_uint(hm[tt]));
                }
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    atomicAdd(&slot_cnt[u.slot], 1u);
            }
        } else {
            // down: one band per warp, x routing weight x tensor scale x 2^-shift
            const int band = 4 * u.idx + wq;
            const float ts = (u.slot < a.n_shared) ? __ldg(a.s_ts2 + u.slot)
                                                   : __ldg(a.r_ts2 + sm.slot_expert[u.slot]);
            float *P = partials + ((size_t)u.slot * H + 16 * band) * MAXT;
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
                const int t = 2 * c + tt;
                if (t < T) {
                    const int sh = act_shift(__uint_as_float(__ldcg(&hmax[u.slot * MAXT + t])));
                    const float f = sm.wts[u.slot][t] * ts * pow2i(-sh);
                    P[g * MAXT + t] = acc[tt] * f;
                    P[(g + 8) * MAXT + t] = acc[2 + tt] * f;
                }
            }
            __threadfence();
            __syncwarp();
            uint32_t prev = 0;
            if (lane == 0)
                prev = atomicAdd(&band_cnt[band], 1u);
            prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
            if (prev == (uint32_t)(n_slots - 1)) {
                // last partial of this band: add all slots in slot order
                __threadfence();
                const int r = lane >> 1, th = lane & 1;      // row r, tokens 4*th .. 4*th+3
                const float4 *src = reinterpret_cast<const float4 *>(partials + ((size_t)16 * band + r) * MAXT) + th;
                float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
                constexpr int BATCH = 16;
                for (int s0 = 0; s0 < n_slots; s0 += BATCH) {
                    float4 v[BATCH];
#pragma unroll
                    for (int j = 0; j < BATCH; ++j)
                        v[j] = (s0 + j < n_slots) ? __ldcg(src + (size_t)(s0 + j) * H * MAXT / 4)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < BATCH; ++j) {
                        s4.x += v[j].x; s4.y += v[j].y; s4.z += v[j].z; s4.w += v[j].w;
                    }
                }
                const float vals[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = 4 * th + j;
                    if (t < T)
                        a.out[(size_t)t * H + 16 * band + r] = __float2bfloat16_rn(vals[j]);
                }
                if (lane == 0)
                    band_cnt[band] = 0u;
            }
        }

        // end of unit: the group's red / hbuf / unit slot are free
        named_barrier_sync(1 + grp, GW * 32);
        if (leader && lane == 0) {
            sm.unit[grp][k % UNITS_AHEAD] = fetch();     // unit k + 3
            const int b = k & 1;                          // h buffer of unit k + 2
            sm.hissued[grp][b] = 0;
            const int id2 = sm.unit[grp][(k + 2) % UNITS_AHEAD];
            if (id2 < end_id) {
                const Unit u2 = decode(id2);
                if (u2.down && slot_ready(u2.slot)) {
                    issue_h(u2.slot, b);
                    sm.hissued[grp][b] = 1;
                }
            }
        }
        named_barrier_sync(1 + grp, GW * 32);
    }

    // ---- the last CTA to finish re-arms the counters for the next call ----
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&ctrl[4], 1u);
        if (prev == gridDim.x - 1) {
            __threadfence();
            ctrl[2] = 0u;
            ctrl[3] = 0u;
            for (int s = 0; s < MAX_SLOTS; ++s)
                slot_cnt[s] = 0u;
            for (int i = 0; i < MAX_SLOTS * MAXT; ++i)
                hmax[i] = 0u;
            __threadfence();
            ctrl[4] = 0u;
        }
    }
}

size_t layer_smem_bytes() { return sizeof(FSmem); }

cudaError_t launch_layer(const LayerArgs &a, int grid, cudaStream_t stream, bool pdl)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(moe_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(FSmem));
        if (e != cudaSuccess)
            return e;
        configured[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(FT);
    cfg.dynamicSmemBytes = sizeof(FSmem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_layer_kernel, a);
}

}  // namespace moe

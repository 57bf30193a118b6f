// expert.cu -- the expert kernels of the small-batch NVFP4 MoE layer:
//   K2 gate/up GEMV fused with SiLU*up,
//   K3 down GEMV fused with the routing weights,
//   K4 the deterministic combine of the per-expert down outputs.
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "From 1,096 kernels to 346": small-batch MoE kernels whose expert GEMVs read
// only the selected experts' weights, the expert combine fused into the
// neighbouring kernels, and programmatic dependent launch so that each kernel
// loads its weights while the previous one still runs.  Section "A 40B MoE
// that activates 2.5B parameters": NVFP4 weights, BF16 activations (W4A16).
//
// Every warp owns a stream of work units and a private ring of shared-memory
// stages filled by bulk async copies (cp.async.bulk + mbarrier): no
// cross-warp handshake sits on the streaming path.  A warp decodes e2m1
// bytes to f16 in registers (cvt.rn.f16x2.e2m1x2), runs mma.m16n8k16 with the
// (up to 8) tokens as the N dimension, and applies each k16 step's e4m3 block
// scale to the fp32 partial.  The packed layout is described in common.cuh.
#include "kernels.cuh"

namespace moe {

// Accumulate `nsc` consecutive super-chunks of one band (at sc_ptr in shared
// memory) times the B fragments starting at k16 step `step0`.
// B fragments are stored compactly: entry (step, lane) at step * blanes + lane
// for the lanes l < blanes = 4 * T that carry tokens; other lanes use zeros.
__device__ __forceinline__ void mma_superchunks(const uint8_t *sc_ptr, int nsc, const uint2 *bfrag,
                                                int blanes, int step0, int lane, float acc[4])
{
    const int g = lane >> 2;
    for (int q = 0; q < nsc; ++q) {
        const uint8_t *base = sc_ptr + q * SC_BYTES;
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
                float d[4];
                mma_f16_16816(d, decode_reg(words[s], 0), decode_reg(words[s], 1),
                              decode_reg(words[s], 2), decode_reg(words[s], 3), b.x, b.y);
                const int sb = half * 4 + s;
                const uint32_t sw = sws[sb >> 1];
                const float2 sf = e4m3x2_to_float2((sb & 1) ? (sw >> 16) : (sw & 0xFFFFu));
                acc[0] = fmaf(sf.x, d[0], acc[0]);
                acc[1] = fmaf(sf.x, d[1], acc[1]);
                acc[2] = fmaf(sf.y, d[2], acc[2]);
                acc[3] = fmaf(sf.y, d[3], acc[3]);
            }
        }
    }
}

// 2^k for |k| <= 126 (a normal float).
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((127 + k) << 23); }

// Shift that brings a token's largest magnitude into [2^ACT_EXP, 2^(ACT_EXP+1)),
// clamped so that both 2^shift and 2^-shift stay normal floats.
__device__ __forceinline__ int act_shift(float maxabs)
{
    int sh = ACT_EXP - exponent_of(maxabs);
    return sh < -100 ? -100 : (sh > 100 ? 100 : sh);
}

// ---------------------------------------------------------------------------
// K2: gate/up + SiLU*up
// ---------------------------------------------------------------------------
struct GuSmem {
    uint8_t ring[GU_WARPS][GU_RING][GU_STAGE_BYTES];
    uint2 xfrag[GU_STEPS * 32];
    float4 red[GU_WARPS][32];
    uint64_t full[GU_WARPS][GU_RING];
    int xshift[MAXT];
    int32_t c_expert[GU_WARPS][MAX_SLOTS];
    float c_ts[GU_WARPS][MAX_SLOTS];
};

__device__ __forceinline__ const uint8_t *gu_band_src(const GateUpArgs &a, const GuSmem &sm, int warp,
                                                      int slot, int band)
{
    const uint8_t *base = (slot < a.n_shared) ? a.shared_w13 + (size_t)slot * W13_BYTES
                                              : a.routed_w13 + (size_t)sm.c_expert[warp][slot] * W13_BYTES;
    return base + (size_t)band * W13_BAND_BYTES;
}

// One warp turns the finished h of a slot into f16 mma B fragments with a
// per-token power-of-two exponent (read by the down kernel).
__device__ void convert_slot(const GateUpArgs &a, int slot, int lane, const __nv_bfloat16 *hbuf,
                             uint2 *hfrag, int32_t *hexp)
{
    int sh_t[MAXT];
#pragma unroll
    for (int t = 0; t < MAXT; ++t) {
        sh_t[t] = 0;
        if (t < a.T) {
            const uint32_t *row = reinterpret_cast<const uint32_t *>(hbuf + ((size_t)slot * MAXT + t) * I);
            float m = 0.f;
#pragma unroll
            for (int i = 0; i < I / 64; ++i) {
                const uint32_t v = __ldcg(row + lane + 32 * i);
                m = fmaxf(m, fmaxf(fabsf(__uint_as_float(v << 16)), fabsf(__uint_as_float(v & 0xFFFF0000u))));
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
            sh_t[t] = act_shift(m);
            if (lane == 0)
                hexp[slot * MAXT + t] = sh_t[t];
        }
    }
    const int blanes = 4 * a.T;
    uint2 *dst = hfrag + (size_t)slot * (I / 16) * 32;
    for (int idx = lane; idx < (I / 16) * blanes; idx += 32) {
        const int step = idx / blanes, l = idx % blanes, g = l >> 2, c = l & 3;
        uint2 v;
        {
            int sh = 0;
#pragma unroll
            for (int t = 0; t < MAXT; ++t)
                if (t == g) sh = sh_t[t];
            const float p = pow2i(sh);
            const uint32_t *hr = reinterpret_cast<const uint32_t *>(hbuf + ((size_t)slot * MAXT + g) * I + 16 * step);
            v.x = bf16x2_to_f16x2_scaled(__ldcg(hr + c), p);
            v.y = bf16x2_to_f16x2_scaled(__ldcg(hr + 4 + c), p);
        }
        dst[idx] = v;
    }
}

__global__ void __launch_bounds__(GU_WARPS * 32, 1) gate_up_kernel(GateUpArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    GuSmem &sm = *reinterpret_cast<GuSmem *>(smem_raw);

    const WsLayout L = ws_layout();
    uint32_t *flag = reinterpret_cast<uint32_t *>(a.ws + L.ctrl);
    uint32_t *slot_cnt = reinterpret_cast<uint32_t *>(a.ws + L.slot_cnt);
    const SlotTable *st = reinterpret_cast<const SlotTable *>(a.ws + L.slots);
    __nv_bfloat16 *hbuf = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.h);
    uint2 *hfrag = reinterpret_cast<uint2 *>(a.ws + L.hfrag);
    int32_t *hexp = reinterpret_cast<int32_t *>(a.ws + L.hexp);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        for (int s = 0; s < GU_RING; ++s)
            mbar_init(&sm.full[warp][s], 1);
        fence_barrier_init();
    }
    // Activations -> f16 B fragments.  x is complete before this grid starts:
    // the router kernel triggers this launch after its own wait on the
    // kernel that produced x.
    if (warp < a.T) {
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
    __syncthreads();
    const int blanes = 4 * a.T;
    for (int idx = threadIdx.x; idx < GU_STEPS * blanes; idx += GU_WARPS * 32) {
        const int step = idx / blanes, l = idx % blanes, g = l >> 2, c = l & 3;
        uint2 v;
        {
            const float p = pow2i(sm.xshift[g]);
            const uint32_t *xr = reinterpret_cast<const uint32_t *>(a.x + (size_t)g * H + 16 * step);
            v.x = bf16x2_to_f16x2_scaled(__ldg(xr + c), p);
            v.y = bf16x2_to_f16x2_scaled(__ldg(xr + 4 + c), p);
        }
        sm.xfrag[idx] = v;
    }
    __syncthreads();

    // ---- this warp's work: units (slot, band), K split KS ways ----
    const int KS = a.KS;
    const int gpc = GU_WARPS / KS;                 // groups per CTA
    const int grp = warp / KS, kpart = warp % KS;
    const int n_groups = gridDim.x * gpc;
    const int gid = blockIdx.x * gpc + grp;
    const int sc_per_unit = (H / 128) / KS;        // super-chunks of a band per warp
    const int st_per_unit = sc_per_unit / GU_SC_PER_STAGE;
    const int sc_base = kpart * sc_per_unit;

    int known_units = a.n_shared * W13_BANDS;      // the shared expert needs no routing
    bool waited = false;
    int issued = 0;

    auto issue_ahead = [&](int limit) {
        while (issued < limit) {
            const int u = gid + (issued / st_per_unit) * n_groups;
            if (u >= known_units)
                break;
            if (lane == 0) {
                const int slot = u / W13_BANDS, band = u % W13_BANDS;
                const uint8_t *src = gu_band_src(a, sm, warp, slot, band) +
                                     (size_t)(sc_base + GU_SC_PER_STAGE * (issued % st_per_unit)) * SC_BYTES;
                uint64_t *bar = &sm.full[warp][issued % GU_RING];
                mbar_arrive_expect_tx(bar, GU_STAGE_BYTES);
                bulk_g2s(sm.ring[warp][issued % GU_RING], src, GU_STAGE_BYTES, bar);
            }
            ++issued;
        }
    };

    issue_ahead(GU_RING);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0;; ++i) {
        const int u = gid + (i / st_per_unit) * n_groups;
        if (u >= known_units) {
            if (!waited) {
                waited = true;
                griddep_wait();
                griddep_launch();
                const int ns = __ldcg(&st->n_slots);
                for (int s = lane; s < MAX_SLOTS; s += 32) {
                    int e = -1;
                    float ts = 0.f;
                    if (s < a.n_shared) {
                        ts = __ldg(a.shared_ts13 + s);
                    } else if (s < ns) {
                        e = __ldcg(&st->expert[s]);
                        if (e < 0 || e >= E) {
                            atomicOr(flag, FLAG_BAD_INDEX);
                            e = 0;
                        }
                        ts = __ldg(a.routed_ts13 + e);
                    }
                    sm.c_expert[warp][s] = e;
                    sm.c_ts[warp][s] = ts;
                }
                __syncwarp();
                known_units = ns * W13_BANDS;
                issue_ahead(i + GU_RING);
            }
            if (u >= known_units)
                break;
        }
        const int stage = i % GU_RING;
        mbar_wait_bounded(&sm.full[warp][stage], (i / GU_RING) & 1, flag);
        const int within = i % st_per_unit;
        mma_superchunks(sm.ring[warp][stage], GU_SC_PER_STAGE, sm.xfrag, blanes,
                        (sc_base + GU_SC_PER_STAGE * within) * 8, lane, acc);
        __syncwarp();
        if (lane == 0)
            fence_proxy_async();   // the stage's reads are done before the next copy lands
        issue_ahead(i + GU_RING + 1);

        if (within != st_per_unit - 1)
            continue;
        // ---- end of a unit: reduce the K parts, SiLU*up, store h ----
        const int slot = u / W13_BANDS, band = u % W13_BANDS;
        if (KS > 1) {
            sm.red[warp][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            named_barrier_sync(1 + grp, KS * 32);
            if (kpart == 0) {
                float4 s4 = sm.red[grp * KS][lane];
                for (int k = 1; k < KS; ++k) {
                    const float4 r = sm.red[grp * KS + k][lane];
                    s4.x += r.x; s4.y += r.y; s4.z += r.z; s4.w += r.w;
                }
                acc[0] = s4.x; acc[1] = s4.y; acc[2] = s4.z; acc[3] = s4.w;
            }
            named_barrier_sync(1 + grp, KS * 32);
        }
        if (kpart == 0) {
            const int g = lane >> 2, c = lane & 3;
            const float ts = (slot < a.n_shared) ? __ldg(a.shared_ts13 + slot) : sm.c_ts[warp][slot];
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
                const int t = 2 * c + tt;
                if (t < a.T) {
                    const float f = ts * pow2i(-sm.xshift[t]);
                    const float gv = acc[tt] * f, uv = acc[2 + tt] * f;
                    const float hv = gv / (1.0f + expf(-gv)) * uv;
                    hbuf[((size_t)slot * MAXT + t) * I + band * 8 + g] = __float2bfloat16_rn(hv);
                }
            }
            __threadfence();
            __syncwarp();
            uint32_t prev = 0;
            if (lane == 0)
                prev = atomicAdd(&slot_cnt[slot], 1u);
            prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
            if (prev == W13_BANDS - 1) {
                // this warp finished the slot's last band
                __threadfence();
                convert_slot(a, slot, lane, hbuf, hfrag, hexp);
                if (lane == 0)
                    slot_cnt[slot] = 0u;
            }
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
    if (!waited) {
        griddep_wait();
        griddep_launch();
    }
    // every issued stage was consumed: no copy is left in flight
}

// ---------------------------------------------------------------------------
// K3: down GEMV x routing weight -> per-slot partials
// ---------------------------------------------------------------------------
struct DnSmem {
    uint8_t ring[DN_WARPS][DN_RING][W2_BAND_BYTES];
    uint2 hbuf[DN_HBUF_ENTRIES];   // per group: two compact h-fragment buffers
    uint64_t full[DN_WARPS][DN_RING];
    uint64_t hbar[DN_WARPS][2];
};

__global__ void __launch_bounds__(DN_WARPS * 32, 1) down_kernel(DownArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    DnSmem &sm = *reinterpret_cast<DnSmem *>(smem_raw);

    const WsLayout L = ws_layout();
    uint32_t *flag = reinterpret_cast<uint32_t *>(a.ws + L.ctrl);
    const SlotTable *st = reinterpret_cast<const SlotTable *>(a.ws + L.slots);
    const uint2 *hfrag = reinterpret_cast<const uint2 *>(a.ws + L.hfrag);
    const int32_t *hexp = reinterpret_cast<const int32_t *>(a.ws + L.hexp);
    float *partials = reinterpret_cast<float *>(a.ws + L.partials);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BG = a.BG;                          // warps (bands) per unit
    const int gpc = DN_WARPS / BG;
    const int grp = warp / BG, wi = warp % BG;
    const int n_groups = gridDim.x * gpc;
    const int gid = blockIdx.x * gpc + grp;
    const int nbg = W2_BANDS / BG;
    const bool leader = (wi == 0);

    if (lane == 0) {
        for (int s = 0; s < DN_RING; ++s)
            mbar_init(&sm.full[warp][s], 1);
        if (leader) {
            mbar_init(&sm.hbar[grp][0], 1);
            mbar_init(&sm.hbar[grp][1], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // The slot table is final: this grid starts only after every gate/up CTA
    // passed its wait on the router kernel.
    const int n_slots = __ldcg(&st->n_slots);
    const int n_units = n_slots * nbg;

    const int blanes = 4 * a.T;
    const int hbuf_entries = DN_STEPS * blanes;            // one slot's compact fragments
    auto hbuf_of = [&](int b) { return sm.hbuf + (size_t)(grp * 2 + b) * hbuf_entries; };
    auto unit_of = [&](int k) { return gid + k * n_groups; };
    auto weight_src = [&](int u) {
        const int slot = u / nbg, bg = u % nbg;
        const uint8_t *base;
        if (slot < a.n_shared) {
            base = a.shared_w2 + (size_t)slot * W2_BYTES;
        } else {
            int e = __ldcg(&st->expert[slot]);
            if (e < 0 || e >= E) { atomicOr(flag, FLAG_BAD_INDEX); e = 0; }
            base = a.routed_w2 + (size_t)e * W2_BYTES;
        }
        return base + (size_t)(bg * BG + wi) * W2_BAND_BYTES;
    };
    auto issue_w = [&](int k) {
        const int u = unit_of(k);
        if (u < n_units && lane == 0) {
            uint64_t *bar = &sm.full[warp][k % DN_RING];
            mbar_arrive_expect_tx(bar, (uint32_t)W2_BAND_BYTES);
            bulk_g2s(sm.ring[warp][k % DN_RING], weight_src(u), (uint32_t)W2_BAND_BYTES, bar);
        }
    };
    auto issue_h = [&](int k) {
        const int u = unit_of(k);
        if (u < n_units && leader && lane == 0) {
            const int slot = u / nbg;
            uint64_t *bar = &sm.hbar[grp][k & 1];
            const uint32_t bytes = (uint32_t)hbuf_entries * 8;
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(hbuf_of(k & 1), hfrag + (size_t)slot * DN_STEPS * 32, bytes, bar);
        }
    };

    // weights first: they do not depend on the gate/up kernel
    for (int k = 0; k < DN_RING; ++k)
        issue_w(k);
    griddep_wait();     // h fragments are complete
    griddep_launch();
    issue_h(0);
    issue_h(1);

    for (int k = 0;; ++k) {
        const int u = unit_of(k);
        if (u >= n_units)
            break;
        const int slot = u / nbg, bg = u % nbg;
        const int band = bg * BG + wi;
        const int c = lane & 3, g = lane >> 2;
        // per-token factors: routing weight x tensor scale x 2^-shift
        float ts;
        if (slot < a.n_shared) {
            ts = __ldg(a.shared_ts2 + slot);
        } else {
            int e = __ldcg(&st->expert[slot]);
            e = (e < 0 || e >= E) ? 0 : e;
            ts = __ldg(a.routed_ts2 + e);
        }
        float f[2];
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            const int t = 2 * c + tt;
            f[tt] = 0.f;
            if (t < a.T)
                f[tt] = __ldcg(&st->wts[slot][t]) * ts * pow2i(-__ldcg(&hexp[slot * MAXT + t]));
        }
        mbar_wait_bounded(&sm.hbar[grp][k & 1], (k >> 1) & 1, flag);
        mbar_wait_bounded(&sm.full[warp][k % DN_RING], (k / DN_RING) & 1, flag);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_superchunks(sm.ring[warp][k % DN_RING], I / 128, hbuf_of(k & 1), blanes, 0, lane, acc);
        __syncwarp();
        if (lane == 0)
            fence_proxy_async();
        issue_w(k + DN_RING);
        // partial for rows 16*band + g (+8), tokens 2c, 2c+1
        float *P = partials + ((size_t)slot * H + 16 * band) * MAXT;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            const int t = 2 * c + tt;
            if (t < a.T) {
                P[g * MAXT + t] = acc[tt] * f[tt];
                P[(g + 8) * MAXT + t] = acc[2 + tt] * f[tt];
            }
        }
        // the group's hbuf[k & 1] is free once every warp of the group is here
        named_barrier_sync(1 + grp, BG * 32);
        if (leader && lane == 0)
            fence_proxy_async();
        issue_h(k + 2);
    }
}

// ---------------------------------------------------------------------------
// K4: out[t][n] = sum over slots (in slot order) of the partials, -> bf16
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) combine_kernel(CombineArgs a)
{
    const WsLayout L = ws_layout();
    const SlotTable *st = reinterpret_cast<const SlotTable *>(a.ws + L.slots);
    const float *partials = reinterpret_cast<const float *>(a.ws + L.partials);
    griddep_wait();
    griddep_launch();
    const int band = blockIdx.x;
    const int r = threadIdx.x >> 3, t = threadIdx.x & 7;
    if (t >= a.T)
        return;
    const int n_slots = __ldcg(&st->n_slots);
    const float *p = partials + ((size_t)16 * band + r) * MAXT + t;
    float sum = 0.f;
    for (int s = 0; s < n_slots; ++s)
        sum += __ldcg(p + (size_t)s * H * MAXT);
    a.out[(size_t)t * H + 16 * band + r] = __float2bfloat16_rn(sum);
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
template <typename Kern, typename Args>
static cudaError_t launch_ex(Kern k, const Args &args, dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args);
}

static cudaError_t set_smem_once(const void *fn, int *configured, size_t bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64 && configured[dev])
        return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        configured[dev] = 1;
    return e;
}

size_t gate_up_smem_bytes() { return sizeof(GuSmem); }
size_t down_smem_bytes() { return sizeof(DnSmem); }

cudaError_t launch_gate_up(const GateUpArgs &a, int grid, cudaStream_t stream, bool pdl)
{
    static int configured[64] = {0};
    cudaError_t e = set_smem_once((const void *)gate_up_kernel, configured, sizeof(GuSmem));
    if (e != cudaSuccess)
        return e;
    return launch_ex(gate_up_kernel, a, dim3(grid), dim3(GU_WARPS * 32), sizeof(GuSmem), stream, pdl);
}

cudaError_t launch_down(const DownArgs &a, int grid, cudaStream_t stream, bool pdl)
{
    static int configured[64] = {0};
    cudaError_t e = set_smem_once((const void *)down_kernel, configured, sizeof(DnSmem));
    if (e != cudaSuccess)
        return e;
    return launch_ex(down_kernel, a, dim3(grid), dim3(DN_WARPS * 32), sizeof(DnSmem), stream, pdl);
}

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream, bool pdl)
{
    return launch_ex(combine_kernel, a, dim3(W2_BANDS), dim3(128), 0, stream, pdl);
}

}  // namespace moe

// expert.cu -- K2 (gate/up GEMV fused with SiLU*up) and K3 (down GEMV fused
// with the routing-weighted combine and the shared expert) of the small-batch
// NVFP4 MoE layer.
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "From 1,096 kernels to 346": small-batch MoE kernels whose expert GEMVs read
// only the selected experts' weights; the expert combine is fused into the
// neighbouring GEMV; programmatic dependent launch lets each kernel load its
// weights while the previous one runs.  Section "A 40B MoE that activates
// 2.5B parameters": W4A16 (NVFP4 weights, BF16 activations).
//
// Both kernels stream packed 16-row bands (see common.cuh) with bulk async
// copies (cp.async.bulk + mbarrier) into shared memory.  Eight consumer warps
// decode e2m1 nibbles to bf16 in registers and run mma.m16n8k16 with the
// (up to 8) tokens as the N dimension; the e4m3 block scale of each 16-wide
// k step is applied to the fp32 accumulator, the tensor scale at the end.
// A ninth warp issues the copies.
#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// K2: gate/up
// ---------------------------------------------------------------------------


__device__ __forceinline__ const uint8_t *w13_band_ptr(const GateUpArgs &a, const SlotTable *st,
                                                       int slot, int band, uint32_t *flag)
{
    const uint8_t *base;
    if (slot < a.n_shared) {
        base = a.shared_w13 + (size_t)slot * W13_BYTES;
    } else {
        int e = __ldcg(&st->expert[slot]);
        if (e < 0 || e >= E) {
            atomicOr(flag, FLAG_BAD_INDEX);
            e = 0;
        }
        base = a.routed_w13 + (size_t)e * W13_BYTES;
    }
    return base + (size_t)band * W13_BAND_BYTES;
}

__device__ __forceinline__ float w13_tscale(const GateUpArgs &a, const SlotTable *st, int slot)
{
    if (slot < a.n_shared)
        return __ldg(a.shared_ts13 + slot);
    int e = __ldcg(&st->expert[slot]);
    e = (e < 0 || e >= E) ? 0 : e;
    return __ldg(a.routed_ts13 + e);
}

// One 16-row band x (a K range of) the activations: accumulate into acc[4]
// (rows g / g+8, tokens 2c / 2c+1) the scaled products of `nchunks` 64-wide
// chunks starting at chunk j0.  K is the row length of the matrix.
template <int K>
__device__ __forceinline__ void band_chunks(const uint8_t *band, const uint2 *bfrag, int j0,
                                            int nchunks, int lane, float acc[4])
{
    const int g = lane >> 2;
    for (int jj = 0; jj < nchunks; ++jj) {
        const int j = j0 + jj;
        const uint4 cw = *reinterpret_cast<const uint4 *>(band + j * 512 + lane * 16);
        const uint4 sc = *reinterpret_cast<const uint4 *>(band + 8 * K + (j >> 1) * 128 + g * 16);
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
        // the 8 blocks of this super-chunk: (j & 1) selects the upper 4
        const uint32_t sw0 = (j & 1) ? sc.z : sc.x;
        const uint32_t sw1 = (j & 1) ? sc.w : sc.y;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint32_t w = words[s];
            const uint2 b = bfrag[(4 * j + s) * 32 + lane];
            float d[4];
            mma_bf16_16816(d, decode_reg(w, 0), decode_reg(w, 1), decode_reg(w, 2), decode_reg(w, 3),
                           b.x, b.y);
            const uint32_t sw = (s < 2) ? sw0 : sw1;
            const float2 sf = e4m3x2_to_float2((s & 1) ? (sw >> 16) : (sw & 0xFFFFu));
            acc[0] = fmaf(sf.x, d[0], acc[0]);
            acc[1] = fmaf(sf.x, d[1], acc[1]);
            acc[2] = fmaf(sf.y, d[2], acc[2]);
            acc[3] = fmaf(sf.y, d[3], acc[3]);
        }
    }
}

__global__ void __launch_bounds__(EXPERT_THREADS, 1) gate_up_kernel(GateUpArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *stages = smem;
    uint2 *xfrag = reinterpret_cast<uint2 *>(smem + GU_SMEM_STAGES);
    float *red = reinterpret_cast<float *>(smem + GU_SMEM_STAGES + GU_SMEM_XFRAG);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + GU_SMEM_STAGES + GU_SMEM_XFRAG + GU_SMEM_RED);
    uint64_t *empty = full + GU_STAGES;

    const WsLayout L = ws_layout();
    uint32_t *flag = reinterpret_cast<uint32_t *>(a.ws + L.ctrl);
    const SlotTable *st = reinterpret_cast<const SlotTable *>(a.ws + L.slots);
    __nv_bfloat16 *hbuf = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.h);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int shared_units = a.n_shared * W13_BANDS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < GU_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CONSUMER_WARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CONSUMER_WARPS) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int i = 0;
            int u = blockIdx.x;
            int n_units = shared_units;   // known before routing: the shared expert
            bool waited = false;
            for (;; u += G, ++i) {
                if (u >= n_units && !waited) {
                    griddep_wait();
                    griddep_launch();
                    waited = true;
                    n_units = __ldcg(&st->n_slots) * W13_BANDS;
                }
                if (u >= n_units)
                    break;
                const int stage = i % GU_STAGES;
                if (i >= GU_STAGES &&
                    !mbar_wait_bounded(&empty[stage], ((i / GU_STAGES) - 1) & 1, flag))
                    break;
                const uint8_t *src = w13_band_ptr(a, st, u / W13_BANDS, u % W13_BANDS, flag);
                mbar_arrive_expect_tx(&full[stage], (uint32_t)W13_BAND_BYTES);
                bulk_g2s(stages + stage * W13_BAND_BYTES, src, (uint32_t)W13_BAND_BYTES, &full[stage]);
            }
            if (!waited) {
                griddep_wait();
                griddep_launch();
            }
            // drain: wait until the copies still in flight have landed
            for (int k = (i > GU_STAGES ? i - GU_STAGES : 0); k < i; ++k)
                mbar_wait_bounded(&full[k % GU_STAGES], (k / GU_STAGES) & 1, flag);
        } else {
            griddep_wait();
            griddep_launch();
        }
        return;
    }

    // ---------------- consumers ----------------
    const int tid = threadIdx.x;   // 0..255
    // Activations as B fragments: step s, lane l = 4g + c holds tokens g,
    // columns 16s + {2c, 2c+1} and 16s + {2c+8, 2c+9}, scaled by 2^96.
    // x is complete before this grid starts: the router kernel triggers this
    // launch only after its own wait on the kernel that produced x.
    for (int idx = tid; idx < GU_STEPS * 32; idx += CONSUMER_THREADS) {
        const int step = idx >> 5, l = idx & 31, g = l >> 2, c = l & 3;
        uint2 v = make_uint2(0u, 0u);
        if (g < a.T) {
            const uint32_t *xr = reinterpret_cast<const uint32_t *>(a.x + (size_t)g * H + 16 * step);
            v.x = scale_bf16x2(__ldg(xr + c));
            v.y = scale_bf16x2(__ldg(xr + 4 + c));
        }
        xfrag[idx] = v;
    }
    named_barrier_sync(1, CONSUMER_THREADS);

    int n_units = shared_units;
    bool waited = false;
    int i = 0;
    for (int u = blockIdx.x;; u += G, ++i) {
        if (u >= n_units && !waited) {
            griddep_wait();
            griddep_launch();
            waited = true;
            n_units = __ldcg(&st->n_slots) * W13_BANDS;
        }
        if (u >= n_units)
            break;
        const int slot = u / W13_BANDS, band = u % W13_BANDS;
        const int stage = i % GU_STAGES;
        mbar_wait_bounded(&full[stage], (i / GU_STAGES) & 1, flag);

        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        band_chunks<H>(stages + stage * W13_BAND_BYTES, xfrag, warp * GU_CHUNKS_PER_WARP,
                       GU_CHUNKS_PER_WARP, lane, acc);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);

        *reinterpret_cast<float4 *>(red + (warp * 32 + lane) * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        named_barrier_sync(1, CONSUMER_THREADS);
        if (tid < 64) {
            const int l = tid >> 1, tt = tid & 1;
            const int g = l >> 2, c = l & 3;
            const int t = 2 * c + tt;
            if (t < a.T) {
                float sg = 0.f, su = 0.f;
#pragma unroll
                for (int w = 0; w < CONSUMER_WARPS; ++w) {
                    sg += red[(w * 32 + l) * 4 + tt];
                    su += red[(w * 32 + l) * 4 + 2 + tt];
                }
                const float ts = w13_tscale(a, st, slot) * OUT_RESCALE;
                const float gv = sg * ts, uv = su * ts;
                const float hv = gv / (1.0f + expf(-gv)) * uv;
                hbuf[((size_t)slot * MAXT + t) * I + band * 8 + g] = __float2bfloat16_rn(hv);
            }
        }
        named_barrier_sync(1, CONSUMER_THREADS);
    }
    if (!waited) {
        griddep_wait();
        griddep_launch();
    }
}

// ---------------------------------------------------------------------------
// K3: down + combine
// ---------------------------------------------------------------------------



__global__ void __launch_bounds__(EXPERT_THREADS) down_combine_kernel(DownArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int BG = a.BG, SG = a.SG;
    uint8_t *stages = smem;
    uint2 *hfrag = reinterpret_cast<uint2 *>(smem + (size_t)SG * BG * W2_BAND_BYTES);
    float *red = reinterpret_cast<float *>(smem + (size_t)SG * BG * W2_BAND_BYTES + (size_t)SG * DN_STEPS * 32 * 8);
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(red) + CONSUMER_WARPS * 32 * 4 * 4);
    __shared__ int s_last;

    const WsLayout L = ws_layout();
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(a.ws + L.ctrl);
    uint32_t *flag = ctrl;
    uint32_t *counters = reinterpret_cast<uint32_t *>(a.ws + L.counters);
    const SlotTable *st = reinterpret_cast<const SlotTable *>(a.ws + L.slots);
    const __nv_bfloat16 *hbuf = reinterpret_cast<const __nv_bfloat16 *>(a.ws + L.h);
    float *partials = reinterpret_cast<float *>(a.ws + L.partials);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bg = blockIdx.x, q = blockIdx.y;

    // The slot table is final: this grid is launched only after every
    // gate/up CTA passed its wait on the router kernel.
    const int n_slots = __ldcg(&st->n_slots);
    const int Q = (n_slots + SG - 1) / SG;
    if (q >= Q)
        return;
    const int slot0 = q * SG;
    const int nsl = min(SG, n_slots - slot0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nsl; ++s)
            mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    const uint32_t stage_bytes = (uint32_t)(BG * W2_BAND_BYTES);
    if (warp == CONSUMER_WARPS && lane == 0) {
        // weights do not depend on the gate/up kernel: start them now
        for (int s = 0; s < nsl; ++s) {
            const int slot = slot0 + s;
            const uint8_t *base;
            if (slot < a.n_shared) {
                base = a.shared_w2 + (size_t)slot * W2_BYTES;
            } else {
                int e = __ldcg(&st->expert[slot]);
                if (e < 0 || e >= E) { atomicOr(flag, FLAG_BAD_INDEX); e = 0; }
                base = a.routed_w2 + (size_t)e * W2_BYTES;
            }
            mbar_arrive_expect_tx(&full[s], stage_bytes);
            bulk_g2s(stages + s * stage_bytes, base + (size_t)bg * BG * W2_BAND_BYTES, stage_bytes, &full[s]);
        }
    }
    griddep_wait();      // the gate/up kernel has finished: h is complete
    griddep_launch();

    // h of the slots as B fragments (scaled by 2^96)
    if (warp < CONSUMER_WARPS) {
        for (int idx = threadIdx.x; idx < nsl * DN_STEPS * 32; idx += CONSUMER_THREADS) {
            const int s = idx / (DN_STEPS * 32), rem = idx % (DN_STEPS * 32);
            const int step = rem >> 5, l = rem & 31, g = l >> 2, c = l & 3;
            uint2 v = make_uint2(0u, 0u);
            if (g < a.T) {
                const uint32_t *hr = reinterpret_cast<const uint32_t *>(
                    hbuf + ((size_t)(slot0 + s) * MAXT + g) * I + 16 * step);
                v.x = scale_bf16x2(__ldcg(hr + c));
                v.y = scale_bf16x2(__ldcg(hr + 4 + c));
            }
            hfrag[idx] = v;
        }
    }
    __syncthreads();

    const int WPB = CONSUMER_WARPS / BG;          // warps per band
    const int chunks_per_warp = (I / 64) / WPB;   // 8 / WPB
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < CONSUMER_WARPS) {
        const int bi = warp / WPB, kp = warp % WPB;
        const int c = lane & 3;
        for (int s = 0; s < nsl; ++s) {
            const int slot = slot0 + s;
            mbar_wait_bounded(&full[s], 0, flag);
            float tmp[4] = {0.f, 0.f, 0.f, 0.f};
            band_chunks<I>(stages + s * stage_bytes + bi * W2_BAND_BYTES, hfrag + s * DN_STEPS * 32,
                           kp * chunks_per_warp, chunks_per_warp, lane, tmp);
            float ts;
            if (slot < a.n_shared) {
                ts = __ldg(a.shared_ts2 + slot);
            } else {
                int e = __ldcg(&st->expert[slot]);
                e = (e < 0 || e >= E) ? 0 : e;
                ts = __ldg(a.routed_ts2 + e);
            }
            ts *= OUT_RESCALE;
            const float f0 = __ldcg(&st->wts[slot][2 * c]) * ts;
            const float f1 = __ldcg(&st->wts[slot][2 * c + 1]) * ts;
            acc[0] = fmaf(f0, tmp[0], acc[0]);
            acc[1] = fmaf(f1, tmp[1], acc[1]);
            acc[2] = fmaf(f0, tmp[2], acc[2]);
            acc[3] = fmaf(f1, tmp[3], acc[3]);
        }
        *reinterpret_cast<float4 *>(red + (warp * 32 + lane) * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
    __syncthreads();
    // sum the K parts of each band, store this CTA's partial for its rows
    for (int idx = threadIdx.x; idx < BG * 32 * 4; idx += blockDim.x) {
        const int bi = idx / 128, rem = idx % 128, l = rem >> 2, v = rem & 3;
        const int g = l >> 2, c = l & 3;
        const int t = 2 * c + (v & 1);
        const int row = 16 * (bg * BG + bi) + g + 8 * (v >> 1);
        if (t < a.T) {
            float sum = 0.f;
            for (int kp = 0; kp < WPB; ++kp)
                sum += red[((bi * WPB + kp) * 32 + l) * 4 + v];
            partials[((size_t)q * H + row) * MAXT + t] = sum;
            __threadfence();
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(&counters[bg], 1u);
        s_last = (prev == (uint32_t)(Q - 1));
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        // the last arriving slot group adds the partials in slot-group order
        for (int idx = threadIdx.x; idx < 16 * BG * a.T; idx += blockDim.x) {
            const int r = idx / a.T, t = idx % a.T;
            const int row = 16 * bg * BG + r;
            float sum = 0.f;
            for (int qq = 0; qq < Q; ++qq)
                sum += __ldcg(&partials[((size_t)qq * H + row) * MAXT + t]);
            a.out[(size_t)t * H + row] = __float2bfloat16_rn(sum);
        }
        if (threadIdx.x == 0)
            counters[bg] = 0u;
    }
    // no copy can still be in flight: every consumer waited on every stage
}

// ---------------------------------------------------------------------------
// Host launchers (called from api.cu)
// ---------------------------------------------------------------------------
cudaError_t launch_gate_up(const GateUpArgs &a, int grid, cudaStream_t stream, bool pdl)
{
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)GU_SMEM);
        if (e != cudaSuccess)
            return e;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(EXPERT_THREADS);
    cfg.dynamicSmemBytes = GU_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gate_up_kernel, a);
}

cudaError_t launch_down(const DownArgs &a, int qmax, cudaStream_t stream, bool pdl)
{
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem_max = down_smem_bytes(8, DN_MAX_SG);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(down_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_max);
        if (e != cudaSuccess)
            return e;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(W2_BANDS / a.BG, qmax);
    cfg.blockDim = dim3(EXPERT_THREADS);
    cfg.dynamicSmemBytes = down_smem_bytes(a.BG, a.SG);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, down_combine_kernel, a);
}

}  // namespace moe

// gemv.cu -- the small-batch dense GEMV on the packed NVFP4 layout (and on
// row-major BF16 weights): y = W x for T <= 8 tokens.
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "From 1,096 kernels to 346": the small-batch dense GEMV (the dense MLP of
// the first layers and the projections) runs on the same packed NVFP4 weights
// as the large-batch kernel.  Here it reads the band layout of the expert
// matrices (common.cuh) with the stage steps of the decode layer
// (stage.cuh); the same kernel serves the BF16 shared experts of a layer
// whose shared experts are routing sinks (TML Inkling page, section "MoE":
// only the routed experts are NVFP4).
//
// One CTA per SM, 16 compute warps and one epilogue warp.  A CTA owns a
// contiguous range of 16-row bands of one matrix.  The 16 compute warps form
// G = 16 / Q groups of Q warps; in round r group g takes band
// b0 + G r + g and warp q of the group its contiguous share of the band's
// stages (a fixed K range, so its B fragments never change).  Each warp
// streams its stages through a private ring of bulk copies (NVFP4) or
// cp.async (BF16), ahead across rounds; the ring's first stages are issued
// before the wait on the preceding kernel (the weights do not depend on it).
// A round's Q partials of a band meet in a shared-memory buffer and the
// epilogue warp adds them in warp order (deterministic), scales and stores.
// x enters shared memory once per CTA by whole-row bulk copies, rows 16
// bytes apart so that the fragment loads of the 32 lanes hit 32 banks (a
// tensor-map box of 32-byte pieces, or 16-byte loads by every thread, took
// several times longer for the same bytes); NVFP4 converts it in place to
// f16 after the exact per-token power-of-two rescale (common.cuh), BF16 uses
// the bf16 words as they are.
// Every wait is bounded and reports MOE_FLAG_WAIT_TIMEOUT instead of hanging.
#include "kernels.cuh"
#include "stage.cuh"

namespace moe {

namespace {

constexpr int GW = 16;                  // compute warps
constexpr int GNT = (GW + 1) * 32;      // + the epilogue warp
constexpr int GSTG = 2 * SC_BYTES;      // ring slot: one NVFP4 stage (a BF16 stage uses 2048 bytes)

template <int RW>
struct GSmem {
    uint8_t ring[GW][RW][GSTG];         // per warp RW stage slots, contiguous (a unit fills 1 or 2 of them)
    float4 red[2][GW][32];              // a round's partials (round r uses r % 2)
    uint64_t full[GW][RW];
    uint64_t pfull[2];                  // all 16 warps stored their round-r partials
    uint64_t pempty[2];                 // the epilogue warp has read them
    uint64_t xbar;                      // x has landed
    float xinv[MAXT];                   // NVFP4: 2^-xshift[t]
    uint32_t xmax[MAXT];                // NVFP4: max |x| of each token (fp32 bits)
    alignas(128) uint32_t xs[1];        // x row-major, 8 rows 2 K + 16 bytes apart (extends past the struct)
};

template <int RW>
constexpr size_t gsmem_bytes(int K)
{
    return offsetof(GSmem<RW>, xs) + (size_t)MAXT * (2 * K + 16);
}

// Ring stages issued before the wait on the preceding kernel (the weights do
// not depend on it): about what lands during that wait; the rest follow x's
// copy so that x does not queue behind them.
constexpr int PRE = 1;

template <bool BW, int RW>
__global__ void __launch_bounds__(GNT, 1) dense_gemv_kernel(GemvArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    GSmem<RW> &sm = *reinterpret_cast<GSmem<RW> *>(smem_raw);
    uint32_t *flag = a.flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, K = a.K, N = a.N;
    const int Q = a.q, G = GW / Q;
    const int m = (int)blockIdx.x / a.ctas_per_mat, cm = (int)blockIdx.x % a.ctas_per_mat;
    const int nbm = N / 16;
    const int b0 = (int)((long)nbm * cm / a.ctas_per_mat), b1 = (int)((long)nbm * (cm + 1) / a.ctas_per_mat);
    const int rounds = (b1 - b0 + G - 1) / G;
    const int S = BW ? K / 64 : K / 256;      // stages per band
    const uint8_t *w = a.w + (size_t)m * a.w_mat_stride;
    // NVFP4 stages move in units of up to UNIT adjacent stages of a band (one
    // bulk copy each): an SM completes only ~10 bulk copies per µs whatever
    // their size, so 4,608-byte copies stream about twice as fast as 2,304
    constexpr int UNIT = (!BW && RW >= 4) ? 2 : 1;
    constexpr int NU = RW / UNIT;             // unit slots per warp

    if (lane == 0 && warp < GW) {
        for (int s = 0; s < NU; ++s)
            mbar_init(&sm.full[warp][s], BW ? 32 : 1);   // BF16: one cp.async arrival per lane
    }
    if (threadIdx.x < 2) {
        mbar_init(&sm.pfull[threadIdx.x], GW);
        mbar_init(&sm.pempty[threadIdx.x], 1);
    }
    if (threadIdx.x == 0)
        mbar_init(&sm.xbar, 1);
    if (threadIdx.x < MAXT)
        sm.xmax[threadIdx.x] = 0u;
    if (lane == 0)
        fence_barrier_init();
    __syncthreads();

    // the compute warp's place: group g, member q; its stages of each band
    const int g = warp / Q, q = warp % Q;
    const int s0 = S * q / Q, s1 = S * (q + 1) / Q, per = s1 - s0;
    const int my_rounds = warp < GW && b1 - b0 > g ? (b1 - b0 - g + G - 1) / G : 0;
    const int upr = (per + UNIT - 1) / UNIT;  // units per round
    const int n_units = my_rounds * upr;

    // unit i: round i / upr, stages s0 + UNIT (i % upr) .. (at most UNIT, within the round)
    auto issue_stage = [&](int rs, int i) {
        const int r = i / upr, s = s0 + UNIT * (i % upr);
        const int nst = min(UNIT, s1 - s);
        const int band = b0 + G * r + g;
        uint64_t *bar = &sm.full[warp][rs];
        uint8_t *slot = sm.ring[warp][UNIT * rs];
        if (BW) {
            // rows of the band (GATE_UP: 8 gate rows 8 band.. and the matching
            // up rows), columns 64 s ..; lane 2 rr + h copies bytes [64 h, 64 h
            // + 64) of band row rr into its swizzled place
            const int rr = lane >> 1, h = lane & 1;
            const int row = a.kind == MOE_PACK_GATE_UP ? (rr < 8 ? 8 * band + rr : N / 2 + 8 * band + (rr - 8))
                                                       : 16 * band + rr;
            const uint8_t *src = w + ((size_t)row * K + 64 * s) * 2 + 64 * h;
            uint8_t *dst = slot + rr * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                cp_async_cg16(dst + 16 * ((4 * h + u) ^ (4 * (rr & 1))), src + 16 * u);
            cp_async_arrive(bar);
            return;
        }
        if (lane != 0)
            return;
        mbar_arrive_expect_tx(bar, (uint32_t)(nst * GSTG));
        bulk_g2s(slot, w + (size_t)band * band_bytes(K) + (size_t)s * GSTG, (uint32_t)(nst * GSTG), bar);
    };
    int ic = 0, ii = 0;                        // units consumed / issued
    auto issue_upto = [&](int depth) {
        while (ii < n_units && ii < ic + depth) {
            issue_stage(ii % NU, ii);
            ++ii;
        }
    };
    auto issue_ahead = [&]() { issue_upto(NU); };
    if (warp < GW)
        issue_upto(PRE);

    griddep_wait();      // x is written by the preceding kernel
    griddep_launch();

    // ---- x -> shared memory, row-major (rows 16 bytes apart) ----
    // Lanes t < T of warp 0 each bulk-copy token t's row (rows T.. stay
    // unwritten: their mma columns are never stored).  NVFP4 then converts
    // the words in place to f16 after the exact per-token power-of-two
    // rescale.
    const int rpw = K / 2 + 4;                 // row pitch in 32-bit words
    if (warp == 0) {
        if (lane == 0)
            mbar_arrive_expect_tx(&sm.xbar, (uint32_t)(T * K * 2));
        __syncwarp();
        if (lane < T)
            bulk_g2s(sm.xs + lane * rpw, a.x + (size_t)m * a.x_mat_stride + (size_t)lane * K, (uint32_t)(K * 2),
                     &sm.xbar);
    }
    if (warp < GW)
        issue_ahead();
    mbar_wait_bounded(&sm.xbar, 0, flag);
    if (!BW) {
        // warp w < 2 T takes half hf = w % 2 of row t = w / 2: K / 16
        // pieces, XH at a time per lane (all of them at K <= 4096); the
        // row's max |x| is one reduction per warp and one shared-memory max
        // per warp, then the pieces go back converted (re-read above 4096)
        constexpr int XH = GEMV_MAX_K_RW4 / 16 / 32;   // 8 pieces per lane
        const int xrow = warp >> 1, xhf = warp & 1;
        const bool xw = warp < 2 * T;
        const int nh = K / 16;                        // pieces per half row
        uint4 *hp = reinterpret_cast<uint4 *>(sm.xs + xrow * rpw) + xhf * nh;
        uint4 hv[XH];
        uint32_t mx = 0u;
        if (xw) {
            for (int c0 = 0; c0 < nh; c0 += 32 * XH) {
#pragma unroll
                for (int i = 0; i < XH; ++i) {
                    const int j = c0 + 32 * i + lane;
                    hv[i] = j < nh ? hp[j] : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int i = 0; i < XH; ++i) {
                    const uint32_t w4[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
                    for (int u = 0; u < 4; ++u)   // |bf16| bit patterns order like their values
                        mx = max(mx, max(w4[u] & 0x7FFFu, (w4[u] >> 16) & 0x7FFFu));
                }
            }
            mx = __reduce_max_sync(0xFFFFFFFFu, mx);
            if (lane == 0)
                atomicMax(&sm.xmax[xrow], mx);
        }
        __syncthreads();
        if (threadIdx.x < MAXT)
            sm.xinv[threadIdx.x] = pow2i(-act_shift(bf16_bits_to_float(sm.xmax[threadIdx.x])));
        if (xw) {
            const float p = pow2i(act_shift(bf16_bits_to_float(sm.xmax[xrow])));
            for (int c0 = 0; c0 < nh; c0 += 32 * XH) {
                if (nh > 32 * XH) {   // more than one chunk: the registers hold the last one only
#pragma unroll
                    for (int i = 0; i < XH; ++i) {
                        const int j = c0 + 32 * i + lane;
                        if (j < nh)
                            hv[i] = hp[j];
                    }
                }
#pragma unroll
                for (int i = 0; i < XH; ++i) {
                    const int j = c0 + 32 * i + lane;
                    if (j < nh)
                        hp[j] = make_uint4(bf16x2_to_f16x2_scaled(hv[i].x, p), bf16x2_to_f16x2_scaled(hv[i].y, p),
                                           bf16x2_to_f16x2_scaled(hv[i].z, p), bf16x2_to_f16x2_scaled(hv[i].w, p));
                }
            }
        }
    }
    __syncthreads();

    if (warp == GW) {
        // ---- the epilogue warp: round r's bands, partials added in warp order ----
        const int gg = lane >> 2, c = lane & 3;
        const float ts = BW ? 1.0f : (a.ts_dev ? __ldg(a.ts_dev + m) : a.ts_host);
#pragma unroll 1
        for (int r = 0; r < rounds; ++r) {
            const int bb = r & 1;
            if (lane == 0)
                mbar_wait_bounded(&sm.pfull[bb], (uint32_t)(r >> 1) & 1u, flag);
            __syncwarp();
#pragma unroll 1
            for (int gi = 0; gi < G; ++gi) {
                const int band = b0 + G * r + gi;
                if (band >= b1)
                    break;
                // the Q partials added in warp order, loaded eight at a time
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int h8 = 0; h8 < GW; h8 += 8) {
                    if (h8 >= Q)
                        break;
                    float4 pv[8];
#pragma unroll
                    for (int qq = 0; qq < 8; ++qq)
                        if (h8 + qq < Q)
                            pv[qq] = sm.red[bb][gi * Q + h8 + qq][lane];
#pragma unroll
                    for (int qq = 0; qq < 8; ++qq)
                        if (h8 + qq < Q) {
                            if (h8 + qq == 0) {
                                sum = pv[0];
                            } else {
                                sum.x += pv[qq].x; sum.y += pv[qq].y; sum.z += pv[qq].z; sum.w += pv[qq].w;
                            }
                        }
                }
                const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int t = 2 * c + tt;
                    if (t >= T)
                        continue;
                    const float f = BW ? 1.0f : ts * sm.xinv[t];
                    const float lo = sv[tt] * f, hi = sv[2 + tt] * f;
                    if (a.epi == GEMV_SILU_H) {
                        // band rows gg (gate 8 band + gg) and gg + 8 (its up row)
                        __nv_bfloat16 *h = static_cast<__nv_bfloat16 *>(a.y) + (size_t)m * a.y_mat_stride;
                        h[(size_t)t * (N / 2) + 8 * band + gg] = __float2bfloat16_rn(lo / (1.0f + expf(-lo)) * hi);
                    } else if (a.epi == GEMV_OUT_F32) {
                        float *y = static_cast<float *>(a.y) + (size_t)m * a.y_mat_stride;
                        y[(size_t)t * N + 16 * band + gg] = lo;
                        y[(size_t)t * N + 16 * band + gg + 8] = hi;
                    } else {
                        __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(a.y) + (size_t)m * a.y_mat_stride;
                        y[(size_t)t * N + 16 * band + gg] = __float2bfloat16_rn(lo);
                        y[(size_t)t * N + 16 * band + gg + 8] = __float2bfloat16_rn(hi);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.pempty[bb]);
        }
        return;
    }

    // ---- a compute warp ----
#pragma unroll 1
    for (int r = 0; r < rounds; ++r) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < my_rounds) {
#pragma unroll 1
            for (int s = s0; s < s1; ++s) {
                const int rs = ic % NU, off = (s - s0) % UNIT;
                if (off == 0)
                    mbar_wait_bounded(&sm.full[warp][rs], (ic / NU) & 1, flag);
                if (BW)
                    bf16_stage_xs(sm.ring[warp][UNIT * rs + off], sm.xs, rpw, 4 * s, lane, acc);
                else
                    mma_stage_xs(sm.ring[warp][UNIT * rs + off], sm.xs, rpw, 16 * s, lane, acc);
                if (off == UNIT - 1 || s == s1 - 1) {   // the unit's last stage: free its slot
                    __syncwarp();
                    ++ic;
                    issue_ahead();
                }
            }
        }
        // every warp reports every round (an idle one with zeros), so the
        // count of pfull is fixed
        const int bb = r & 1;
        if (r >= 2 && lane == 0)
            mbar_wait_bounded(&sm.pempty[bb], (uint32_t)((r >> 1) - 1) & 1u, flag);
        __syncwarp();
        sm.red[bb][warp][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.pfull[bb]);
    }
}

template <bool BW, int RW>
int configure(PerDevice &pd)
{
    return per_device(pd, [](int) {
        const int smem = (int)gsmem_bytes<RW>(RW == 4 ? GEMV_MAX_K_RW4 : GEMV_MAX_K);
        return cudaFuncSetAttribute(dense_gemv_kernel<BW, RW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem) == cudaSuccess
                   ? 1
                   : -1;
    });
}

PerDevice g_gemv_attr[4];

}  // namespace

// Warps per band: the power of two Q <= 16 that minimises a warp's stage
// steps plus its bulk copies (units of `unit` stages), both about 0.1 µs on
// GB300 (ties: more bands at once, i.e. fewer rounds).
int gemv_warps_per_band(int bands_per_cta, int stages, int unit)
{
    int best_q = 16;
    long best = -1;
    for (int qq = 16; qq >= 1; qq >>= 1) {
        const int gq = 16 / qq;
        const long per = (stages + qq - 1) / qq;
        const long cost = (long)((bands_per_cta + gq - 1) / gq) * (per + (per + unit - 1) / unit);
        if (best < 0 || cost <= best) {
            best = cost;
            best_q = qq;
        }
    }
    return best_q;
}

cudaError_t launch_gemv(GemvArgs a, int sm_count, cudaStream_t stream)
{
    const bool bw = a.bf16w != 0;
    const bool rw4 = a.K <= GEMV_MAX_K_RW4;
    const int which = (bw ? 2 : 0) + (rw4 ? 0 : 1);
    const int ok = bw ? (rw4 ? configure<true, 4>(g_gemv_attr[which]) : configure<true, 2>(g_gemv_attr[which]))
                      : (rw4 ? configure<false, 4>(g_gemv_attr[which]) : configure<false, 2>(g_gemv_attr[which]));
    if (ok <= 0)
        return cudaErrorInvalidValue;
    const int nbm = a.N / 16;
    int cpm = sm_count / a.n_mat;
    if (cpm < 1)
        cpm = 1;
    if (cpm > nbm)
        cpm = nbm;
    a.ctas_per_mat = cpm;
    const int stages = bw ? a.K / 64 : a.K / 256;
    a.q = gemv_warps_per_band((nbm + cpm - 1) / cpm, stages, (!bw && rw4) ? 2 : 1);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cpm * a.n_mat));
    cfg.blockDim = dim3(GNT);
    cfg.dynamicSmemBytes = rw4 ? gsmem_bytes<4>(a.K) : gsmem_bytes<2>(a.K);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (bw)
        return rw4 ? cudaLaunchKernelEx(&cfg, dense_gemv_kernel<true, 4>, a)
                   : cudaLaunchKernelEx(&cfg, dense_gemv_kernel<true, 2>, a);
    return rw4 ? cudaLaunchKernelEx(&cfg, dense_gemv_kernel<false, 4>, a)
               : cudaLaunchKernelEx(&cfg, dense_gemv_kernel<false, 2>, a);
}

}  // namespace moe

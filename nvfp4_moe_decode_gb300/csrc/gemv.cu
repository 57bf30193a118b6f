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
// x enters as mma B fragments in shared memory, built once per CTA: NVFP4,
// f16 after the exact per-token power-of-two rescale (common.cuh); BF16, bf16
// in the column order of bf16_bcol.
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
    uint8_t ring[GW][RW][GSTG];
    float4 red[2][GW][32];              // a round's partials (round r uses r % 2)
    uint64_t full[GW][RW];
    uint64_t pfull[2];                  // all 16 warps stored their round-r partials
    uint64_t pempty[2];                 // the epilogue warp has read them
    float xinv[MAXT];                   // NVFP4: 2^-xshift[t]
    float hmx[MAXT][2];                 // NVFP4: max |x| of each half of a token's row
    uint2 xfrag[1];                     // [K / 16][32]: B fragments (extends past the struct)
};

template <int RW>
constexpr size_t gsmem_bytes(int K)
{
    return offsetof(GSmem<RW>, xfrag) + (size_t)K * 16;
}

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

    if (lane == 0 && warp < GW) {
        for (int s = 0; s < RW; ++s)
            mbar_init(&sm.full[warp][s], BW ? 32 : 1);   // BF16: one cp.async arrival per lane
    }
    if (threadIdx.x < 2) {
        mbar_init(&sm.pfull[threadIdx.x], GW);
        mbar_init(&sm.pempty[threadIdx.x], 1);
    }
    if (lane == 0)
        fence_barrier_init();
    __syncthreads();

    // the compute warp's place: group g, member q; its stages of each band
    const int g = warp / Q, q = warp % Q;
    const int s0 = S * q / Q, s1 = S * (q + 1) / Q, per = s1 - s0;
    const int my_rounds = warp < GW && b1 - b0 > g ? (b1 - b0 - g + G - 1) / G : 0;
    const int n_stages = my_rounds * per;

    auto issue_stage = [&](int rs, int i) {
        const int r = i / per, s = s0 + i % per;
        const int band = b0 + G * r + g;
        uint64_t *bar = &sm.full[warp][rs];
        if (BW) {
            // rows of the band (GATE_UP: 8 gate rows 8 band.. and the matching
            // up rows), columns 64 s ..; lane 2 rr + h copies bytes [64 h, 64 h
            // + 64) of band row rr into its swizzled place
            const int rr = lane >> 1, h = lane & 1;
            const int row = a.kind == MOE_PACK_GATE_UP ? (rr < 8 ? 8 * band + rr : N / 2 + 8 * band + (rr - 8))
                                                       : 16 * band + rr;
            const uint8_t *src = w + ((size_t)row * K + 64 * s) * 2 + 64 * h;
            uint8_t *dst = sm.ring[warp][rs] + rr * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                cp_async_cg16(dst + 16 * ((4 * h + u) ^ (4 * (rr & 1))), src + 16 * u);
            cp_async_arrive(bar);
            return;
        }
        if (lane != 0)
            return;
        mbar_arrive_expect_tx(bar, GSTG);
        bulk_g2s(sm.ring[warp][rs], w + (size_t)band * band_bytes(K) + (size_t)s * GSTG, GSTG, bar);
    };
    int ic = 0, ii = 0;
    auto issue_ahead = [&]() {
        while (ii < n_stages && ii < ic + RW) {
            issue_stage(ii % RW, ii);
            ++ii;
        }
    };
    if (warp < GW)
        issue_ahead();

    griddep_wait();      // x is written by the preceding kernel
    griddep_launch();

    // ---- x -> B fragments [k16 step][lane] in shared memory ----
    // Two warps per token (warp 2 t + hf takes columns [hf K / 2, (hf + 1)
    // K / 2)); each lane holds up to XCH 16-byte pieces at once, all loads of
    // a chunk issued before any is used.  NVFP4: the token's max |x| first
    // (both halves, exchanged through shared memory), then each piece -- 8
    // columns = the .x (or .y) words of the 4 lanes (t, c) of one k16 step --
    // is scaled into f16.  BF16: a piece is the two uint2 fragments of lane
    // (t, c) for a pair of steps (the column order of bf16_bcol).
    const __nv_bfloat16 *x = a.x + (size_t)m * a.x_mat_stride;
    constexpr int XCH = 8;
    const int nh = K / 16;                    // pieces per half row
    const int nper = (nh + 31) / 32;          // per lane
    const int xt = warp >> 1, hf = warp & 1;
    const bool xwarp = warp < 2 * T;
    const uint4 *xrow = reinterpret_cast<const uint4 *>(x + (size_t)xt * K) + hf * nh;
    uint4 xv[XCH];
    auto load_chunk = [&](int c0) {
#pragma unroll
        for (int i = 0; i < XCH; ++i) {
            const int j = lane + 32 * (c0 + i);
            xv[i] = (c0 + i < nper && j < nh) ? __ldg(xrow + j) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    uint32_t *xf32 = reinterpret_cast<uint32_t *>(sm.xfrag);
    auto store_chunk = [&](int c0, float p) {
#pragma unroll
        for (int i = 0; i < XCH; ++i) {
            const int j = lane + 32 * (c0 + i);
            if (c0 + i >= nper || j >= nh)
                continue;
            const int jj = hf * nh + j;        // piece index in the row: columns 8 jj .. 8 jj + 7
            const uint32_t w4[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
            if (BW) {
                // columns 64 ch + 32 aa + 8 c + 0..7: steps 4 ch + 2 aa (+1), lane 4 t + c
                const int ch = jj >> 3, aa = (jj >> 2) & 1, c = jj & 3;
                const int s0 = 4 * ch + 2 * aa;
                uint2 *f = sm.xfrag;
                f[s0 * 32 + 4 * xt + c] = make_uint2(w4[0], w4[1]);
                f[(s0 + 1) * 32 + 4 * xt + c] = make_uint2(w4[2], w4[3]);
            } else {
                // columns 16 step + 8 h + 2 c, +1 for c = 0..3: token t's words
                // of a step lie in 8 banks, so each store takes c in lane
                // order (8 distinct banks per instruction, not 2)
                const int step = jj >> 1, h = jj & 1;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = (cc + lane) & 3;
                    const uint32_t wc = c == 0 ? w4[0] : c == 1 ? w4[1] : c == 2 ? w4[2] : w4[3];
                    xf32[(step * 32 + 4 * xt + c) * 2 + h] = bf16x2_to_f16x2_scaled(wc, p);
                }
            }
        }
    };
    // fragments of the lanes of absent tokens (4 T ..) are zero
    for (int i = threadIdx.x; i < (K / 16) * 32; i += GNT)
        if (((i & 31) >> 2) >= T)
            sm.xfrag[i] = make_uint2(0u, 0u);
    if (BW) {
        if (xwarp)
            for (int c0 = 0; c0 < nper; c0 += XCH) {
                load_chunk(c0);
                store_chunk(c0, 1.0f);
            }
    } else {
        float mx = 0.0f;
        if (xwarp)
            for (int c0 = 0; c0 < nper; c0 += XCH) {
                load_chunk(c0);
                __nv_bfloat162 m2 = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < XCH; ++i) {
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(xv[i].x)));
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(xv[i].y)));
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(xv[i].z)));
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(xv[i].w)));
                }
                mx = fmaxf(mx, fmaxf(__low2float(m2), __high2float(m2)));
            }
        // max |x| >= 0: its fp32 bit pattern orders like an unsigned int
        mx = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mx)));
        if (xwarp && lane == 0)
            sm.hmx[xt][hf] = mx;
        __syncthreads();
        if (xwarp) {
            const int sh = act_shift(fmaxf(sm.hmx[xt][0], sm.hmx[xt][1]));
            if (hf == 0 && lane == 0)
                sm.xinv[xt] = pow2i(-sh);
            const float p = pow2i(sh);
            if (nper <= XCH) {
                store_chunk(0, p);   // the only chunk is still in registers
            } else {
                for (int c0 = 0; c0 < nper; c0 += XCH) {
                    load_chunk(c0);
                    store_chunk(c0, p);
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
                float4 sum = sm.red[bb][gi * Q][lane];
#pragma unroll 1
                for (int qq = 1; qq < Q; ++qq) {
                    const float4 v = sm.red[bb][gi * Q + qq][lane];
                    sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
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
    const uint2 *bfrag = sm.xfrag;
#pragma unroll 1
    for (int r = 0; r < rounds; ++r) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < my_rounds) {
#pragma unroll 1
            for (int s = s0; s < s1; ++s) {
                const int rs = ic % RW;
                mbar_wait_bounded(&sm.full[warp][rs], (ic / RW) & 1, flag);
                if (BW)
                    bf16_stage(sm.ring[warp][rs], bfrag, 4 * s, lane, acc);
                else
                    mma_stage(sm.ring[warp][rs], bfrag, 16 * s, lane, acc);
                __syncwarp();
                ++ic;
                issue_ahead();
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

// Warps per band: the power of two Q <= 16 that minimises rounds x stages per
// warp (ties: more bands at once, i.e. fewer rounds).
int gemv_warps_per_band(int bands_per_cta, int stages)
{
    int best_q = 16;
    long best = -1;
    for (int qq = 16; qq >= 1; qq >>= 1) {
        const int gq = 16 / qq;
        const long cost = (long)((bands_per_cta + gq - 1) / gq) * ((stages + qq - 1) / qq);
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
    a.q = gemv_warps_per_band((nbm + cpm - 1) / cpm, stages);

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

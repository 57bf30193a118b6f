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
// One CTA per SM: 16 compute warps in 4 groups of 4, plus a sync warp.
// Phases:
//  1. before waiting on the preceding kernel: router CTAs load their slice of
//     the router weights; group 0 of the first 64 CTAs starts the bulk copies
//     of one band of the shared expert (it needs no routing);
//  2. x arrives in shared memory by one bulk copy; in CTAs 0..127 the 16
//     compute warps compute the fp32 logits of two experts and store each
//     with the launch's tag in one 64-bit word; warps 0..7 then turn x into
//     f16 mma fragments;
//  3. every CTA reads the logits until each carries the launch's tag, takes
//     the top-6 of each token (one warp per token, identical in every CTA)
//     and builds the slot table: the shared expert, then the distinct
//     selected experts in ascending order, each with its per-token routing
//     weight;
//  4. units are dealt round-robin to the 4 x #CTA groups (group id
//     grp * #CTA + cta; a group takes ids gid, gid + G, gid + 2G, ...):
//       gate/up unit (slot, band): the 4 warps take one K quarter each of
//         a 16-row band of W13 (8 gate + 8 up rows); warp k % 4 adds the
//         four partials in warp order and applies SiLU*up -> h (bf16);
//       down unit (slot, 4 bands): once the slot's 64 gate/up bands are done,
//         the slot's h arrives by bulk copy, each token's row is scaled by the
//         power of two of its max |h| (found there) into f16 fragments in
//         place; each warp computes one 16-row band of W2 h, times the
//         routing weight;
//     gate/up ids precede down ids and every group walks its ids in
//     increasing order, so a down unit only waits on gate/up units that other
//     groups reach without waiting themselves.  A compute warp reports a
//     finished h band or down partial through a shared-memory counter only;
//     the sync warp turns those into the cross-CTA counts (slot counters,
//     band counters) behind one gpu-scope fence per pass, because such a
//     fence costs a warp about a microsecond while the SM streams weights,
//     and it issues the h copies;
//  5. the warp that computes a band's partial for the last slot waits until
//     the other slots' partials of the band are counted, then adds all of
//     them in slot order (deterministic) and writes out (bf16).
// NVFP4: every warp streams its units' weights through a private 3-stage ring
// of shared-memory buffers filled by cp.async.bulk and decodes them in
// registers.  BF16 (the W16A16 variant of the Flint page, section "From 1,096
// kernels to 346": BF16 decode): the rows are row-major in HBM, and each warp
// loads its 16 rows straight into registers, two 64-column chunks ahead.
// Every wait is bounded and reports MOE_FLAG_WAIT_TIMEOUT instead of hanging.
#include "kernels.cuh"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int FW = 16;                 // compute warps per CTA
constexpr int FT = FW * 32;            // compute threads
constexpr int SYNC_WARP = FW;          // warp 16: cross-CTA counts and the h copies
constexpr int NT = FT + 32;            // threads per CTA
constexpr int NG = 4;                  // unit groups per CTA
constexpr int GW = 4;                  // warps per group
constexpr int RING = 3;                // stages per warp
constexpr int STG = 2 * SC_BYTES;      // 2304 bytes: two super-chunks
constexpr int ROUTER_CTAS = E / 2;     // 128 CTAs x 2 experts
constexpr int HROW = H_PITCH * 2;      // padded bytes of one token's h row (shared memory and workspace)
constexpr int HBUF = MAXT * HROW;      // one slot's h, 8.1 KB at T = 8
constexpr uint32_t SLOT_DONE = W13_BANDS; // gate/up bands that complete a slot
constexpr int GUU = W13_BANDS;            // 64 gate/up units (one band each) per slot
constexpr int DN_UNITS = W2_BANDS / GW;   // 32 down units of 4 bands per slot
constexpr int GU_PARTS = (H / 128) / 2;   // 8 stages per W13 band
constexpr int DN_PARTS = (I / 128) / 2;   // 2 stages per W2 band

struct FSmem {
    uint8_t ring[FW][RING][STG];
    uint2 xfrag[(H / 16) * 32];        // entry (step, l) at step * 32 + l; zero for l >= 4T
    uint8_t hbuf[NG][2][HBUF];         // raw h rows, rescaled in place into fragments;
                                       // before the unit loop: x (T x 4 KB)
    uint64_t full[FW][RING];
    uint64_t hbar[NG][2];
    uint64_t kfull[NG][2];             // K-split gate/up: the three partials of the unit are in kred
    uint64_t kempty[NG][2];            // K-split gate/up: the unit's writer has read kred
    uint64_t xbar;
    int32_t sel[MAXT][TOPK];
    float selw[MAXT][TOPK];
    uint32_t bitmap[E / 32];
    int bcnt[E / 32];
    int n_slots;
    int32_t slot_expert[MAX_SLOTS];
    float wts[MAX_SLOTS][MAXT];
    int xshift[MAXT];
    float sumsq[FW];                   // pre-norm: per-warp partial sums of squares
    int hshift[NG][2][MAXT];           // power-of-two exponents of the h in hbuf[grp][b]
    float hmx[NG][GW][32];             // per-thread max |h| of the down unit being converted
    float4 kred[NG][2][GW - 1][32];    // K-split gate/up: the non-writers' partials, by unit parity
    uint32_t gu_done[NG][GW];          // gate/up units whose h warp wq of the group has stored
    uint32_t dn_done[NG][GW];          // down units whose partial warp wq of the group has stored
    uint32_t hrel[NG];                 // down units of the group done with their h buffer
    uint32_t hclaim[NG];               // down units of the group whose h copy has been issued
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

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acquire.gpu;" ::: "memory"); }
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// 64-bit relaxed accesses at gpu scope (single-copy atomic)
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_relaxed_add(uint32_t *p, uint32_t v)
{
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// CTA-scope release store / acquire load (shared-memory progress counters)
__device__ __forceinline__ void st_release_cta(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.cta.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.cta.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

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

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32.
__device__ __forceinline__ void mma_bf16_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// BF16 rows are consumed in a k order chosen so that each lane's A registers
// come from two 16-byte words per row and 64-column chunk: lane
// (g, c) loads columns 8c..8c+7 and 32+8c..32+8c+7 of rows g and g+8, and k16
// step s of the chunk pairs its words 2s, 2s+1 with the activation columns
// 32*(s/2) + 8c + 4*(s%2) + 0..3 (a permutation of the chunk's 64 columns,
// applied to both operands, so the dot products are unchanged).
__host__ __device__ __forceinline__ int bf16_bcol(int step, int c)
{
    const int s = step & 3;
    return 64 * (step >> 2) + 32 * (s >> 1) + 8 * c + 4 * (s & 1);
}

// One 64-column chunk of a BF16 band in a ring stage (16 rows x 128 bytes,
// 16-byte unit u of row r at position u ^ 4 (r & 1), so the reads below are
// free of bank conflicts) times the B fragments of k16 steps step0 ..
// step0 + 3.  Lane (g, c) takes units c and 4 + c of rows g and g + 8.
__device__ __forceinline__ void bf16_stage(const uint8_t *stage, const uint2 *bfrag, int step0, int lane,
                                           float acc[4])
{
    const int g = lane >> 2, c = lane & 3, sw = 4 * (g & 1);
    const uint8_t *ra = stage + g * 128, *rb = stage + (g + 8) * 128;
    const uint4 a0 = *reinterpret_cast<const uint4 *>(ra + 16 * (c ^ sw));
    const uint4 a1 = *reinterpret_cast<const uint4 *>(ra + 16 * ((4 + c) ^ sw));
    const uint4 b0 = *reinterpret_cast<const uint4 *>(rb + 16 * (c ^ sw));
    const uint4 b1 = *reinterpret_cast<const uint4 *>(rb + 16 * ((4 + c) ^ sw));
    const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int step = step0 + s;
        const uint2 b = bfrag[step * 32 + lane];
        mma_bf16_16816(acc, wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1], b.x, b.y);
    }
}

// 16-byte global -> shared copy that skips L1, and an arrival on an mbarrier
// once all of this thread's earlier copies have landed.
__device__ __forceinline__ void cp_async_cg16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Two consecutive super-chunks of one band (one stage) times the B fragments
// from k16 step `step0`.  The fragments of a step fill all 32 lanes (lanes
// 4T.. hold zeros), so every lane loads unconditionally: a predicated load
// here cost the loop 18% when measured alone.
__device__ __forceinline__ void mma_stage(const uint8_t *stage, const uint2 *bfrag, int step0, int lane,
                                          float acc[4])
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
                const uint2 b = bfrag[step * 32 + lane];
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
    int band;    // this warp's 16-row band (W13 band for gate/up, W2 band for down)
};

}  // namespace

template <bool BW>
__global__ void __launch_bounds__(NT, 1) moe_layer_kernel(LayerArgs a)
{
    static_assert(sizeof(RouterRed) <= sizeof(FSmem::ring) / 2, "router partials fit the router warps' rings");
    static_assert(sizeof(FSmem::hbuf) >= (size_t)2 * MAXT * H * 2, "x and delta fit the h buffers");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    FSmem &sm = *reinterpret_cast<FSmem *>(smem_raw);

    const WsLayout L = ws_layout();
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(a.ws + L.ctrl);
    uint32_t *flag = ctrl;
    uint32_t *slot_cnt = reinterpret_cast<uint32_t *>(a.ws + L.slot_cnt);
    uint32_t *band_cnt = reinterpret_cast<uint32_t *>(a.ws + L.band_cnt);
    unsigned long long *tlogits = reinterpret_cast<unsigned long long *>(a.ws + L.tlogits);
    __nv_bfloat16 *hglob = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.h);
    float *partials = reinterpret_cast<float *>(a.ws + L.partials);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = warp / GW, wq = warp % GW;
    const bool leader = (wq == 0);
    const bool lead_thread = leader && lane == 0;
    const int T = a.T;
    const int blanes = 4 * T;

    if (lane == 0 && warp < FW) {
        for (int s = 0; s < RING; ++s)
            mbar_init(&sm.full[warp][s], BW ? 32 : 1);   // BF16: one cp.async arrival per lane
        if (leader) {
            mbar_init(&sm.hbar[grp][0], 1);
            mbar_init(&sm.hbar[grp][1], 1);
            for (int q = 0; q < 2; ++q) {
                mbar_init(&sm.kfull[grp][q], GW - 1);
                mbar_init(&sm.kempty[grp][q], 1);
            }
        }
        if (threadIdx.x == 0)
            mbar_init(&sm.xbar, 1);
        fence_barrier_init();
    }
    __syncthreads();

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
    // BF16 banks: W13 [2I][H] and W2 [H][I] row-major per expert
    auto bf_w13 = [&](int slot) -> const __nv_bfloat16 * {
        const uint8_t *base = (slot < a.n_shared) ? a.s_w13 + (size_t)slot * W13_BYTES_BF
                                                  : a.r_w13 + (size_t)sm.slot_expert[slot] * W13_BYTES_BF;
        return reinterpret_cast<const __nv_bfloat16 *>(base);
    };
    auto bf_w2 = [&](int slot) -> const __nv_bfloat16 * {
        const uint8_t *base = (slot < a.n_shared) ? a.s_w2 + (size_t)slot * W2_BYTES_BF
                                                  : a.r_w2 + (size_t)sm.slot_expert[slot] * W2_BYTES_BF;
        return reinterpret_cast<const __nv_bfloat16 *>(base);
    };
    // one stage = two super-chunks (2304 bytes) of this warp's band: part p
    auto stage_src = [&](const Unit &u, int p) -> const uint8_t * {
        return (u.down ? w2_src(u.slot, u.band) : w13_src(u.slot, u.band)) + (size_t)(2 * p) * SC_BYTES;
    };
    auto issue_stage = [&](int ring_slot, const Unit &u, int p) {
        uint64_t *bar = &sm.full[warp][ring_slot];
        if (BW) {
            // chunk p (64 columns) of the 16 rows: lane 2r + h copies bytes
            // [64 h, 64 h + 64) of row r, then arrives when they have landed
            const int r = lane >> 1, h = lane & 1;
            const uint8_t *src;
            if (!u.down) {
                const int row = r < 8 ? 8 * u.band + r : I + 8 * u.band + (r - 8);
                src = reinterpret_cast<const uint8_t *>(bf_w13(u.slot)) + ((size_t)row * H + 64 * p) * 2 + 64 * h;
            } else {
                src = reinterpret_cast<const uint8_t *>(bf_w2(u.slot)) + ((size_t)(16 * u.band + r) * I + 64 * p) * 2 +
                      64 * h;
            }
            uint8_t *dst = sm.ring[warp][ring_slot] + r * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                cp_async_cg16(dst + 16 * ((4 * h + i) ^ (4 * (r & 1))), src + 16 * i);
            cp_async_arrive(bar);
            return;
        }
        if (lane != 0)
            return;
        mbar_arrive_expect_tx(bar, STG);
        bulk_g2s(sm.ring[warp][ring_slot], stage_src(u, p), STG, bar);
    };

    // ---- phase 1: work that needs nothing from the preceding kernel ----
    // units are dealt round-robin: group gid takes ids gid, gid + G, ...; the
    // shared expert's gate/up units (ids 0..63) go to group 0 of the first
    // CTAs.  A gate/up unit is one band and each warp takes a K quarter (two
    // of the band's eight stages), so the few slots of a small batch still
    // spread over every warp.
    // stages of a unit per warp: NVFP4 two super-chunks each, BF16 one
    // 64-column chunk of the 16 rows each
    auto nparts = [&](const Unit &u) {
        return BW ? (u.down ? I / 64 : H / 64 / GW) : (u.down ? DN_PARTS : GU_PARTS / GW);
    };
    auto part0 = [&](const Unit &u) { return u.down ? 0 : nparts(u) * wq; };
    const int n_groups = NG * (int)gridDim.x;
    const int gid = grp * (int)gridDim.x + (int)blockIdx.x;
    const bool static_shared = !BW && warp < FW && (a.n_shared > 0) && gid < GUU;
    const Unit u0 = Unit{false, 0, gid};
    const int n_pre = static_shared ? min(RING, nparts(u0)) : 0;
    for (int p = 0; p < n_pre; ++p)
        issue_stage(p, u0, part0(u0) + p);
    // router CTAs: warp w of the 16 takes expert 2 * cta + w / 8, columns
    // [256 (w % 8), 256 (w % 8) + 256), eight per lane
    const bool router_warp = blockIdx.x < ROUTER_CTAS && warp < FW;
    const int r_e = blockIdx.x * 2 + (warp >> 3);
    const int r_k8 = warp & 7;
    uint4 wv = make_uint4(0u, 0u, 0u, 0u);
    if (router_warp)
        wv = ldg_nc_v4(a.wr + (size_t)r_e * H + 256 * r_k8 + 8 * lane);

    griddep_wait();      // x is written by the preceding kernel; the counters are re-armed
    griddep_launch();    // the next kernel may start its own phase 1
    // this launch's tag on the logits (never 0, the value a zeroed workspace holds)
    const uint32_t ltag = __ldcg(&ctrl[5]) + 1u;

    // ---- phase 2: x -> shared memory; router logits | activation fragments ----
    uint8_t *xs = &sm.hbuf[0][0][0];   // T x 4 KB, free until the unit loop
    uint8_t *ds = xs + MAXT * H * 2;   // pre-norm: the previous layer's output, T x 4 KB
    const bool has_delta = a.prenorm && a.delta != nullptr;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&sm.xbar, (uint32_t)(T * H * 2) * (has_delta ? 2u : 1u));
        bulk_g2s(xs, a.x, (uint32_t)(T * H * 2), &sm.xbar);
        if (has_delta)
            bulk_g2s(ds, a.delta, (uint32_t)(T * H * 2), &sm.xbar);
    }
    mbar_wait_bounded(&sm.xbar, 0, flag);
    if (a.prenorm) {
        // Pre-norm residual stream of a decoder stack: v = bf16(x + delta)
        // (the residual after the previous layer), and the layer's input is
        // xn = bf16(v / sqrt(mean(v^2) + eps)) with unit weight.  Two warps
        // per token; each lane sums its 32 squares in order, then the warp
        // butterfly, then the two halves (fixed order).
        uint4 *xv = reinterpret_cast<uint4 *>(xs);
        const uint4 *dv = reinterpret_cast<const uint4 *>(ds);
        const int t = warp >> 1, half = warp & 1;
        uint4 vv[4];
        float ss = 0.f;
        if (t < T) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int idx = t * (H / 8) + half * (H / 16) + 32 * i + lane;
                uint4 r = xv[idx];
                if (has_delta) {
                    const uint4 d = dv[idx];
                    uint32_t *rw = &r.x;
                    const uint32_t *dw = &d.x;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const __nv_bfloat16 lo = __float2bfloat16_rn(bf16_bits_to_float(rw[q] & 0xFFFFu) + bf16_bits_to_float(dw[q] & 0xFFFFu));
                        const __nv_bfloat16 hi = __float2bfloat16_rn(bf16_bits_to_float(rw[q] >> 16) + bf16_bits_to_float(dw[q] >> 16));
                        rw[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
                    }
                }
                vv[i] = r;
                const uint32_t *rw = &r.x;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float lo = bf16_bits_to_float(rw[q] & 0xFFFFu), hi = bf16_bits_to_float(rw[q] >> 16);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
        if (lane == 0 && warp < FW)
            sm.sumsq[warp] = ss;
        __syncthreads();
        if (t < T) {
            const float ms = (sm.sumsq[2 * t] + sm.sumsq[2 * t + 1]) * (1.0f / H);
            const float rinv = 1.0f / sqrtf(ms + a.eps);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int idx = t * (H / 8) + half * (H / 16) + 32 * i + lane;
                uint4 n = vv[i];
                uint32_t *nw = &n.x;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat16 lo = __float2bfloat16_rn(bf16_bits_to_float(nw[q] & 0xFFFFu) * rinv);
                    const __nv_bfloat16 hi = __float2bfloat16_rn(bf16_bits_to_float(nw[q] >> 16) * rinv);
                    nw[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
                }
                xv[idx] = n;
                if (blockIdx.x == 0) {
                    if (a.resid_out)
                        reinterpret_cast<uint4 *>(a.resid_out)[idx] = vv[i];
                    if (a.xn_out)
                        reinterpret_cast<uint4 *>(a.xn_out)[idx] = n;
                }
            }
        }
        __syncthreads();
    }
    const __nv_bfloat16 *xsh = reinterpret_cast<const __nv_bfloat16 *>(xs);

    if (router_warp) {
        float acc[MAXT];
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
            acc[t] = 0.0f;
            if (t < T) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xsh + (size_t)t * H + 256 * r_k8 + 8 * lane);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[t] = fmaf(bf16_bits_to_float(xw[q] & 0xFFFFu), bf16_bits_to_float(ww[q] & 0xFFFFu), acc[t]);
                    acc[t] = fmaf(bf16_bits_to_float(xw[q] >> 16), bf16_bits_to_float(ww[q] >> 16), acc[t]);
                }
            }
        }
        // the stage rings of warps 8..15 are idle until the unit loop (the
        // shared expert's early copies go to warps 0..3)
        RouterRed &red = *reinterpret_cast<RouterRed *>(&sm.ring[8][0][0]);
        float logit;
        // each logit carries the launch tag in the same 64-bit word, so a
        // reader that sees the tag sees the logit: no fence, no counter
        if (router_reduce(acc, (int)threadIdx.x, T, red, 5, &logit))
            st_relaxed_u64(&tlogits[(threadIdx.x % MAXT) * E + blockIdx.x * 2 + threadIdx.x / MAXT],
                           ((unsigned long long)ltag << 32) | __float_as_uint(logit));
        fence_proxy_async();               // the ring is refilled by bulk copies later
    }
    if (warp < 8) {
        // x -> mma fragments [step][32] (zeros in lanes 4T..): lane l < 4T of
        // warp w holds steps w, w + 8, ... of token l / 4.  BF16 weights:
        // bf16 in the permuted column order of bf16_bcol.  NVFP4: f16, each
        // token's row scaled by the power of two of its max |x| (found first,
        // one warp per token).
        const uint32_t *xw = reinterpret_cast<const uint32_t *>(xs);
        const int g = lane >> 2, c = lane & 3;
        float p = 1.0f;
        if (!BW) {
            if (warp < T) {
                const uint4 *row = reinterpret_cast<const uint4 *>(xsh + (size_t)warp * H);
                __nv_bfloat162 m2 = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < H / 256; ++i) {
                    const uint4 v = row[lane + 32 * i];
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(v.x)));
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(v.y)));
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(v.z)));
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(v.w)));
                }
                // max |x| >= 0: its fp32 bit pattern orders like an unsigned int
                const float m = __uint_as_float(
                    __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fmaxf(__low2float(m2), __high2float(m2)))));
                if (lane == 0)
                    sm.xshift[warp] = act_shift(m);
            }
            named_barrier_sync(6, 256);
            if (lane < blanes)
                p = pow2i(sm.xshift[g]);
        }
        {
#pragma unroll 4
            for (int step = warp; step < H / 16; step += 8) {
                uint2 v = make_uint2(0u, 0u);   // lanes 4T.. carry no token
                if (lane < blanes) {
                    if (BW) {
                        const int w0 = (g * H + bf16_bcol(step, c)) / 2;
                        v = make_uint2(xw[w0], xw[w0 + 1]);
                    } else {
                        const int w0 = (g * H + 16 * step) / 2 + c;
                        v = make_uint2(bf16x2_to_f16x2_scaled(xw[w0], p), bf16x2_to_f16x2_scaled(xw[w0 + 4], p));
                    }
                }
                sm.xfrag[step * 32 + lane] = v;
            }
        }
    }

    // ---- phase 3: routing (every CTA, identically) ----
    for (int i = threadIdx.x; i < MAX_SLOTS * MAXT; i += FT)
        sm.wts[i / MAXT][i % MAXT] = 0.0f;
    if (threadIdx.x < E / 32)
        sm.bitmap[threadIdx.x] = 0u;
    if (threadIdx.x < NG * GW) {
        (&sm.gu_done[0][0])[threadIdx.x] = 0u;
        (&sm.dn_done[0][0])[threadIdx.x] = 0u;
    }
    if (threadIdx.x < NG) {
        sm.hrel[threadIdx.x] = 0u;
        sm.hclaim[threadIdx.x] = 0u;
    }

    __syncthreads();
    if (warp < T) {
        // the token's 256 logits, re-read until every one carries this launch's tag
        const unsigned long long *row = tlogits + warp * E;
        float v[8];
        bool have = false;
        for (uint32_t it = 0;; ++it) {
            have = true;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const unsigned long long w = ld_relaxed_u64(row + lane + 32 * m);
                v[m] = __uint_as_float((uint32_t)w);
                have = have && (uint32_t)(w >> 32) == ltag;
            }
            if (__all_sync(0xFFFFFFFFu, have))
                break;
            if (it == SPIN_LIMIT) {
                if (lane == 0)
                    atomicOr(flag, FLAG_TIMEOUT);
                break;
            }
            __nanosleep(32);
        }
        int ex;
        float wt;
        bool bad;
        warp_route_values(v, lane, ex, wt, bad);
        if (lane < TOPK) {
            sm.sel[warp][lane] = ex;
            sm.selw[warp][lane] = wt;
            atomicOr(&sm.bitmap[ex >> 5], 1u << (ex & 31));
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
    __syncthreads();
    if (warp == 0) {
        // slot table by one warp: ranks of the selected experts (bitmap
        // prefix counts), then the per-token weights
        const uint32_t bits = lane < E / 32 ? sm.bitmap[lane] : 0u;
        if (lane < E / 32)
            sm.bcnt[lane] = __popc(bits);
        __syncwarp();
        int base = a.n_shared, total = 0;
#pragma unroll
        for (int w = 0; w < E / 32; ++w) {
            const int c = sm.bcnt[w];
            base += (w < lane) ? c : 0;
            total += c;
        }
        {
            uint32_t b = bits;
            int r = 0;
            while (b) {
                const int bit = __ffs(b) - 1;
                sm.slot_expert[base + r] = lane * 32 + bit;
                ++r;
                b &= b - 1;
            }
        }
        if (lane < a.n_shared) {
            sm.slot_expert[lane] = -1 - lane;
            for (int t = 0; t < T; ++t)
                sm.wts[lane][t] = 1.0f;
        }
        if (lane == 0)
            sm.n_slots = a.n_shared + total;
        __syncwarp();
        // slot of expert e = base of bitmap word e / 32 + the set bits below it
#pragma unroll
        for (int i0 = 0; i0 < MAXT * TOPK; i0 += 32) {
            const int i = i0 + lane;
            const bool ok = i < T * TOPK;
            const int t = i / TOPK, ei = ok ? sm.sel[t][i % TOPK] : 0;
            const uint32_t wbits = __shfl_sync(0xFFFFFFFFu, bits, ei >> 5);
            const int b0 = __shfl_sync(0xFFFFFFFFu, base, ei >> 5);
            if (ok)
                sm.wts[b0 + __popc(wbits & ((1u << (ei & 31)) - 1u))][t] = sm.selw[t][i % TOPK];
        }
    }
    fence_proxy_async();   // generic writes to the x / h region precede later bulk copies into it
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

    // ---- phase 4: the units ----
    const int gu_total = n_slots * GUU;                             // unit ids [0, gu_total): gate/up
    const int end_id = gu_total + n_slots * DN_UNITS;               // then down units
    auto unit_id_of = [&](int group, int k) { return group + k * n_groups; };
    auto unit_id = [&](int k) { return unit_id_of(gid, k); };
    auto decode = [&](int id) -> Unit {
        if (id < gu_total)
            return Unit{false, (int)((unsigned)id / GUU), (int)((unsigned)id % GUU)};
        const int d = id - gu_total;
        return Unit{true, (int)((unsigned)d / DN_UNITS), 4 * (int)((unsigned)d % DN_UNITS) + wq};
    };
    // first down unit of this group, and the down-unit index of unit k
    const int k_down0 = gid >= gu_total ? 0 : (gu_total - gid + n_groups - 1) / n_groups;
    // h of down unit dk of group g: the slot's T padded rows, one bulk copy
    // into hbuf[g][dk & 1] (the slot counter has been acquired)
    auto issue_h = [&](int g, int slot, int b) {
        fence_proxy_async_global();   // h was published to the generic proxy by releases
        uint64_t *bar = &sm.hbar[g][b];
        const uint32_t bytes = (uint32_t)((T - 1) * HROW + I * 2);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(sm.hbuf[g][b], hglob + (size_t)slot * MAXT * H_PITCH, bytes, bar);
    };

    // The warp that computed a band's partial for the last slot adds up the
    // band once the other n_slots - 1 partials are counted: every slot's
    // partial in slot order, its own last.
    auto combine_band = [&](int band) {
        const int r = lane >> 1, th = lane & 1;      // row r, tokens 4*th .. 4*th+3
        const float4 *src = reinterpret_cast<const float4 *>(partials + ((size_t)16 * band + r) * MAXT) + th;
        if (lane == 0) {
            for (uint32_t it = 0; ld_acquire(&band_cnt[band]) < (uint32_t)(n_slots - 1); ++it) {
                if (it == SPIN_LIMIT) {
                    atomicOr(flag, FLAG_TIMEOUT);
                    break;
                }
                __nanosleep(32);
            }
        }
        __syncwarp();
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
    };

    // ---- the sync warp: every cross-CTA step of the unit phase ----
    // Lane g < NG follows group g.  Each pass it (1) copies h for the
    // group's next down unit once the slot's 64 gate/up bands are counted
    // (two h buffers per group, refilled when the group has released one);
    // (2) counts the bands whose h the group's warps have stored into the
    // slot counters and their down partials (all but the last slot's) into
    // the band counters, with one gpu-scope fence ahead of all the counts of
    // the pass, so that no compute warp ever waits on a fence or an atomic.
    auto run_sync_warp = [&]() {
        const int g = lane;
        const bool gl = lane < NG;
        const int gid_g = g * (int)gridDim.x + (int)blockIdx.x;
        int kd0 = 0, ndn = 0;
        if (gl) {
            kd0 = gid_g >= gu_total ? 0 : (gu_total - gid_g + n_groups - 1) / n_groups;
            const int kend = gid_g >= end_id ? 0 : (end_id - gid_g + n_groups - 1) / n_groups;
            ndn = kend - kd0;
        }
        uint32_t gsig[GW], dsig[GW], n_gu[GW];
#pragma unroll
        for (int q = 0; q < GW; ++q) {
            gsig[q] = dsig[q] = 0u;
            n_gu[q] = kd0 > q ? (uint32_t)((kd0 - q + GW - 1) / GW) : 0u;   // units k = q + 4n < kd0
        }
        int h_next = 0, probe_for = -1;
        uint32_t probe_val = 0u;
        bool counted_out = false;        // this CTA reads no slot counter any more
        for (uint32_t it = 0;; ++it) {
            if (it == 4 * SPIN_LIMIT) {
                if (lane == 0)
                    atomicOr(flag, FLAG_TIMEOUT);
                break;
            }
            bool busy = false;
            // (1) h of the next down unit
            if (gl && h_next < ndn) {   // copies the group's leader claimed
                const int claimed = (int)*reinterpret_cast<volatile uint32_t *>(&sm.hclaim[g]);
                if (claimed > h_next) {
                    h_next = claimed;
                    probe_for = -1;
                }
            }
            if (gl && h_next < ndn && h_next < (int)ld_acquire_cta(&sm.hrel[g]) + 2) {
                const int slot = (unit_id_of(gid_g, kd0 + h_next) - gu_total) / DN_UNITS;
                if (probe_for == h_next && probe_val >= SLOT_DONE) {
                    fence_acquire_gpu();     // pairs with the fences ahead of the slot's counts
                    if (atomicCAS(&sm.hclaim[g], (uint32_t)h_next, (uint32_t)h_next + 1u) == (uint32_t)h_next)
                        issue_h(g, slot, h_next & 1);
                    ++h_next;
                    probe_for = -1;
                    busy = true;
                } else {
                    probe_val = ld_relaxed(&slot_cnt[slot]);   // looked at on the next pass
                    probe_for = h_next;
                }
            }
            // (2) counts
            uint32_t gd[GW], dd[GW];
            bool fresh = false;
#pragma unroll
            for (int q = 0; q < GW; ++q) {
                gd[q] = gl ? ld_acquire_cta(&sm.gu_done[g][q]) : 0u;
                dd[q] = gl ? ld_acquire_cta(&sm.dn_done[g][q]) : 0u;
                fresh |= gd[q] != gsig[q] || dd[q] != dsig[q];
            }
            // new counts to add (the last slot's partials are not counted)
            bool need = false;
#pragma unroll
            for (int q = 0; q < GW; ++q) {
                need |= gd[q] != gsig[q];
                if (dd[q] != dsig[q])
                    need |= (unit_id_of(gid_g, kd0 + (int)dsig[q]) - gu_total) / DN_UNITS < n_slots - 1;
            }
            if (__any_sync(0xFFFFFFFFu, fresh)) {
                busy = true;
                if (__any_sync(0xFFFFFFFFu, need))
                    fence_acq_rel_gpu();   // the stores counted below become visible before their counts
                if (gl) {
#pragma unroll
                    for (int q = 0; q < GW; ++q)
                        for (; gsig[q] < gd[q]; ++gsig[q]) {
                            const int kq = q + GW * (int)gsig[q];
                            if (kq != kd0 - 1)   // the group's last gate/up band is counted by its writer
                                red_relaxed_add(&slot_cnt[(unsigned)unit_id_of(gid_g, kq) / GUU], 1u);
                        }
#pragma unroll
                    for (int q = 0; q < GW; ++q)
                        for (; dsig[q] < dd[q]; ++dsig[q]) {
                            const int d = unit_id_of(gid_g, kd0 + (int)dsig[q]) - gu_total;
                            // the last slot's partial is added where it is made; the
                            // group's last down unit is counted by its own warps
                            if (d / DN_UNITS < n_slots - 1 && (int)dsig[q] != ndn - 1)
                                red_relaxed_add(&band_cnt[4 * (d % DN_UNITS) + q], 1u);
                        }
                }
            }
            bool slots_done = !gl || h_next == ndn;
#pragma unroll
            for (int q = 0; q < GW; ++q)
                slots_done = slots_done && (!gl || gsig[q] == n_gu[q]);
            if (!counted_out && __all_sync(0xFFFFFFFFu, slots_done)) {
                // this CTA neither reads nor adds to a slot counter any more:
                // count it out (the fence orders those accesses first)
                __syncwarp();
                if (lane == 0) {
                    fence_acq_rel_gpu();
                    red_relaxed_add(&ctrl[4], 1u);
                }
                counted_out = true;
            }
            bool done = counted_out && (!gl || h_next == ndn);
#pragma unroll
            for (int q = 0; q < GW; ++q)
                done = done && (!gl || (gsig[q] == n_gu[q] && dsig[q] == (uint32_t)ndn));
            if (__all_sync(0xFFFFFFFFu, done))
                break;
            if (!__any_sync(0xFFFFFFFFu, busy))
                __nanosleep(64);
        }
    };

    if (warp == SYNC_WARP) {
        run_sync_warp();
    } else {
        // ---- stage stream of this warp: (unit k, part p) in order, RING in flight ----
        int ik = 0, ip = 0, icount = 0;      // next stage to issue
        if (n_pre > 0) {                     // the first n_pre parts of unit 0 were issued before the wait
            icount = n_pre;
            if (n_pre == nparts(u0))
                ik = 1;
            else
                ip = n_pre;
        }
        auto issue_ahead = [&](int limit) {
            while (icount < limit) {
                const int id = unit_id(ik);
                if (id >= end_id)
                    break;
                const Unit u = decode(id);
                issue_stage(icount % RING, u, part0(u) + ip);
                ++icount;
                if (++ip == nparts(u)) {
                    ip = 0;
                    ++ik;
                }
            }
        };
        issue_ahead(RING);

        int ccount = 0;                  // stages consumed
        uint32_t n_written = 0;          // gate/up units whose h this warp wrote
        uint32_t n_partials = 0;         // down units whose partial this warp wrote
        // stores of the warp, then one lane counts them (CTA scope; the sync
        // warp makes them visible to the other CTAs)
        auto publish = [&](uint32_t *ctr, uint32_t v) {
            __syncwarp();
            if (lane == 0)
                st_release_cta(ctr, v);
        };
        // The writer of the group's last gate/up unit goes on to a down unit
        // that waits for h anyway (or to nothing), so it counts its band
        // itself; the sync warp skips that count.
        auto count_now_if_last_gu = [&](int k, int slot) {
            if (k == k_down0 - 1) {
                __syncwarp();
                if (lane == 0) {
                    fence_acq_rel_gpu();
                    red_relaxed_add(&slot_cnt[slot], 1u);
                }
            }
        };
        float acc[4];
        for (int k = 0;; ++k) {
            const int id = unit_id(k);
            if (id >= end_id)
                break;
            const Unit u = decode(id);

            const uint2 *bfrag = sm.xfrag;
            int b = 0;
            if (u.down) {
                const int dk = k - k_down0;
                b = dk & 1;
                // The sync warp copies h once the slot's gate/up bands are
                // counted.  If it has not yet, the leader waits on the slot
                // counter itself and claims the copy (whoever moves the claim
                // counter from dk to dk + 1 issues it).
                if (lead_thread && *reinterpret_cast<volatile uint32_t *>(&sm.hclaim[grp]) <= (uint32_t)dk) {
                    for (uint32_t it = 0; ld_acquire(&slot_cnt[u.slot]) < SLOT_DONE; ++it) {
                        if (it == SPIN_LIMIT) {
                            atomicOr(flag, FLAG_TIMEOUT);
                            break;
                        }
                        __nanosleep(32);
                    }
                    __threadfence_block();   // the counter read precedes the claim the sync warp sees
                    if (atomicCAS(&sm.hclaim[grp], (uint32_t)dk, (uint32_t)dk + 1u) == (uint32_t)dk)
                        issue_h(grp, u.slot, b);
                }
                mbar_wait_bounded(&sm.hbar[grp][b], (dk >> 1) & 1, flag);
                // rescale h (padded bf16 rows) in place into fragments [step][32]
                // (zeros in lanes 4T..): lane l < 4T of warp wq holds steps wq,
                // wq + 4, ... of token l / 4; NVFP4 scales each token's row by the
                // power of two of its max |h|, taken over the 16 threads that
                // hold the row.
                const uint32_t *hw = reinterpret_cast<const uint32_t *>(sm.hbuf[grp][b]);
                const bool hl = lane < blanes;
                const int hg = lane >> 2, hc = lane & 3;
                constexpr int HJ = (I / 16) / GW;              // steps per warp
                uint32_t src0[HJ], src1[HJ];
                __nv_bfloat162 m2 = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < HJ; ++j) {
                    const int step = wq + GW * j;
                    src0[j] = src1[j] = 0u;
                    if (hl) {
                        if (BW) {
                            const int w0 = (hg * HROW) / 4 + bf16_bcol(step, hc) / 2;
                            src0[j] = hw[w0];
                            src1[j] = hw[w0 + 1];
                        } else {
                            const int w0 = (hg * HROW) / 4 + 8 * step + hc;
                            src0[j] = hw[w0];
                            src1[j] = hw[w0 + 4];
                        }
                    }
                    if (!BW) {
                        m2 = __hmax2(m2, __habs2(u32_as_bf162(src0[j])));
                        m2 = __hmax2(m2, __habs2(u32_as_bf162(src1[j])));
                    }
                }
                if (!BW)
                    sm.hmx[grp][wq][lane] = fmaxf(__low2float(m2), __high2float(m2));
                named_barrier_sync(1 + grp, GW * 32);
                int sh = 0;
                if (!BW) {
                    float mx = 0.f;
#pragma unroll
                    for (int w = 0; w < GW; ++w) {
                        const float4 v = reinterpret_cast<const float4 *>(sm.hmx[grp][w])[hg];
                        mx = fmaxf(mx, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
                    }
                    sh = act_shift(mx);
                }
                const float p = pow2i(sh);
                if (wq == 0 && hc == 0 && hl)
                    sm.hshift[grp][b][hg] = sh;
                uint2 *hf = reinterpret_cast<uint2 *>(sm.hbuf[grp][b]);
#pragma unroll
                for (int j = 0; j < HJ; ++j) {
                    // all 32 lanes: lanes 4T.. hold zeros (their src words are 0)
                    const int e = (wq + GW * j) * 32 + lane;
                    hf[e] = BW ? make_uint2(src0[j], src1[j])
                               : make_uint2(bf16x2_to_f16x2_scaled(src0[j], p), bf16x2_to_f16x2_scaled(src1[j], p));
                }
                named_barrier_sync(1 + grp, GW * 32);
                bfrag = hf;
            }

            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            {
                const int np = nparts(u);
                for (int p = 0; p < np; ++p) {
                    const int rs = ccount % RING;
                    mbar_wait_bounded(&sm.full[warp][rs], (ccount / RING) & 1, flag);
                    if (BW)
                        bf16_stage(sm.ring[warp][rs], bfrag, 4 * (part0(u) + p), lane, acc);
                    else
                        mma_stage(sm.ring[warp][rs], bfrag, 16 * (part0(u) + p), lane, acc);
                    __syncwarp();
                    ++ccount;
                    issue_ahead(ccount + RING);
                }
            }

            const int g = lane >> 2, c = lane & 3;
            bool gu_writer = !u.down;
            if (!u.down) {
                // The four K quarters of the band are added in warp order by the
                // unit's writer, warp k % 4; the other three hand over their
                // partials through kred[k & 1] and go on.  A partial buffer is
                // refilled only after its previous writer has read it.
                const int wr = k & (GW - 1), par = k & 1;
                gu_writer = (wq == wr);
                // Every warp, the writer too, first waits until unit k - 2's
                // writer has read kred[par]: then all of unit k - 2's handovers
                // have landed, so neither barrier can be a phase behind when a
                // parity wait below looks at it (a parity wait cannot tell phase
                // j from phase j - 2).
                if (k >= 2)
                    mbar_wait_bounded(&sm.kempty[grp][par], ((k >> 1) - 1) & 1, flag);
                if (!gu_writer) {
                    sm.kred[grp][par][(wq - wr + GW - 1) & (GW - 1)][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&sm.kfull[grp][par]);
                } else {
                    mbar_wait_bounded(&sm.kfull[grp][par], (k >> 1) & 1, flag);
                    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < GW; ++q) {
                        const float4 v = (q == wr) ? make_float4(acc[0], acc[1], acc[2], acc[3])
                                                   : sm.kred[grp][par][(q - wr + GW - 1) & (GW - 1)][lane];
                        if (q == 0) {
                            sum = v;
                        } else {
                            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                        }
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&sm.kempty[grp][par]);
                    acc[0] = sum.x; acc[1] = sum.y; acc[2] = sum.z; acc[3] = sum.w;
                }
            }
            if (gu_writer && BW) {
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int t = 2 * c + tt;
                    if (t < T) {
                        const float gv = acc[tt], uv = acc[2 + tt];
                        hglob[((size_t)u.slot * MAXT + t) * H_PITCH + u.band * 8 + g] =
                            __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
                    }
                }
                count_now_if_last_gu(k, u.slot);
                publish(&sm.gu_done[grp][wq], ++n_written);
            } else if (gu_writer) {
                // SiLU*up for h rows 8 * band + g
                const float ts = (u.slot < a.n_shared) ? __ldg(a.s_ts13 + u.slot)
                                                       : __ldg(a.r_ts13 + sm.slot_expert[u.slot]);
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int t = 2 * c + tt;
                    if (t < T) {
                        const float f = ts * pow2i(-sm.xshift[t]);
                        const float gv = acc[tt] * f, uv = acc[2 + tt] * f;
                        hglob[((size_t)u.slot * MAXT + t) * H_PITCH + u.band * 8 + g] =
                            __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
                    }
                }
                count_now_if_last_gu(k, u.slot);
                publish(&sm.gu_done[grp][wq], ++n_written);
            } else if (u.down) {
                // down: one band per warp, x routing weight x tensor scale x 2^-shift
                const float ts = BW ? 1.0f
                                    : (u.slot < a.n_shared) ? __ldg(a.s_ts2 + u.slot)
                                                            : __ldg(a.r_ts2 + sm.slot_expert[u.slot]);
                float *P = partials + ((size_t)u.slot * H + 16 * u.band) * MAXT;
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int t = 2 * c + tt;
                    if (t < T) {
                        const float f = sm.wts[u.slot][t] * ts * pow2i(-sm.hshift[grp][b][t]);
                        P[g * MAXT + t] = acc[tt] * f;
                        P[(g + 8) * MAXT + t] = acc[2 + tt] * f;
                    }
                }
                if (unit_id(k + 1) >= end_id && u.slot < n_slots - 1) {
                    // the group's last unit: nothing else to do, so count it here
                    __syncwarp();
                    if (lane == 0) {
                        fence_acq_rel_gpu();
                        red_relaxed_add(&band_cnt[u.band], 1u);
                    }
                }
                publish(&sm.dn_done[grp][wq], ++n_partials);
                if (u.slot == n_slots - 1)
                    combine_band(u.band);
                // the group's hbuf[b] is free once all four warps are done with it
                fence_proxy_async();   // the fragments were written in place; a bulk copy refills the buffer
                named_barrier_sync(1 + grp, GW * 32);
                if (lead_thread)
                    st_release_cta(&sm.hrel[grp], (uint32_t)(k - k_down0 + 1));
            }
        }
    }

    // ---- CTA 0 re-arms the counters for the next call once every CTA has
    // stopped reading them (each sync warp counts itself in ctrl[4] after its
    // last h copy, long after its logits were read; the band counters are
    // re-armed by the warps that add the bands up) ----
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (uint32_t it = 0; ld_acquire(&ctrl[4]) < gridDim.x; ++it) {
            if (it == SPIN_LIMIT) {
                atomicOr(flag, FLAG_TIMEOUT);
                return;
            }
            __nanosleep(64);
        }
        for (int s = 0; s < MAX_SLOTS; ++s)
            slot_cnt[s] = 0u;
        ctrl[4] = 0u;
        ctrl[5] = ltag;   // the next launch tags its logits ltag + 1
    }
}

size_t layer_smem_bytes() { return sizeof(FSmem); }

namespace {
PerDevice g_layer_attr;   // 1 + resident CTAs per SM, once the attributes are set
}

int layer_resident_ctas_per_sm()
{
    const int v = per_device(g_layer_attr, [](int) {
        const int smem = (int)sizeof(FSmem);
        if (cudaFuncSetAttribute(moe_layer_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(moe_layer_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess)
            return -1;
        int n0 = 0, n1 = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n0, moe_layer_kernel<false>, NT, smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, moe_layer_kernel<true>, NT, smem) != cudaSuccess)
            return -1;
        return 1 + (n0 < n1 ? n0 : n1);
    });
    return v > 0 ? v - 1 : -1;
}

cudaError_t launch_layer(const LayerArgs &a, int grid, cudaStream_t stream, bool pdl)
{
    if (layer_resident_ctas_per_sm() < 0)
        return cudaErrorUnknown;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = sizeof(FSmem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return a.bf16w ? cudaLaunchKernelEx(&cfg, moe_layer_kernel<true>, a)
                   : cudaLaunchKernelEx(&cfg, moe_layer_kernel<false>, a);
}

// After a call that gave up on a bounded wait, the workspace's counters may
// hold that call's partial counts and its launch tag may not have advanced
// (CTA 0 returns before re-arming them).  If the flag word shows a timeout,
// clear the counters and advance the tag, so that the next layer call
// ignores the stale tagged logits; the flag bits stay for the caller to read.
// Runs after the preceding kernel has finished (it waits on it first).
__global__ void __launch_bounds__(128) rearm_kernel(uint8_t *ws)
{
    griddep_launch();
    griddep_wait();
    const WsLayout L = ws_layout();
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(ws + L.ctrl);
    if ((__ldcg(&ctrl[0]) & FLAG_TIMEOUT) == 0u)
        return;
    uint32_t *slot_cnt = reinterpret_cast<uint32_t *>(ws + L.slot_cnt);
    uint32_t *band_cnt = reinterpret_cast<uint32_t *>(ws + L.band_cnt);
    for (int i = threadIdx.x; i < MAX_SLOTS; i += blockDim.x)
        slot_cnt[i] = 0u;
    for (int i = threadIdx.x; i < W2_BANDS; i += blockDim.x)
        band_cnt[i] = 0u;
    if (threadIdx.x == 0) {
        ctrl[1] = 0u;
        ctrl[4] = 0u;
        ctrl[5] = ctrl[5] + 1u;
    }
}

cudaError_t launch_rearm(uint8_t *ws, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rearm_kernel, ws);
}

}  // namespace moe

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
// One CTA per SM, 20 warps: 16 compute warps (each with a private ring of
// stage copies), two epilogue warps (they finish gate/up bands) and two h
// warps (they prepare the down projections' B operands).  Phases:
//  1. before waiting on the preceding kernel: router CTAs load their slice of
//     the router weights; in CTAs 0..63 the compute warps of band parity 0
//     start the bulk copy of their slice of one band of the shared expert
//     (it needs no routing); every tensor scale goes to shared memory;
//  2. x arrives in shared memory by bulk copies (in a stack, also the
//     previous layer's output: every CTA forms the residual and its RMSNorm);
//     CTAs 0..127 compute the fp32 logits of two experts each (CTA 128 those
//     of up to two expert sinks) and store each with the launch's tag in one
//     64-bit word; every compute warp turns its 256-column slice of x into
//     mma fragments held in registers;
//  3. every CTA reads the logits until each carries the launch's tag (a
//     reader that sees the tag sees the logit: no fence, no counter), takes
//     the top-6 of each token (one warp per token, identical in every CTA;
//     sink scores join the denominator) and builds the slot table: the shared
//     expert, then the distinct selected experts in ascending order, each
//     with its per-token routing weight;
//  4. the unit phase.  With U slots and G CTAs:
//       gate/up: the 64 U bands of W13 (16 rows each: 8 gate + 8 up rows),
//         slot-major, are dealt round-robin, CTA c taking bands c, c + G,
//         ...; within the CTA, band k goes to the 8 warps of parity k % 2,
//         warp q of them taking the band's 256-column slice q (the x
//         fragments of that slice never leave its registers).  The eight K
//         partials of a band meet in a shared-memory buffer; an epilogue
//         warp adds them in slice order, applies SiLU*up and stores h as
//         tagged 64-bit words (two bf16 values and the launch tag);
//       down: the 128 (U - 1) bands of W2 (16 rows) of the first U - 1 slots
//         are cut into G contiguous ranges (a range touches at most two
//         slots), and band b of the last slot goes to CTA b; within the CTA
//         the bands are dealt to the 16 warps round-robin, one warp per band
//         (all of its 512 columns).  The h warps read a slot's tagged h words
//         until every one carries the tag, scale each token by a power of two
//         into f16 fragments once for the whole CTA, and count themselves
//         done; each down partial goes out as tagged fp32 words;
//     NVFP4 gate/up bands arrive whole (one 18,432-byte bulk copy each) in
//     four band slots per parity group; each warp reads its slice there, and
//     the eighth warp done with a slot refills it with the group's next band.
//     Every compute warp streams its own down bands (4,608-byte copies)
//     through a ring that takes its share of its group's band slots once
//     their last bands are read (BF16: every stage through the warp's own
//     ring).  Slots complete in order on every CTA, so by the time a warp
//     reaches its down bands their h is normally ready;
//  5. CTA b < 128 writes out rows 16 b .. 16 b + 15: its compute warps read
//     every slot's tagged partials of the band, each warp summing every 16th
//     slot in order, then warp 0 adds the 16 sums in warp order and the
//     shared experts run ahead of the kernel (if any), and rounds once to
//     bf16 (deterministic, bit-identical between calls).
// NVFP4: the stages are decoded in registers (cvt.rn.f16x2.e2m1x2) straight
// into mma.sync A fragments.  BF16 (the W16A16 variant of the Flint page,
// section "From 1,096 kernels to 346": BF16 decode): a stage is 16 rows x 64
// columns copied by per-lane cp.async into a swizzled ring slot.
// Every wait is bounded and reports MOE_FLAG_WAIT_TIMEOUT instead of hanging.
#include "kernels.cuh"
#include "stage.cuh"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int FW = 16;                 // compute warps per CTA
constexpr int FT = FW * 32;            // compute threads
constexpr int EP_WARP = FW;            // warps 16, 17: gate/up epilogues (band parity 0, 1)
constexpr int HW_WARP = FW + 2;        // warps 18, 19: h fragments of the CTA's down slots (half of the steps each)
constexpr int NHB = 3;                 // h buffers: the two range slots and the last slot
constexpr int NT = FT + 128;           // threads per CTA (20 warps: a multiple of 4 keeps 96 registers a thread)
constexpr int RW = 4;                  // ring stages per compute warp (BF16)
constexpr int GBS = 4;                 // NVFP4: whole-band gate/up slots per band-parity group
constexpr int STG = 2 * SC_BYTES;      // 2304 bytes: two NVFP4 super-chunks (a BF16 stage uses 2048)
constexpr int GQ = 8;                  // 256-column slices of a gate/up band
constexpr int NB = 8;                  // gate/up reduction buffers (band k uses k % NB)
constexpr int XPITCH = H * 2 + 16;     // bytes per staged x row: rows 4 banks apart, so the fragment reads do not conflict
constexpr int ROUTER_CTAS = E / 2;     // 128 CTAs x 2 experts
constexpr int HS = I / 16;             // 32 k16 steps of the down GEMV
constexpr int HBUF = HS * 32 * 8;      // one slot's h as B fragments [step][lane] (uint2), 8 KB
// With at least 128 CTAs a CTA has at most ceil(64 * 49 / 128) = 25 gate/up
// bands and ceil(128 * 48 / 128) = 48 range down bands, and its down range
// touches at most two slots (hence three h buffers: two range slots and the
// last slot).

struct FSmem {
    // Stage memory.  BF16: per-warp rings of RW stages.  NVFP4: gate/up bands
    // move whole (one 18,432-byte copy per band: an SM completes only ~10
    // bulk copies per us whatever their size, so eight 2,304-byte slices
    // per band would cap the stream near 3.5 TB/s), into GBS slots per
    // band-parity group, and each warp reads its slice there; once its
    // group's gate/up bands are done, warp q's ring of RW down stages is
    // bytes [q, q + 1) * RW * STG of the group's slots.  Phase 2 stages x
    // (and delta) in the second half, which the unit phase writes first.
    union {
        uint8_t ring[FW][RW][STG];
        struct {
            uint8_t gband[2][GBS][W13_BAND_BYTES];
        } nv;
    };
    union {
        RouterRed rred;                // phase 2: the router's partial sums
        struct {
            float4 red[NB][GQ][32];    // gate/up K partials, [buffer][slice][lane]
            uint8_t hbuf[NHB][HBUF];   // h of a down slot as B fragments (f16 scaled, or bf16)
        } u;
    };
    uint64_t full[FW][RW];
    uint64_t gfull[2][GBS];            // NVFP4: a gate/up band slot holds its band
    uint32_t gdone[2][GBS];            // NVFP4: warps done with the slot's band (the eighth refills it)
    uint32_t sfree[2][GBS];            // NVFP4: the slot's last band has been read (down rings may use it)
    uint64_t xbar;
    int32_t sel[MAXT][TOPK];
    float selw[MAXT][TOPK];
    uint32_t bitmap[E / 32];
    int bcnt[E / 32];
    int n_slots;
    int32_t slot_expert[MAX_SLOTS];
    float wts[MAX_SLOTS][MAXT];
    int xshift[MAXT];
    float xinv[MAXT];                  // NVFP4: 2^-xshift[t]
    float ts13[MAX_SLOTS];             // tensor scales of the slots' W13 and W2 (NVFP4)
    float ts2[MAX_SLOTS];
    float all_ts13[E + MAX_SHARED];    // every expert's tensor scales, routed then shared (NVFP4)
    float all_ts2[E + MAX_SHARED];
    float sumsq[FW];
    int hshift[NHB][MAXT];
    uint64_t pfull[NB];                // a band's eight K partials are in buffer b
    uint64_t pempty[NB];               // the epilogue warp has read buffer b
    uint32_t hready[NHB];              // h warps done with the buffer (2 when ready)
    float4 dhalf[8][32];               // BF16: the second K half of a down band, per warp pair
    uint32_t dh_full[8];               // BF16: halves written by the pair's second warp
    uint32_t dh_empty[8];              // BF16: halves read by the pair's first warp
    float4 comb[FW][32];               // the final sum of band cta: per-warp sums of every 16th slot
    float hmax[NHB][2][MAXT];          // per h warp, each token's max |h| over its half of a slot
    float extw[MAX_EXT][MAXT];         // weight of each shared expert run ahead, per token
};

__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acquire.gpu;" ::: "memory"); }

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// 64-bit relaxed accesses at gpu scope (single-copy atomic)
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// The same with the B fragments of the warp's own 256-column K slice held in
// registers: xf[s] is k16 step s of the slice (one NVFP4 stage is the whole
// slice of one band).
__device__ __forceinline__ void mma_stage_r(const uint8_t *stage, const uint2 (&xf)[16], int lane, float acc[4])
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
                const uint2 b = xf[q * 8 + half * 4 + s];
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

// BF16: sub-stage SUB (64 columns) of the warp's slice, B fragments xf[4 SUB ..].
template <int SUB>
__device__ __forceinline__ void bf16_stage_r(const uint8_t *stage, const uint2 (&xf)[16], int lane, float acc[4])
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
        const uint2 b = xf[4 * SUB + s];
        mma_bf16_16816(acc, wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1], b.x, b.y);
    }
}

// Bounded wait until a shared-memory counter reaches v.
__device__ __forceinline__ bool smem_wait_geq(const uint32_t *p, uint32_t v, uint32_t *flag)
{
    for (uint32_t it = 0; it < SPIN_LIMIT; ++it) {
        if (ld_acquire_cta(p) >= v)
            return true;
        __nanosleep(20);
    }
    atomicOr(flag, FLAG_TIMEOUT);
    return false;
}

// Bounded wait until a global counter reaches v: relaxed polls (an acquire
// load costs about as much as a fence while the SM streams), then one
// acquire fence.
__device__ __forceinline__ bool gmem_wait_geq(const uint32_t *p, uint32_t v, uint32_t *flag)
{
    for (uint32_t it = 0; it < SPIN_LIMIT; ++it) {
        if (ld_relaxed_gpu(p) >= v) {
            fence_acquire_gpu();
            return true;
        }
        __nanosleep(32);
    }
    atomicOr(flag, FLAG_TIMEOUT);
    return false;
}

}  // namespace

template <bool BW>
__global__ void __launch_bounds__(NT, 1) moe_layer_kernel(LayerArgs a)
{
    static_assert(sizeof(RouterRed) <= sizeof(FSmem::u), "router partials fit the unit-phase buffers");
    static_assert((size_t)2 * MAXT * XPITCH <= sizeof(FSmem::ring) / 2, "x and delta fit the rings of warps 8..15");
    static_assert(sizeof(FSmem::nv) == sizeof(FSmem::ring) && GBS * W13_BAND_BYTES == (size_t)GQ * RW * STG,
                  "NVFP4: a group's band slots hold its eight warps' down rings");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    FSmem &sm = *reinterpret_cast<FSmem *>(smem_raw);

    const WsLayout L = ws_layout();
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(a.ws + L.ctrl);
    uint32_t *flag = ctrl;
    unsigned long long *tlogits = reinterpret_cast<unsigned long long *>(a.ws + L.tlogits);
    unsigned long long *htag = reinterpret_cast<unsigned long long *>(a.ws + L.htag);
    unsigned long long *ptag = reinterpret_cast<unsigned long long *>(a.ws + L.ptag);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & (GQ - 1), par = warp >> 3;   // compute warps: K slice and band parity
    const int T = a.T;
    const int blanes = 4 * T;
    const int G = (int)gridDim.x, cta = (int)blockIdx.x;

    if (lane == 0 && warp < FW) {
        for (int s = 0; s < RW; ++s)
            mbar_init(&sm.full[warp][s], BW ? 32 : 1);   // BF16: one cp.async arrival per lane
    }
    if (threadIdx.x < NB) {
        mbar_init(&sm.pfull[threadIdx.x], GQ);   // the band's eight K partials are in
        mbar_init(&sm.pempty[threadIdx.x], 1);   // the epilogue warp has read them
    }
    if (threadIdx.x < 2 * GBS) {
        mbar_init(&sm.gfull[threadIdx.x / GBS][threadIdx.x % GBS], 1);
        sm.gdone[threadIdx.x / GBS][threadIdx.x % GBS] = 0u;
    }
    if (threadIdx.x < 2 * GBS)
        sm.sfree[threadIdx.x / GBS][threadIdx.x % GBS] = 0u;
    if (threadIdx.x == 0)
        mbar_init(&sm.xbar, 1);
    if (lane == 0 && warp <= FW)
        fence_barrier_init();
    if (threadIdx.x < NHB)
        sm.hready[threadIdx.x] = 0u;
    if (threadIdx.x < 8) {
        sm.dh_full[threadIdx.x] = 0u;
        sm.dh_empty[threadIdx.x] = 0u;
    }
    __syncthreads();

    auto bank13 = [&](int slot) -> const uint8_t * {
        return (slot < a.n_shared) ? a.s_w13 + (size_t)slot * (BW ? W13_BYTES_BF : W13_BYTES)
                                   : a.r_w13 + (size_t)sm.slot_expert[slot] * (BW ? W13_BYTES_BF : W13_BYTES);
    };
    auto bank2 = [&](int slot) -> const uint8_t * {
        return (slot < a.n_shared) ? a.s_w2 + (size_t)slot * (BW ? W2_BYTES_BF : W2_BYTES)
                                   : a.r_w2 + (size_t)sm.slot_expert[slot] * (BW ? W2_BYTES_BF : W2_BYTES);
    };

    // ---- phase 1: work that needs nothing from the preceding kernel ----
    // CTA c's first gate/up band is band c of slot 0: the shared expert when
    // there is one.  Its copy into band slot 0 of parity group 0 starts now
    // (NVFP4; the slot table is not built yet, so the address is computed
    // directly).
    const bool pre_shared = !BW && a.n_shared > 0 && cta < W13_BANDS;
    if (pre_shared && threadIdx.x == 0) {
        mbar_arrive_expect_tx(&sm.gfull[0][0], W13_BAND_BYTES);
        bulk_g2s(sm.nv.gband[0][0], a.s_w13 + (size_t)cta * W13_BAND_BYTES, W13_BAND_BYTES, &sm.gfull[0][0]);
    }
    // every expert's tensor scales (NVFP4), for the slot table built later
    if (!BW) {
        for (int i = threadIdx.x; i < E + a.n_shared; i += NT) {
            sm.all_ts13[i] = i < E ? __ldg(a.r_ts13 + i) : __ldg(a.s_ts13 + (i - E));
            sm.all_ts2[i] = i < E ? __ldg(a.r_ts2 + i) : __ldg(a.s_ts2 + (i - E));
        }
    }
    // router CTAs: warp w of the 16 takes expert 2 * cta + w / 8, columns
    // [256 (w % 8), 256 (w % 8) + 256), eight per lane; CTA 128 takes the
    // router rows of the expert sinks (experts 256, 257)
    const int n_rows = E + a.n_sink;
    const bool router_warp = (cta < ROUTER_CTAS || (cta == ROUTER_CTAS && a.n_sink > 0)) && warp < FW;
    const int r_e = cta * 2 + (warp >> 3);
    const int r_k8 = warp & 7;
    uint4 wv = make_uint4(0u, 0u, 0u, 0u);
    if (router_warp && r_e < n_rows)
        wv = ldg_nc_v4(a.wr + (size_t)r_e * H + 256 * r_k8 + 8 * lane);

    griddep_wait();      // x is written by the preceding kernel; the counters are re-armed
    griddep_launch();    // the next kernel may start its own phase 1
    // this launch's tag on the logits (never 0, the value a zeroed workspace holds)
    const uint32_t ltag = __ldcg(&ctrl[5]) + 1u;

    // ---- phase 2: x -> shared memory; router logits | activation fragments ----
    // T rows of XPITCH bytes each, free until the unit phase; lane t of warp 0
    // copies row t (several issuing threads: one thread issues bulk copies
    // only about every 200 ns)
    uint8_t *xs = &sm.ring[8][0][0];
    uint8_t *ds = xs + MAXT * XPITCH;  // pre-norm: the previous layer's output
    const bool has_delta = a.prenorm && a.delta != nullptr;
    if (warp == 0) {
        if (lane == 0)
            mbar_arrive_expect_tx(&sm.xbar, (uint32_t)(T * H * 2) * (has_delta ? 2u : 1u));
        __syncwarp();
        if (lane < T)
            bulk_g2s(xs + lane * XPITCH, a.x + (size_t)lane * H, (uint32_t)(H * 2), &sm.xbar);
        else if (has_delta && lane >= MAXT && lane < MAXT + T)
            bulk_g2s(ds + (lane - MAXT) * XPITCH, a.delta + (size_t)(lane - MAXT) * H, (uint32_t)(H * 2),
                     &sm.xbar);
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
                const int idx = t * (XPITCH / 16) + half * (H / 16) + 32 * i + lane;
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
                const int idx = t * (XPITCH / 16) + half * (H / 16) + 32 * i + lane;
                const int gidx = t * (H / 8) + half * (H / 16) + 32 * i + lane;
                uint4 n = vv[i];
                uint32_t *nw = &n.x;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat16 lo = __float2bfloat16_rn(bf16_bits_to_float(nw[q] & 0xFFFFu) * rinv);
                    const __nv_bfloat16 hi = __float2bfloat16_rn(bf16_bits_to_float(nw[q] >> 16) * rinv);
                    nw[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
                }
                xv[idx] = n;   // (followed by fence_proxy_async below: the rings are refilled by bulk copies)
                if (blockIdx.x == 0) {
                    if (a.resid_out)
                        reinterpret_cast<uint4 *>(a.resid_out)[gidx] = vv[i];
                    if (a.xn_out)
                        reinterpret_cast<uint4 *>(a.xn_out)[gidx] = n;
                }
            }
        }
        fence_proxy_async();
        __syncthreads();
    }

    if (router_warp) {
        float acc[MAXT];
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
            acc[t] = 0.0f;
            if (t < T) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xs + (size_t)t * XPITCH + 2 * (256 * r_k8 + 8 * lane));
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    acc[t] = fmaf(bf16_bits_to_float(xw[qq] & 0xFFFFu), bf16_bits_to_float(ww[qq] & 0xFFFFu), acc[t]);
                    acc[t] = fmaf(bf16_bits_to_float(xw[qq] >> 16), bf16_bits_to_float(ww[qq] >> 16), acc[t]);
                }
            }
        }
        float logit;
        // each logit carries the launch tag in the same 64-bit word, so a
        // reader that sees the tag sees the logit: no fence, no counter
        if (router_reduce(acc, (int)threadIdx.x, T, sm.rred, 5, &logit) && cta * 2 + (int)threadIdx.x / MAXT < n_rows)
            st_relaxed_u64(&tlogits[(threadIdx.x % MAXT) * LE + cta * 2 + threadIdx.x / MAXT],
                           ((unsigned long long)ltag << 32) | __float_as_uint(logit));
        fence_proxy_async();   // these generic writes precede the bulk copies of h into the same buffer
    }
    // x -> the B fragments of this warp's 256-column slice q, in registers:
    // entry s is k16 step 16 q + s; lane l < 4T holds token l / 4 (zeros
    // above).  NVFP4: f16, each token's row scaled by the power of two of its
    // max |x| (found first, one warp per token).  BF16: bf16 in the permuted
    // column order of bf16_bcol.
    uint2 xf[16];
    if (warp < FW) {
        const uint32_t *xw = reinterpret_cast<const uint32_t *>(xs);
        const int g = lane >> 2, c = lane & 3;
        float p = 1.0f;
        if (!BW) {
            if (warp < T) {
                const uint4 *row = reinterpret_cast<const uint4 *>(xs + (size_t)warp * XPITCH);
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
                if (lane == 0) {
                    sm.xshift[warp] = act_shift(m);
                    sm.xinv[warp] = pow2i(-act_shift(m));
                }
            }
            named_barrier_sync(6, FT);
            if (lane < blanes)
                p = pow2i(sm.xshift[g]);
        }
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const int step = 16 * q + s;
            uint2 v = make_uint2(0u, 0u);   // lanes 4T.. carry no token
            if (lane < blanes) {
                if (BW) {
                    const int w0 = g * (XPITCH / 4) + bf16_bcol(step, c) / 2;
                    v = make_uint2(xw[w0], xw[w0 + 1]);
                } else {
                    const int w0 = g * (XPITCH / 4) + 8 * step + c;
                    v = make_uint2(bf16x2_to_f16x2_scaled(xw[w0], p), bf16x2_to_f16x2_scaled(xw[w0 + 4], p));
                }
            }
            xf[s] = v;
        }
    }

    // ---- phase 3: routing (every CTA, identically) ----
    for (int i = threadIdx.x; i < MAX_SLOTS * MAXT; i += FT)
        sm.wts[i / MAXT][i % MAXT] = 0.0f;
    if (threadIdx.x < E / 32)
        sm.bitmap[threadIdx.x] = 0u;

    __syncthreads();
    if (warp < T) {
        // the token's 256 logits (and its sink logits, lanes < n_sink),
        // re-read until every one carries this launch's tag
        const unsigned long long *row = tlogits + warp * LE;
        float v[8], sv = 0.0f;
        bool have = false;
        for (uint32_t it = 0;; ++it) {
            have = true;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const unsigned long long w = ld_relaxed_u64(row + lane + 32 * m);
                v[m] = __uint_as_float((uint32_t)w);
                have = have && (uint32_t)(w >> 32) == ltag;
            }
            if (lane < a.n_sink) {
                const unsigned long long w = ld_relaxed_u64(row + E + lane);
                sv = __uint_as_float((uint32_t)w);
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
        float wt, swt;
        bool bad;
        warp_route_values_t<true>(v, lane, ex, wt, bad, sv, a.n_sink, swt);
        if (lane < TOPK) {
            sm.sel[warp][lane] = ex;
            sm.selw[warp][lane] = wt;
            atomicOr(&sm.bitmap[ex >> 5], 1u << (ex & 31));
        }
        // the shared experts run ahead: a sink's weight, else 1
        if (lane < a.n_ext)
            sm.extw[lane][warp] = a.n_sink ? swt : 1.0f;
        if (blockIdx.x == 0) {
            if (bad && lane == 0)
                atomicOr(flag, FLAG_NONFINITE);
            if (lane < TOPK) {
                reinterpret_cast<int32_t *>(a.ws + L.topk_idx)[warp * TOPK + lane] = ex;
                reinterpret_cast<float *>(a.ws + L.topk_w)[warp * TOPK + lane] = wt;
            }
            if (lane < a.n_ext)
                reinterpret_cast<float *>(a.ws + L.sinkw)[warp * MAX_EXT + lane] = a.n_sink ? swt : 1.0f;
            if (a.r_idx) {
                const int tg = a.t0 + warp;
                if (lane < TOPK) {
                    a.r_idx[tg * TOPK + lane] = ex;
                    a.r_w[tg * TOPK + lane] = wt;
                }
#pragma unroll
                for (int mm = 0; mm < 8; ++mm)
                    a.r_logits[(size_t)tg * E + lane + 32 * mm] = v[mm];
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
    __syncthreads();
    if (!BW && threadIdx.x < (unsigned)sm.n_slots) {
        const int sl = threadIdx.x;
        const int ie = sl < a.n_shared ? E + sl : sm.slot_expert[sl];
        sm.ts13[sl] = sm.all_ts13[ie];
        sm.ts2[sl] = sm.all_ts2[ie];
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


    // ---- phase 4: the units ----
    const int U = n_slots;
    // gate/up: CTA band k is global band cta + G k (slot-major: slot gb / 64)
    const int gu_total = W13_BANDS * U;
    const int n_gu_cta = cta < gu_total ? (gu_total - cta + G - 1) / G : 0;
    // down: the first U - 1 slots' bands in G contiguous ranges, and band
    // cta of the last slot (CTA down band j = n_rng for it)
    const long rng_total = (long)W2_BANDS * (U - 1);
    const int d0 = (int)(rng_total * cta / G), d1 = (int)(rng_total * (cta + 1) / G);
    const int n_rng = d1 - d0;
    const bool has_last = cta < W2_BANDS;
    const int n_dn_cta = n_rng + (has_last ? 1 : 0);
    const int s_first = d0 / W2_BANDS;          // h buffer 0 (and 1 for s_first + 1); buffer 2: the last slot
    auto dn_band = [&](int j, int &slot, int &band, int &hb) {
        if (j < n_rng) {
            const int db = d0 + j;
            slot = db / W2_BANDS;
            band = db % W2_BANDS;
            hb = slot - s_first;
        } else {
            slot = U - 1;
            band = cta;
            hb = 2;
        }
    };

    if (warp == EP_WARP || warp == EP_WARP + 1) {
        // ---- the epilogue warps: the gate/up bands' h ----
        // Epilogue warp p takes the CTA's gate/up bands k = p, p + 2, ... in
        // order: once buffer k % NB holds band k's eight K partials it adds
        // them in slice order, frees the buffer, applies SiLU*up (NVFP4:
        // times the tensor scale and the token's inverse power of two) and
        // stores h with the launch tag in every 64-bit word (two bf16 values
        // of one token per word), so a reader that sees the tag sees the
        // values: no fence, no counter.
        const int p = warp - EP_WARP;
        const int g = lane >> 2, c = lane & 3;
#pragma unroll 1
        for (int k = p; k < n_gu_cta; k += 2) {
            const int b = k % NB;
            if (lane == 0)
                mbar_wait_bounded(&sm.pfull[b], (uint32_t)(k / NB) & 1u, flag);
            __syncwarp();   // lane 0 saw the partials complete; the others read after it
            float4 sum = sm.u.red[b][0][lane];
#pragma unroll
            for (int qq = 1; qq < GQ; ++qq) {
                const float4 v = sm.u.red[b][qq][lane];
                sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.pempty[b]);
            const int gb = cta + G * k, slot = gb / W13_BANDS, band = gb % W13_BANDS;
            const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
                const int t = 2 * c + tt;
                // h row 8 band + g of token t (bf16 bits); the lane of row g + 1
                // hands its value down, and the even rows store the pair
                uint32_t hb = 0u;
                if (t < T) {
                    const float f = BW ? 1.0f : sm.ts13[slot] * sm.xinv[t];
                    const float gv = sv[tt] * f, uv = sv[2 + tt] * f;
                    hb = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv));
                }
                const uint32_t ob = __shfl_down_sync(0xFFFFFFFFu, hb, 4);
                if (t < T && (g & 1) == 0)
                    st_relaxed_u64(&htag[(((size_t)slot * W13_BANDS + band) * MAXT + t) * 4 + (g >> 1)],
                                   ((unsigned long long)ltag << 32) | (ob << 16) | hb);
            }
        }
    } else if (warp >= HW_WARP) {
        // ---- the h warps: h of the CTA's down slots as B fragments ----
        // Buffers: the first range slot (r = 0), the second (r = 1, when the
        // range reaches it) and the last slot (r = 2, CTAs below 128), in
        // that order.  h warp hw takes k16 steps 16 hw .. 16 hw + 15 of each:
        // lane (g, c) needs, for step s, rows 16 s + 2 c, +1 (band 2 s) and
        // 16 s + 8 + 2 c, +1 (band 2 s + 1) of token g, 32 tagged words in
        // all.  It probes the tag of one pending word, then reads all 32
        // words in one batch, until every one carries this launch's tag.
        // NVFP4 then scales each token by the power of two of its max |h|
        // (over both halves: the two warps exchange their maxima) into f16;
        // BF16 permutes the pairs into the column order of bf16_bcol.  The
        // fragments go to the slot's buffer, [k16 step][lane], zeros in
        // lanes 4T..; hready[r] counts the two warps done.  h warp 0 first
        // counts this CTA in ctrl[4] (every thread of the CTA has read the
        // launch tag by now; CTA 0 advances the tag once all CTAs are
        // counted).
        const int hw = warp - HW_WARP;
        if (hw == 0 && lane == 0)
            red_release_add(&ctrl[4], 1u);
        const int hg = lane >> 2, hc = lane & 3;
        const bool hl = lane < blanes;
        constexpr int HH = HS / 2;
        uint2 *hfa = nullptr;
#pragma unroll 1
        for (int r = 0; r < NHB; ++r) {
            const int hslot = r == 0 ? s_first : r == 1 ? s_first + 1 : U - 1;
            const bool hneed = r == 0   ? n_rng > 0
                               : r == 1 ? n_rng > 0 && (d1 - 1) / W2_BANDS == s_first + 1
                                        : has_last;
            if (!hneed)
                continue;
            // word j (0..31): band 32 hw + j, i.e. step 16 hw + j / 2, .x (j even) or .y
            const unsigned long long *src =
                htag + (((size_t)hslot * W13_BANDS + 2 * HH * hw) * MAXT + hg) * 4 + hc;
            uint32_t vx[HH], vy[HH];
            for (uint32_t it = 0;; ++it) {
                bool ok = true;
                // the probe: this lane's last word (the band written latest in
                // the CTAs' band order is the likeliest to be missing).  The
                // last slot, whose h gates the end of the launch and which
                // these warps usually wait for, is read whole on every poll
                // instead (one L2 round trip fewer once it is complete).
                if (hl && r != 2)
                    ok = ld_relaxed_u32(reinterpret_cast<const uint32_t *>(src + (size_t)(2 * HH - 1) * MAXT * 4) +
                                        1) == ltag;
                if (__all_sync(0xFFFFFFFFu, ok)) {
                    unsigned long long w[2 * HH];
#pragma unroll
                    for (int j = 0; j < 2 * HH; ++j)
                        w[j] = hl ? ld_relaxed_u64(src + (size_t)j * MAXT * 4) : ((unsigned long long)ltag << 32);
#pragma unroll
                    for (int j = 0; j < 2 * HH; ++j) {
                        ok = ok && (uint32_t)(w[j] >> 32) == ltag;
                        if (j & 1)
                            vy[j >> 1] = hl ? (uint32_t)w[j] : 0u;
                        else
                            vx[j >> 1] = hl ? (uint32_t)w[j] : 0u;
                    }
                    if (__all_sync(0xFFFFFFFFu, ok))
                        break;
                }
                if (it == SPIN_LIMIT) {
                    if (lane == 0)
                        atomicOr(flag, FLAG_TIMEOUT);
                    break;
                }
                __nanosleep(64);
            }
            hfa = reinterpret_cast<uint2 *>(sm.u.hbuf[r]);
            int sh = 0;
            if (!BW) {
                __nv_bfloat162 m2 = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
                for (int st = 0; st < HH; ++st) {
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(vx[st])));
                    m2 = __hmax2(m2, __habs2(u32_as_bf162(vy[st])));
                }
                float mx = fmaxf(__low2float(m2), __high2float(m2));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
                if (hc == 0 && hl)
                    sm.hmax[r][hw][hg] = mx;
                named_barrier_sync(8, 64);   // the two h warps
                if (hl)
                    mx = fmaxf(sm.hmax[r][0][hg], sm.hmax[r][1][hg]);
                sh = act_shift(mx);
                const float pw = pow2i(sh);
#pragma unroll
                for (int st = 0; st < HH; ++st)
                    hfa[(HH * hw + st) * 32 + lane] =
                        make_uint2(bf16x2_to_f16x2_scaled(vx[st], pw), bf16x2_to_f16x2_scaled(vy[st], pw));
            } else {
                // Lane (g, c) holds columns 16 s + 2 c, +1 (vx) and 16 s + 8 +
                // 2 c, +1 (vy) of the steps s of its half.  Step st needs the
                // pairs starting at column bf16_bcol(st, c) and 2 after it: for
                // every c they come from lanes (g, 2 (st & 1)) and
                // (g, 2 (st & 1) + 1), from vx (c even) or vy (c odd) of step
                // b16 (c < 2) or b16 + 1 (c >= 2); a step's pairs stay within
                // its half (b16 + 1 < 16 (hw + 1)).
#pragma unroll
                for (int st = 0; st < HH; ++st) {
                    // HH * hw is a multiple of 4, so the register index and the
                    // source lane depend on st alone: written that way they are
                    // compile-time constants (vx, vy stay in registers)
                    const int gst = HH * hw + st;
                    const int b16 = 4 * (st >> 2) + 2 * ((st & 3) >> 1);
                    const int sl = 4 * hg + 2 * (st & 1);
                    const uint32_t a00 = __shfl_sync(0xFFFFFFFFu, vx[b16], sl);
                    const uint32_t a01 = __shfl_sync(0xFFFFFFFFu, vy[b16], sl);
                    const uint32_t a10 = __shfl_sync(0xFFFFFFFFu, vx[b16 + 1], sl);
                    const uint32_t a11 = __shfl_sync(0xFFFFFFFFu, vy[b16 + 1], sl);
                    const uint32_t b00 = __shfl_sync(0xFFFFFFFFu, vx[b16], sl + 1);
                    const uint32_t b01 = __shfl_sync(0xFFFFFFFFu, vy[b16], sl + 1);
                    const uint32_t b10 = __shfl_sync(0xFFFFFFFFu, vx[b16 + 1], sl + 1);
                    const uint32_t b11 = __shfl_sync(0xFFFFFFFFu, vy[b16 + 1], sl + 1);
                    const uint32_t x0 = hc == 0 ? a00 : hc == 1 ? a01 : hc == 2 ? a10 : a11;
                    const uint32_t x1 = hc == 0 ? b00 : hc == 1 ? b01 : hc == 2 ? b10 : b11;
                    hfa[gst * 32 + lane] = hl ? make_uint2(x0, x1) : make_uint2(0u, 0u);
                }
            }
            if (hw == 0 && hc == 0 && hl)
                sm.hshift[r][hg] = sh;
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                atomicAdd(&sm.hready[r], 1u);
            }
        }
    } else {
        // ---- a compute warp ----
        // its gate/up bands: CTA bands k = par, par + 2, ... (slice q each);
        // its down bands: CTA down bands j = jw, jw + 16, ... (the parity-1
        // warps start the dealing when the CTA has an odd number of gate/up
        // bands, so that they, with one band fewer, take the first ones)
        const int n_gub = n_gu_cta > par ? (n_gu_cta - par + 1) / 2 : 0;
        const int jw = (warp - ((n_gu_cta & 1) ? 8 : 0) + 16) & 15;
        // BF16: a down band (eight 64-column stages) is split between the
        // warps jw and jw + 8 (four stages each, all of them in the ring at
        // once), which take the bands jw % 8, jw % 8 + 8, ...
        const int jp = BW ? (jw & 7) : jw, dh = BW ? (jw >> 3) : 0, jstride = BW ? 8 : 16;
        const int n_dnb = n_dn_cta > jp ? (n_dn_cta - jp + jstride - 1) / jstride : 0;
        constexpr int SPG = BW ? 4 : 1;   // stages per gate/up slice
        constexpr int SPD = BW ? 4 : 2;   // stages per down band (BF16: per half band)
        constexpr int RWX = RW;            // the warp's ring stages
        // the warp's own ring carries its gate/up slices (BF16) and its down
        // bands; NVFP4 gate/up bands come whole through the group's band slots
        const int n_gu_ring = BW ? n_gub * SPG : 0;
        const int n_stages = n_gu_ring + n_dnb * SPD;
        auto wring = [&](int rs) -> uint8_t * {
            return BW ? sm.ring[warp][rs] : &sm.nv.gband[par][0][0] + (size_t)(q * RW + rs) * STG;
        };

        // stage i of this warp into ring slot rs
        auto issue_stage = [&](int rs, int i) {
            uint64_t *bar = &sm.full[warp][rs];
            const uint8_t *src;
            if (i < n_gu_ring) {
                const int k = par + 2 * (i / SPG), sub = i % SPG;
                const int gb = cta + G * k, slot = gb / W13_BANDS, band = gb % W13_BANDS;
                if (BW) {
                    // rows: 8 gate rows 8 band.. and the matching up rows;
                    // columns 256 q + 64 sub ..; lane 2r + h copies bytes
                    // [64 h, 64 h + 64) of row r
                    const int r = lane >> 1, h = lane & 1;
                    const int row = r < 8 ? 8 * band + r : I + 8 * band + (r - 8);
                    src = bank13(slot) + ((size_t)row * H + 256 * q + 64 * sub) * 2 + 64 * h;
                } else {
                    src = bank13(slot) + (size_t)band * W13_BAND_BYTES + (size_t)q * STG;
                }
            } else {
                const int d = i - n_gu_ring;
                const int j = jp + jstride * (d / SPD), sub = d % SPD + SPD * dh;
                int slot, band, hb;
                dn_band(j, slot, band, hb);
                if (BW) {
                    const int r = lane >> 1, h = lane & 1;
                    src = bank2(slot) + ((size_t)(16 * band + r) * I + 64 * sub) * 2 + 64 * h;
                } else {
                    src = bank2(slot) + (size_t)band * W2_BAND_BYTES + (size_t)sub * STG;
                }
            }
            if (BW) {
                const int r = lane >> 1, h = lane & 1;
                uint8_t *dst = wring(rs) + r * 128;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    cp_async_cg16(dst + 16 * ((4 * h + u) ^ (4 * (r & 1))), src + 16 * u);
                cp_async_arrive(bar);
                return;
            }
            if (lane != 0)
                return;
            mbar_arrive_expect_tx(bar, STG);
            bulk_g2s(wring(rs), src, STG, bar);
        };
        int ic = 0;                                  // next stage to consume
        int ii = 0;                                  // next stage to issue
        auto issue_ahead = [&]() {
            while (ii < n_stages && ii < ic + RWX) {
                const int rs = ii % RWX;
                const int d = ii - n_gu_ring;
                if (!BW && d >= 0 && (d & 1) == 0 && rs + 1 < RWX && ii + 1 < ic + RWX) {
                    // both stages of an NVFP4 down band into adjacent slots by
                    // one copy; the second slot's barrier completes at once
                    // (its data is covered by the first slot's)
                    if (lane == 0) {
                        int slot, band, hb;
                        dn_band(jp + jstride * (d >> 1), slot, band, hb);
                        mbar_arrive_expect_tx(&sm.full[warp][rs], 2 * STG);
                        bulk_g2s(wring(rs), bank2(slot) + (size_t)band * W2_BAND_BYTES, 2 * STG,
                                 &sm.full[warp][rs]);
                        mbar_arrive(&sm.full[warp][rs + 1]);
                    }
                    ii += 2;
                    continue;
                }
                issue_stage(rs, ii);
                ++ii;
            }
        };
        auto wait_stage = [&]() -> const uint8_t * {
            const int rs = ic % RWX;
            mbar_wait_bounded(&sm.full[warp][rs], (ic / RWX) & 1, flag);
            return wring(rs);
        };
        auto next_stage = [&]() {
            __syncwarp();
            ++ic;
            issue_ahead();
        };
        if (BW)
            issue_ahead();
        const int g = lane >> 2, c = lane & 3;

        // NVFP4: band bi of this parity group (CTA band par + 2 bi) into the
        // group's slot bi % GBS, one copy of the whole band
        auto issue_band = [&](int bi) {
            const int k = par + 2 * bi;
            const int gb = cta + G * k, slot = gb / W13_BANDS, band = gb % W13_BANDS;
            uint64_t *bar = &sm.gfull[par][bi % GBS];
            mbar_arrive_expect_tx(bar, W13_BAND_BYTES);
            bulk_g2s(sm.nv.gband[par][bi % GBS], bank13(slot) + (size_t)band * W13_BAND_BYTES, W13_BAND_BYTES, bar);
        };
        if (!BW && q == 0 && lane == 0) {
            // the group's first GBS bands (group 0's first: already in flight
            // when it is the shared expert's)
            for (int bi = (par == 0 && pre_shared) ? 1 : 0; bi < GBS && bi < n_gub; ++bi)
                issue_band(bi);
        }

        // ---- gate/up slices ----
#pragma unroll 1
        for (int bi = 0; bi < n_gub; ++bi) {
            const int k = par + 2 * bi;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (BW) {
                bf16_stage_r<0>(wait_stage(), xf, lane, acc);
                next_stage();
                bf16_stage_r<1>(wait_stage(), xf, lane, acc);
                next_stage();
                bf16_stage_r<2>(wait_stage(), xf, lane, acc);
                next_stage();
                bf16_stage_r<3>(wait_stage(), xf, lane, acc);
                next_stage();
            } else {
                // slice q of the band in slot bi % GBS; the eighth warp done
                // with the slot refills it with the group's band bi + GBS (its
                // reads are ordered before the copy by the fence and the count)
                const int sl = bi % GBS;
                mbar_wait_bounded(&sm.gfull[par][sl], (uint32_t)(bi / GBS) & 1u, flag);
                mma_stage_r(sm.nv.gband[par][sl] + (size_t)q * STG, xf, lane, acc);
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    if (atomicAdd(&sm.gdone[par][sl], 1u) == GQ - 1) {
                        sm.gdone[par][sl] = 0u;
                        __threadfence_block();
                        if (bi + GBS < n_gub)
                            issue_band(bi + GBS);
                        else
                            st_release_cta(&sm.sfree[par][sl], 1u);   // the slot's last band is read
                    }
                }
            }
            // the band's eight K partials meet in buffer k % NB (its previous
            // use, band k - NB, must have been read by the epilogue warp)
            const int b = k % NB, u = k / NB;
            if (u > 0)
                mbar_wait_bounded(&sm.pempty[b], (uint32_t)(u - 1) & 1u, flag);
            sm.u.red[b][q][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.pfull[b]);
        }

        if (!BW) {
            // the warp's down ring lives in band slot q / 2 of its group: wait
            // until the slot's last band has been read by all eight warps (a
            // slot the group never used is free)
            const int ds = q * RW * STG / (int)W13_BAND_BYTES;
            if (lane == 0 && ds < n_gub)
                smem_wait_geq(&sm.sfree[par][ds], 1u, flag);
            __syncwarp();
            issue_ahead();
        }

        // ---- down bands ----
#pragma unroll 1
        for (int m = 0; m < n_dnb; ++m) {
            const int j = jp + jstride * m;
            int slot, band, hb;
            dn_band(j, slot, band, hb);
            if (lane == 0)
                smem_wait_geq(&sm.hready[hb], 2u, flag);   // both h warps
            __syncwarp();
            const uint2 *bfrag = reinterpret_cast<const uint2 *>(sm.u.hbuf[hb]);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int sub = 0; sub < SPD; ++sub) {
                if (BW)
                    bf16_stage(wait_stage(), bfrag, 4 * (sub + SPD * dh), lane, acc);
                else
                    mma_stage(wait_stage(), bfrag, 16 * sub, lane, acc);
                next_stage();
            }
            if (BW) {
                // the pair's two K halves meet in shared memory: the second
                // warp hands its half over, the first adds it to its own
                // (first half + second half, always in that order)
                if (dh == 1) {
                    if (lane == 0)
                        smem_wait_geq(&sm.dh_empty[jp], (uint32_t)m, flag);
                    __syncwarp();
                    sm.dhalf[jp][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    __syncwarp();
                    if (lane == 0)
                        st_release_cta(&sm.dh_full[jp], (uint32_t)m + 1u);
                    continue;
                }
                if (lane == 0)
                    smem_wait_geq(&sm.dh_full[jp], (uint32_t)m + 1u, flag);
                __syncwarp();
                const float4 o = sm.dhalf[jp][lane];
                acc[0] += o.x; acc[1] += o.y; acc[2] += o.z; acc[3] += o.w;
                __syncwarp();
                if (lane == 0)
                    st_release_cta(&sm.dh_empty[jp], (uint32_t)m + 1u);
            }
            // one band per warp, times the routing weight, the tensor scale and
            // the token's inverse power of two
            const float ts = BW ? 1.0f : sm.ts2[slot];
            // tagged partials: (launch tag, fp32) per row and token
            unsigned long long *P = ptag + ((size_t)slot * W2_BANDS + band) * 16 * MAXT;
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
                const int t = 2 * c + tt;
                if (t < T) {
                    const float f = sm.wts[slot][t] * ts * pow2i(-sm.hshift[hb][t]);
                    const unsigned long long tag = (unsigned long long)ltag << 32;
                    st_relaxed_u64(&P[g * MAXT + t], tag | __float_as_uint(acc[tt] * f));
                    st_relaxed_u64(&P[(g + 8) * MAXT + t], tag | __float_as_uint(acc[2 + tt] * f));
                }
            }
        }
        // ---- the out rows of band cta (CTA b < 128): every slot's partial
        // of the band, once each carries this launch's tag.  Warp w adds the
        // slots w, w + 16, w + 32 in order (one round trip of loads), then
        // warp 0 adds the 16 warp sums in warp order: a fixed order, so the
        // result is the same from call to call.  Lane (r, th): row r, tokens
        // 4 th .. 4 th + 3.
        if (has_last) {
            const int band = cta;
            const int r = lane >> 1, th = lane & 1;
            const unsigned long long *srcp = ptag + ((size_t)band * 16 + r) * MAXT + 4 * th;
            float s4[4];
            for (uint32_t it = 0;; ++it) {
                bool ok = true;
                s4[0] = s4[1] = s4[2] = s4[3] = 0.f;
                constexpr int PER_WARP = (MAX_SLOTS + FW - 1) / FW;
                unsigned long long v[PER_WARP][4];
#pragma unroll
                for (int jj = 0; jj < PER_WARP; ++jj)
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int sl = warp + FW * jj;
                        v[jj][q4] = (sl < U && 4 * th + q4 < T)
                                        ? ld_relaxed_u64(srcp + (size_t)sl * W2_BANDS * 16 * MAXT + q4)
                                        : ((unsigned long long)ltag << 32);
                    }
#pragma unroll
                for (int jj = 0; jj < PER_WARP; ++jj)
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        ok = ok && (uint32_t)(v[jj][q4] >> 32) == ltag;
                        s4[q4] += __uint_as_float((uint32_t)v[jj][q4]);
                    }
                if (__all_sync(0xFFFFFFFFu, ok))
                    break;
                if (it == SPIN_LIMIT) {
                    if (lane == 0)
                        atomicOr(flag, FLAG_TIMEOUT);
                    break;
                }
                __nanosleep(64);
            }
            sm.comb[warp][lane] = make_float4(s4[0], s4[1], s4[2], s4[3]);
            named_barrier_sync(7, FT);
            if (warp == 0) {
                float4 tot = sm.comb[0][lane];
#pragma unroll 1
                for (int w = 1; w < FW; ++w) {
                    const float4 v = sm.comb[w][lane];
                    tot.x += v.x; tot.y += v.y; tot.z += v.z; tot.w += v.w;
                }
                float vals[4] = {tot.x, tot.y, tot.z, tot.w};
                // the shared experts run ahead, in order, after the slots
                for (int j = 0; j < a.n_ext; ++j)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int t = 4 * th + jj;
                        if (t < T)
                            vals[jj] = fmaf(sm.extw[j][t],
                                            __ldcg(a.ext_y + ((size_t)j * MAXT + t) * H + 16 * band + r), vals[jj]);
                    }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int t = 4 * th + jj;
                    if (t < T)
                        a.out[(size_t)t * H + 16 * band + r] = __float2bfloat16_rn(vals[jj]);
                }
            }
        }
    }

    // ---- CTA 0 advances the launch tag once every CTA has read it (the h
    // warp of each CTA counts its CTA in ctrl[4]) ----
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (!gmem_wait_geq(&ctrl[4], gridDim.x, flag))
            return;
        ctrl[4] = 0u;
        ctrl[5] = ltag;   // the next launch tags its words ltag + 1
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

// After a call that gave up on a bounded wait, the workspace's count of CTAs
// may hold that call's partial count and its launch tag may not have advanced
// (CTA 0 returns before advancing it), so the words that call stored (router
// logits, h, down partials) may carry the tag the next call would use.  If
// the flag word shows a timeout, clear the counts and advance the tag, so
// that the next layer call ignores every stale word; the flag bits stay for
// the caller to read.  Runs after the preceding kernel has finished (it
// waits on it first).
__global__ void __launch_bounds__(32) rearm_kernel(uint8_t *ws)
{
    griddep_launch();
    griddep_wait();
    const WsLayout L = ws_layout();
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(ws + L.ctrl);
    if (threadIdx.x == 0 && (__ldcg(&ctrl[0]) & FLAG_TIMEOUT) != 0u) {
        ctrl[1] = 0u;
        ctrl[4] = 0u;
        ctrl[5] = ctrl[5] + 1u;
    }
}

cudaError_t launch_rearm(uint8_t *ws, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
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

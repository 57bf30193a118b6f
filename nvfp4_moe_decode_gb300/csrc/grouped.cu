// grouped.cu -- the MoE layer for many tokens (T > MOE_MAX_DECODE_T): the
// tokens are grouped by expert and every contraction runs on the tcgen05
// tensor cores.
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "From 1,096 kernels to 346": the same packed NVFP4 layout serves the
// small-batch GEMVs and the grouped GEMMs of large batches (the largest
// prefill gain); the weights are dequantised for the tensor cores and the
// activations stay 16-bit.
//
// Kernel chain (programmatic dependent launch between them):
//  1. router GEMM   logits[T][E] = x Wr^T (bf16 operands, fp32 accumulator);
//  2. top-k         one warp per token on the fp32 logits (the decode path's
//                   selection routine), per-CTA counts per expert, and (NVFP4
//                   weights) the token in f16 times a power of two, x16;
//  3. lists         a scan of the counts and a scatter: per expert, the
//                   (token, choice) pairs v = 6 t + i that selected it, in
//                   increasing v (and the inverse map); then a gather copies
//                   each listed token's row to xs[list row] (the GEMM
//                   operand, x16 or x), so that every GEMM reads consecutive
//                   rows;
//  4. gate/up GEMM  for every routed expert its listed tokens, and for the
//                   shared expert all tokens: SiLU(g) * u -> h (bf16);
//  5. h rescale     (NVFP4 weights) every h row in place to f16 times a
//                   power of two;
//  6. down GEMM     routed experts: y * routing weight -> ybuf[list row];
//  7. shared down   the shared expert's down projection -> ysh[token];
//  8. combine       out = sum over choices of ybuf[inverse map] (in choice
//                   order) + ysh, rounded once to bf16 (deterministic: no
//                   atomics), a streaming kernel of 16-byte loads.
// Without a shared expert step 7 is skipped.
// Every GEMM epilogue fetches its tile's per-column factors (routing weight,
// tensor scale, inverse power of two) into shared memory while the tile's
// MMAs run, so its loop over columns makes no dependent global loads.
//
// NVFP4 operands enter the tensor cores as f16, like the decode path: a
// weight is e2m1 x e4m3, exact in f16 (at most 6 significant bits, magnitude
// in [2^-10, 2688]); a token row of x (or of h) is multiplied by the power of
// two that puts its largest magnitude in [2^14, 2^15), exact for every
// element within 2^28 of the largest, and the epilogue multiplies by the
// inverse power and the tensor scale.  BF16 weights use bf16 operands as they
// are.
//
// GEMM kernel (steps 1, 4, 6, 7): persistent, one CTA per SM, 512 threads.
// A tile is (group, chunk of <= 256 tokens, 128-row M tile) with
// D[128 weight rows][N tokens] = A[128][K] . B[N][K]^T, N = the chunk's
// tokens rounded up to 16; tiles are dealt round-robin.  Roles:
//   warps 0-7   A producers, one 16-row band each: every lane loads its raw
//               NVFP4 bytes (codes and scales) three super-chunks (six
//               64-column chunks) ahead into registers and dequantises them
//               into the 128B-swizzled K-major A stage (bf16 rows are copied
//               there with cp.async instead);
//   warp 8      B producer: the tile's token rows, consecutive rows of xs,
//               x16, h or x, by 64- and 16-row TMA boxes;
//   warp 10     TMEM allocation and the MMA issue (one thread, 8 MMAs of
//               K = 16 per pair of 64-column chunks, one commit to the pair's
//               empty barrier, and one to the accumulator's full barrier per
//               tile);
//   warps 12-15 epilogue: tcgen05.ld of the accumulator (two 256-column
//               buffers, so a tile's epilogue overlaps the next tile's MMAs).
// Synchronisation is per pair of chunks (128 columns of K; every K here is a
// multiple of 128): the A and B tiles of both chunks share one full/empty
// barrier pair.  On GB300 an mbarrier wait costs ~200 cycles even when the
// phase is complete, and the MMA thread's waits and commits sit between its
// MMAs (measured: four MMAs of N = 192 take 0.22 us, with two waits and two
// commits 0.55 us), so every role makes one wait and one signal per 128
// columns: the MMA thread 8 MMAs per wait and commit, the A warps one fence
// and arrive per super-chunk, the B producer one expect-tx for both chunks.
// Every wait is bounded: a wait that runs out sets MOE_FLAG_WAIT_TIMEOUT
// and makes the CTA skip the rest of its work.
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc.cuh"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int G_STAGES = 4;                            // 64-column sub-stages (an A and a B tile each)
constexpr int G_PAIRS = G_STAGES / 2;                  // barrier slots, one per two sub-stages
constexpr int G_A_BYTES = 128 * TC_ROW_BYTES;          // 16 KB: 128 rows x 64 16-bit values
constexpr int G_B_BYTES = G_NMAX * TC_ROW_BYTES;       // 32 KB: 256 rows x 64 16-bit values
constexpr int G_AWARPS = 8;                            // A producers: one 16-row band each
constexpr int G_BWARP = 8;                             // B producer
constexpr int G_MMA_WARP = 10;
constexpr int G_EPI_WARP0 = 12;                        // epilogue warps 12..15 (TMEM lane quarters 0..3)
constexpr int G_THREADS = 512;
constexpr int G_MAX_GROUPS = E + 1;
constexpr int G_TMEM_COLS = 512;
constexpr uint32_t G_SPIN = 1u << 16;                  // suspended polls before a wait gives up
constexpr uint32_t G_SUSPEND_NS = 20000;               // suspend-time hint of one poll

struct GSmem {
    uint8_t a[G_STAGES][G_A_BYTES];                    // 1024-byte aligned tiles
    uint8_t b[G_STAGES][G_B_BYTES];
    // one barrier pair per two sub-stages (128 columns of K) for both
    // operands: full completes once the eight A warps have arrived and the B
    // tiles' bytes have landed, empty once the pair's MMAs have completed
    uint64_t full[G_PAIRS], empty[G_PAIRS];
    uint64_t d_full[2], d_empty[2];
    alignas(16) float colf[2][G_NMAX];                 // per-column epilogue factor of the tile (by accumulator)
    uint32_t tmem;
    int abort;
    int n_groups;
    int gn[G_MAX_GROUPS];                              // tokens of group g
    int goff[G_MAX_GROUPS];                            // first list row of group g
    int gtile[G_MAX_GROUPS + 1];                       // first tile of group g
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return smem_addr(p); }

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes (or the hint expires) instead of taking issue slots from the
// producer warps on the same scheduler.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"(G_SUSPEND_NS) : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase; false once the CTA has given up.
__device__ __forceinline__ bool gwait(uint64_t *bar, uint32_t parity, GSmem &sm, uint32_t *flag)
{
    for (uint32_t it = 0; it < G_SPIN; ++it) {
        if (mbar_try_wait_suspend(bar, parity))
            return true;
        if (*(volatile int *)&sm.abort)
            return false;
    }
    atomicOr(flag, FLAG_TIMEOUT);
    *(volatile int *)&sm.abort = 1;
    return false;
}

// gwait by lane 0, result shared with the warp.
__device__ __forceinline__ bool gwait_warp(uint64_t *bar, uint32_t parity, GSmem &sm, uint32_t *flag, int lane)
{
    bool ok = true;
    if (lane == 0)
        ok = gwait(bar, parity, sm, flag);
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

// TMA: one box (64 columns x the map's box rows, 128-byte swizzled rows) at (col, row).
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap *map, int col, int row, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(map), "r"(col), "r"(row), "r"(smem_addr(bar)) : "memory");
}

// Four e2m1 code pairs (one 32-bit word, byte r = codes of two columns, low
// nibble first) as f16x2 registers.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t &h0, uint32_t &h1, uint32_t &h2, uint32_t &h3)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(w));
}

// Two e4m3 scale bytes (low byte first) as one f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t h2;
    asm("{\n\t.reg .b16 b;\n\tcvt.u16.u32 b, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, b;\n\t}" : "=r"(h2) : "r"(two));
    return h2;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float pow2f(int k) { return __int_as_float((127 + k) << 23); }

// Power of two that puts max|row| in [2^14, 2^15) (0 for an all-zero row).
__device__ __forceinline__ int row_shift(float maxabs)
{
    const int sh = ACT_EXP - exponent_of(maxabs);
    return sh < -100 ? -100 : (sh > 100 ? 100 : sh);
}

struct Tile {
    int g, n0, nvalid, npad, mt;
};

__device__ __forceinline__ Tile decode_tile(const GSmem &sm, const GArgs &a, int id)
{
    int lo = 0, hi = sm.n_groups - 1;   // last group whose first tile <= id
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.gtile[mid] <= id)
            lo = mid;
        else
            hi = mid - 1;
    }
    Tile t;
    t.g = lo;
    const int local = id - sm.gtile[lo];
    const int j = local / a.mtiles, mt = local % a.mtiles;
    t.mt = mt;
    t.n0 = j * a.nmax;
    t.nvalid = min(a.nmax, sm.gn[lo] - t.n0);
    t.npad = (t.nvalid + 15) & ~15;
    return t;
}

// The routed expert of group g, or -1 for the shared expert / the router.
__device__ __forceinline__ int group_expert(const GArgs &a, int g)
{
    if (a.mode == GM_ROUTER || a.mode == GM_SHARED_DOWN)
        return -1;
    return g < E ? g : -1;
}

}  // namespace

__global__ void __launch_bounds__(G_THREADS, 1)
    moe_grouped_gemm_kernel(const __grid_constant__ GArgs a, const __grid_constant__ CUtensorMap map_routed64,
                            const __grid_constant__ CUtensorMap map_routed16,
                            const __grid_constant__ CUtensorMap map_shared64,
                            const __grid_constant__ CUtensorMap map_shared16)
{
    extern __shared__ uint8_t g_smem_raw[];
    GSmem &sm = *reinterpret_cast<GSmem *>((uint8_t *)(((uintptr_t)g_smem_raw + 1023) & ~(uintptr_t)1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    griddep_wait();       // lists, x16, h and ybuf come from the preceding kernels
    griddep_launch();

    if (threadIdx.x == 0) {
        for (int p = 0; p < G_PAIRS; ++p) {
            mbar_init(&sm.full[p], G_AWARPS + 1);
            mbar_init(&sm.empty[p], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.d_full[i], 1);
            mbar_init(&sm.d_empty[i], 4);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    // group table: tokens, first list row and first tile of every group
    if (warp == 0) {
        int ng;
        if (a.mode == GM_GATE_UP)
            ng = E + (a.n_shared ? 1 : 0);
        else if (a.mode == GM_DOWN)
            ng = E;
        else
            ng = 1;
        int run = 0;
        for (int base = 0; base < ng; base += 32) {
            const int g = base + lane;
            int n = 0, off = 0;
            if (g < ng) {
                if ((a.mode == GM_GATE_UP || a.mode == GM_DOWN) && g < E) {
                    n = a.counts[g];
                    off = a.offsets[g];
                } else {
                    n = a.T;
                }
                sm.gn[g] = n;
                sm.goff[g] = off;
            }
            int tiles = (g < ng) ? ((n + a.nmax - 1) / a.nmax) * a.mtiles : 0;
            int incl = tiles;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (g < ng)
                sm.gtile[g] = run + incl - tiles;
            run += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) {
            sm.gtile[ng] = run;
            sm.n_groups = ng;
        }
    }
    if (warp == G_MMA_WARP)
        tc_alloc(&sm.tmem, G_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const int total_tiles = sm.gtile[sm.n_groups];
    const int nch = a.K / TC_KCHUNK;
    const int my_tiles = (int)blockIdx.x < total_tiles ? (total_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int stream_len = my_tiles * nch;          // chunks this CTA streams
    // gate/up walks the tiles from the last expert down: the gather wrote
    // the sorted rows in list order, so its last rows are still in L2 when
    // the GEMM starts (measured: 670 -> 664 us per layer at T = 8192)
    auto tile_id = [&](int ti) {
        const int id = (int)blockIdx.x + ti * (int)gridDim.x;
        return a.mode == GM_GATE_UP ? total_tiles - 1 - id : id;
    };
    uint32_t *flag = a.flag;

    // A-operand base of group g (bytes): packed NVFP4 or bf16 rows of one matrix
    auto a_base = [&](int g) -> const uint8_t * {
        if (a.mode == GM_ROUTER)
            return reinterpret_cast<const uint8_t *>(a.wr);
        const int e = group_expert(a, g);
        return e >= 0 ? a.ra + (size_t)e * a.a_stride : a.sa;
    };
    auto a_tscale = [&](int g) -> float {
        if (a.a_bf16 || a.mode == GM_ROUTER)
            return 1.0f;
        const int e = group_expert(a, g);
        return e >= 0 ? __ldg(a.rts + e) : __ldg(a.sts);
    };

    if (warp < G_AWARPS) {
        // ------------------------------------------------------------ A producers
        if (!a.a_bf16) {
            // warp w dequantises band 8 mt + w (16 rows) of every chunk to f16.
            // Each lane loads its own raw bytes with ld.global three
            // super-chunks ahead (a super-chunk = 1152 bytes of the band: the
            // codes of two 64-column chunks and their scales): 16 code bytes
            // per chunk and the 16 scale bytes of its row pair.
            const int g4 = lane >> 2, c4 = lane & 3;
            const size_t band_bytes_k = (size_t)9 * a.K;
            const int nsc_tile = nch >> 1;                 // super-chunks per tile
            const int nsc = stream_len >> 1;               // super-chunks of this CTA's stream
            int pf_ti = -1;
            const uint8_t *pf_band = nullptr;
            auto sc_ptr = [&](int sci) -> const uint8_t * {   // called with increasing sci
                const int ti = sci / nsc_tile;
                if (ti != pf_ti) {
                    pf_ti = ti;
                    const Tile t = decode_tile(sm, a, tile_id(ti));
                    pf_band = a_base(t.g) + (size_t)(8 * t.mt + warp) * band_bytes_k;
                }
                return pf_band + (size_t)(sci % nsc_tile) * SC_BYTES;
            };
            uint4 rc0[3], rc1[3], rs[3];
            auto load = [&](int j, int sci) {
                if (sci < nsc) {
                    const uint8_t *p = sc_ptr(sci);
                    rc0[j] = ldg_nc_v4(p + 16 * lane);
                    rc1[j] = ldg_nc_v4(p + 512 + 16 * lane);
                    rs[j] = ldg_nc_v4(p + 1024 + 16 * g4);
                }
            };
            // lane (g, c) writes 4 bytes at row 16 w + g + 8 (r & 1), 16-byte
            // chunk (2 st + (r >> 1)) ^ g, byte 4 c, for word st and byte r
            const uint32_t row0 = (uint32_t)((16 * warp + g4) * TC_ROW_BYTES) + 4u * c4;
            auto fill = [&](int s, const uint4 &cw, uint32_t s01, uint32_t s23) {
                const uint32_t abase = smem_u32(sm.a[s]) + row0;
                const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int st = 0; st < 4; ++st) {
                    // scale bytes 2 st (row g) and 2 st + 1 (row g + 8)
                    const uint32_t sc = e4m3x2_to_f16x2(((st < 2 ? s01 : s23) >> (16 * (st & 1))) & 0xFFFFu);
                    const uint32_t s_lo = __byte_perm(sc, 0, 0x1010), s_hi = __byte_perm(sc, 0, 0x3232);
                    uint32_t h[4];
                    e2m1x8_to_f16(words[st], h[0], h[1], h[2], h[3]);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint32_t v = hmul2_u32(h[r], (r & 1) ? s_hi : s_lo);
                        const uint32_t off = (uint32_t)(8 * (r & 1) * TC_ROW_BYTES) +
                                             (uint32_t)(((2 * st + (r >> 1)) ^ g4) << 4);
                        st_shared32(abase + off, v);
                    }
                }
            };
            // super-chunk sci fills sub-stages 2 (sci % 2) and 2 (sci % 2) + 1:
            // one wait, one fence and one arrive per super-chunk
            auto process = [&](int sci, const uint4 &c0, const uint4 &c1, const uint4 &sw) -> bool {
                const int p = sci % G_PAIRS;
                if (sci >= G_PAIRS && !gwait_warp(&sm.empty[p], ((sci / G_PAIRS) - 1) & 1, sm, flag, lane))
                    return false;
                fill(2 * p, c0, sw.x, sw.y);
                fill(2 * p + 1, c1, sw.z, sw.w);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sm.full[p]);
                return true;
            };
            load(0, 0);
            load(1, 1);
            load(2, 2);
            bool ok = true;
            for (int sc0 = 0; sc0 < nsc && ok; sc0 += 3) {
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const int sci = sc0 + j;
                    if (sci < nsc && ok) {
                        const uint4 c0 = rc0[j], c1 = rc1[j], sw = rs[j];
                        load(j, sci + 3);                  // refill this slot
                        ok = process(sci, c0, c1, sw);
                    }
                }
            }
        } else {
            // bf16 rows: warp w copies rows 16 w .. 16 w + 15 (16 x 8 chunks of
            // 16 bytes) of both chunks of a pair, one cp.async group per pair;
            // a pair is signalled once the next one has been issued
            const int c8 = lane & 7;
            const int npairs = stream_len >> 1;
            int pk = 0;
            for (; pk < npairs; ++pk) {
                const int p = pk % G_PAIRS;
                if (pk >= G_PAIRS && !gwait_warp(&sm.empty[p], ((pk / G_PAIRS) - 1) & 1, sm, flag, lane))
                    break;
                const Tile t = decode_tile(sm, a, tile_id((2 * pk) / nch));
                const __nv_bfloat16 *base = reinterpret_cast<const __nv_bfloat16 *>(a_base(t.g));
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int ch = (2 * pk + h2) % nch;
                    const uint32_t abase = smem_u32(sm.a[2 * p + h2]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int R = 16 * warp + (lane >> 3) + 4 * i;
                        int row;
                        if (a.mode == GM_GATE_UP) {
                            const int ii = R & 15, b = 8 * t.mt + (R >> 4);
                            row = ii < 8 ? 8 * b + ii : I + 8 * b + (ii - 8);
                        } else {
                            row = 128 * t.mt + R;
                        }
                        cp_async16(abase + sw128_offset(R, c8), base + (size_t)row * a.K + ch * TC_KCHUNK + 8 * c8,
                                   16u);
                    }
                }
                cp_async_commit();
                if (pk >= 1) {
                    cp_async_wait<1>();
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&sm.full[(pk - 1) % G_PAIRS]);
                }
            }
            cp_async_wait<0>();
            fence_proxy_async();
            __syncwarp();
            if (lane == 0 && pk >= 1)
                mbar_arrive(&sm.full[(pk - 1) % G_PAIRS]);
        }
    } else if (warp == G_BWARP) {
        // ------------------------------------------------------------ B producer
        // routed groups read their list rows (xs, or h in list order), the
        // shared group / the router its token rows; columns beyond the tile's
        // tokens are loaded too (other rows, or zeros past the end) and are
        // never stored
        int cur_tile = -1, npad = 0, row0 = 0;
        bool routed = false;
        const int npairs = stream_len >> 1;
        for (int pk = 0; pk < npairs; ++pk) {
            const int ti = (2 * pk) / nch, ch0 = (2 * pk) % nch;   // a pair never straddles two tiles
            if (ti != cur_tile) {
                cur_tile = ti;
                const Tile t = decode_tile(sm, a, tile_id(ti));
                npad = t.npad;
                routed = group_expert(a, t.g) >= 0;
                row0 = (routed ? sm.goff[t.g] : 0) + t.n0;
            }
            const int p = pk % G_PAIRS;
            if (pk >= G_PAIRS && !gwait_warp(&sm.empty[p], ((pk / G_PAIRS) - 1) & 1, sm, flag, lane))
                break;
            if (lane == 0)
                mbar_arrive_expect_tx(&sm.full[p], (uint32_t)(2 * npad * TC_ROW_BYTES));
            __syncwarp();
            // per chunk 64-row boxes, then 16-row boxes for the rest (at most 3 + 3 copies)
            const int n64 = npad >> 6, n16 = (npad & 63) >> 4, nb = n64 + n16;
            if (lane < 2 * nb) {
                const int h2 = lane >= nb ? 1 : 0, j = lane - h2 * nb;
                const int r = j < n64 ? 64 * j : 64 * n64 + 16 * (j - n64);
                const CUtensorMap *map = j < n64 ? (routed ? &map_routed64 : &map_shared64)
                                                 : (routed ? &map_routed16 : &map_shared16);
                tma_box(smem_u32(sm.b[2 * p + h2]) + (uint32_t)(r * TC_ROW_BYTES), map, (ch0 + h2) * TC_KCHUNK,
                        row0 + r, &sm.full[p]);
            }
        }
    } else if (warp == G_MMA_WARP) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t tbase = sm.tmem;
            int pk = 0;                                // pairs of chunks so far
            bool ok = true;
            for (int ti = 0; ti < my_tiles && ok; ++ti) {
                const Tile t = decode_tile(sm, a, tile_id(ti));
                const uint32_t idesc = a.f16 ? idesc_f16_m128(t.npad) : idesc_bf16_m128(t.npad);
                const int ab = ti & 1;
                ok = gwait(&sm.d_empty[ab], ((ti >> 1) & 1) ^ 1, sm, flag);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t d = tbase + (uint32_t)(ab * 256);
                for (int ch = 0; ch < nch; ch += 2, ++pk) {
                    const int p = pk % G_PAIRS;
                    if (!gwait(&sm.full[p], (pk / G_PAIRS) & 1, sm, flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const uint32_t aa = smem_u32(sm.a[2 * p + h2]), bb = smem_u32(sm.b[2 * p + h2]);
#pragma unroll
                        for (int k16 = 0; k16 < 4; ++k16)
                            tc_mma(d, sw128_desc(aa + 32 * k16), sw128_desc(bb + 32 * k16), idesc,
                                   (ch > 0 || h2 > 0 || k16 > 0) ? 1u : 0u);
                    }
                    tc_commit(&sm.empty[p]);
                }
                if (ok)
                    tc_commit(&sm.d_full[ab]);
            }
        }
        __syncwarp();
    } else if (warp >= G_EPI_WARP0) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int R = 32 * q + lane;                   // tile row = TMEM lane
        const uint32_t tbase = sm.tmem + ((uint32_t)(32 * q) << 16);
        for (int ti = 0; ti < my_tiles; ++ti) {
            const Tile t = decode_tile(sm, a, tile_id(ti));
            const int ab = ti & 1;
            const float ts = a_tscale(t.g);
            const int e = group_expert(a, t.g);
            // the tile's per-column factors (and ybuf rows), fetched into
            // shared memory by the four epilogue warps while its MMAs run:
            // ts times the column's inverse power of two, times its routing
            // weight for the down projection
            for (int c = R; c < t.nvalid; c += 128) {
                float fc = ts;
                if (a.mode == GM_GATE_UP) {
                    if (a.xshift) {
                        const int tok = (e >= 0) ? __ldg(a.list + sm.goff[t.g] + t.n0 + c) / TOPK : t.n0 + c;
                        fc = ts * pow2f(-__ldg(a.xshift + tok));
                    }
                } else if (a.mode == GM_DOWN) {
                    const int row = sm.goff[t.g] + t.n0 + c;
                    fc = __ldg(a.topk_w + __ldg(a.list + row)) * ts;
                    if (a.hshift_r)
                        fc *= pow2f(-__ldg(a.hshift_r + row));
                } else if (a.mode == GM_SHARED_DOWN) {
                    if (a.hshift_s)
                        fc = ts * pow2f(-__ldg(a.hshift_s + t.n0 + c));
                }
                sm.colf[ab][c] = fc;
            }
            // the four epilogue warps: tables written before any is read (the
            // other buffer may still be in use by a warp on the previous tile)
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (!gwait_warp(&sm.d_full[ab], (ti >> 1) & 1, sm, flag, lane))
                break;
            tc_fence_after();
            const float *colf = sm.colf[ab];
            for (int c0 = 0; c0 < t.npad; c0 += 32) {
                float v[32];
                tc_ld32(tbase + (uint32_t)(ab * 256 + c0), v);
                // the block's 32 column factors in registers up front (eight
                // broadcast loads), so no load sits between the stores below
                float cf[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 q4 = reinterpret_cast<const float4 *>(colf + c0)[i];
                    cf[4 * i] = q4.x;
                    cf[4 * i + 1] = q4.y;
                    cf[4 * i + 2] = q4.z;
                    cf[4 * i + 3] = q4.w;
                }
                if (a.mode == GM_GATE_UP) {
                    // rows 16 bb + i: i < 8 gate, i >= 8 up of feature 8 (8 mt + bb) + (i & 7);
                    // column pair (2 m, 2 m + 1): gate lanes finish column 2 m, up lanes 2 m + 1
                    const int bb = R >> 4, ii = R & 15;
                    const bool up = ii >= 8;
                    const int f = 8 * (8 * t.mt + bb) + (ii & 7);
                    __nv_bfloat16 *hrow = (e >= 0) ? a.h_routed + (size_t)(sm.goff[t.g] + t.n0) * I
                                                   : a.h_shared + (size_t)t.n0 * I;
                    float hv[16];
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        // branch-free, so the 16 chains interleave; padding
                        // columns are computed and not stored
                        const float send = up ? v[2 * m] : v[2 * m + 1];
                        const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 8);
                        const float fc = up ? cf[2 * m + 1] : cf[2 * m];
                        const float gv = (up ? recv : v[2 * m]) * fc;
                        const float uv = (up ? v[2 * m + 1] : recv) * fc;
                        hv[m] = gv / (1.0f + __expf(-gv)) * uv;
                    }
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const int col = c0 + 2 * m + (up ? 1 : 0);
                        if (col < t.nvalid)
                            hrow[(size_t)col * I + f] = __float2bfloat16_rn(hv[m]);
                    }
                } else if (a.mode == GM_DOWN || a.mode == GM_SHARED_DOWN) {
                    // routed: weighted rows of ybuf in list order; shared: its own rows (ysh)
                    float *dst = (a.mode == GM_DOWN ? a.ybuf + (size_t)(sm.goff[t.g] + t.n0 + c0) * H
                                                    : a.ysh + (size_t)(t.n0 + c0) * H) +
                                 128 * t.mt + R;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < t.nvalid)
                            dst[(size_t)j * H] = v[j] * cf[j];
                } else {
                    const int ee = 128 * t.mt + R;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int col = c0 + j;
                        if (col < t.nvalid)
                            a.logits[(size_t)(t.n0 + col) * E + ee] = v[j];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.d_empty[ab]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == G_MMA_WARP) {
        tc_fence_after();
        tc_dealloc(sm.tmem, G_TMEM_COLS);
    }
}

// One warp per token: top-k of the fp32 logits, renormalised weights; CTA
// c (G_TOK_PER_CTA tokens) counts its selections per expert into hist[c][E];
// with x16 given, the token row is also written as f16 times 2^xshift[t].
constexpr int G_TOPK_WARPS = 16;                       // warps per top-k CTA (two tokens each)

__global__ void __launch_bounds__(G_TOPK_WARPS * 32) moe_grouped_topk_kernel(const float *logits, int T, int32_t *idx, float *w,
                                                             int32_t *hist, const __nv_bfloat16 *x, __half *x16,
                                                             int32_t *xshift, uint32_t *flag)
{
    griddep_wait();
    griddep_launch();
    __shared__ int h[E];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < E; i += blockDim.x)
        h[i] = 0;
    __syncthreads();
    for (int k = 0; k < G_TOK_PER_CTA / G_TOPK_WARPS; ++k) {
        const int t = blockIdx.x * G_TOK_PER_CTA + k * G_TOPK_WARPS + warp;
        if (t >= T)
            break;
        int ex;
        float wt;
        bool bad;
        warp_route_token(logits + (size_t)t * E, lane, ex, wt, bad);
        if (bad && lane == 0)
            atomicOr(flag, FLAG_NONFINITE);
        if (lane < TOPK) {
            idx[(size_t)t * TOPK + lane] = ex;
            w[(size_t)t * TOPK + lane] = wt;
            if (ex >= 0 && ex < E)
                atomicAdd(&h[ex], 1);
        }
        if (x16) {
            const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
            uint4 v[H / 256];
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < H / 256; ++i) {
                v[i] = __ldg(row + lane + 32 * i);
                const uint32_t q4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_float(q4[j] & 0xFFFFu)), fabsf(bf16_bits_to_float(q4[j] >> 16))));
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            const int sh = row_shift(m);
            const float p = pow2f(sh);
            uint4 *dst = reinterpret_cast<uint4 *>(x16 + (size_t)t * H);
#pragma unroll
            for (int i = 0; i < H / 256; ++i) {
                const uint32_t q4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t o4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    o4[j] = bf16x2_to_f16x2_scaled(q4[j], p);
                dst[lane + 32 * i] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
            if (lane == 0)
                xshift[t] = sh;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x)
        hist[(size_t)blockIdx.x * E + i] = h[i];
}

// Expert lists, step 1 of 2 (one CTA; a thread takes four experts over one
// of G_SCAN_PARTS ranges of the CTA rows): the per-CTA counts hist[c][e] become the
// first list row of (c, e), base[c][e] = offsets[e] + sum over c' < c of
// hist[c'][e], where offsets is the exclusive prefix of the expert totals
// (counts): partial sums, then the totals and offsets, then each part writes
// its rows from its starting value.
constexpr int G_SCAN_PARTS = 16;                       // row ranges of the scan (4 experts per thread)

__global__ void __launch_bounds__(E / 4 * G_SCAN_PARTS) moe_grouped_scan_kernel(const int32_t *hist, int nc,
                                                                                int32_t *base, int32_t *counts,
                                                                                int32_t *offsets)
{
    griddep_wait();
    griddep_launch();
    const int g4 = threadIdx.x % (E / 4), part = threadIdx.x / (E / 4);   // experts 4 g4 .. 4 g4 + 3
    const int per = (nc + G_SCAN_PARTS - 1) / G_SCAN_PARTS;
    const int c_lo = min(nc, part * per), c_hi = min(nc, c_lo + per);
    auto sweep = [&](int4 run, bool store) {
        for (int c0 = c_lo; c0 < c_hi; c0 += 8) {
            int4 hv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                hv[j] = (c0 + j < c_hi) ? __ldcg(reinterpret_cast<const int4 *>(hist + (size_t)(c0 + j) * E) + g4)
                                        : make_int4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (store && c0 + j < c_hi)
                    reinterpret_cast<int4 *>(base + (size_t)(c0 + j) * E)[g4] = run;
                run.x += hv[j].x;
                run.y += hv[j].y;
                run.z += hv[j].z;
                run.w += hv[j].w;
            }
        }
        return run;
    };
    __shared__ int psum[G_SCAN_PARTS][E];
    __shared__ int off_s[E];
    {
        const int4 r = sweep(make_int4(0, 0, 0, 0), false);
        psum[part][4 * g4] = r.x;
        psum[part][4 * g4 + 1] = r.y;
        psum[part][4 * g4 + 2] = r.z;
        psum[part][4 * g4 + 3] = r.w;
    }
    __syncthreads();
    if (threadIdx.x < E) {
        const int e = threadIdx.x;
        int tot = 0;
#pragma unroll
        for (int q = 0; q < G_SCAN_PARTS; ++q)
            tot += psum[q][e];
        // exclusive prefix over experts (E = 256 totals, one warp-scan per 32)
        const int lane = e & 31, warp = e >> 5;
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += v;
        }
        __shared__ int wtot[E / 32];
        if (lane == 31)
            wtot[warp] = incl;
        asm volatile("bar.sync 1, %0;" ::"n"(E) : "memory");   // the first E threads
        int before = 0;
        for (int w2 = 0; w2 < warp; ++w2)
            before += wtot[w2];
        const int off = before + incl - tot;
        counts[e] = tot;
        offsets[e] = off;
        if (e == E - 1)
            offsets[E] = off + tot;
        off_s[e] = off;
    }
    __syncthreads();
    int4 start = make_int4(off_s[4 * g4], off_s[4 * g4 + 1], off_s[4 * g4 + 2], off_s[4 * g4 + 3]);
    for (int q = 0; q < part; ++q) {
        start.x += psum[q][4 * g4];
        start.y += psum[q][4 * g4 + 1];
        start.z += psum[q][4 * g4 + 2];
        start.w += psum[q][4 * g4 + 3];
    }
    sweep(start, true);
}

// Expert lists, step 2 of 2: CTA c writes the pairs v = 6 t + i of its
// tokens to list[base[c][e] + rank], rank = earlier pairs of the CTA that
// chose the same expert, so every expert's rows are in increasing v, and
// inv[v] = that list row (-1 for an invalid selection).
__global__ void __launch_bounds__(G_TOK_PER_CTA * TOPK) moe_grouped_scatter_kernel(const int32_t *idx, int T,
                                                                                 const int32_t *base, int32_t *list,
                                                                                 int32_t *inv, uint32_t *flag)
{
    griddep_wait();
    griddep_launch();
    __shared__ int ex[G_TOK_PER_CTA * TOPK];
    const int n = min(G_TOK_PER_CTA, T - (int)blockIdx.x * G_TOK_PER_CTA) * TOPK;
    const int v0 = blockIdx.x * G_TOK_PER_CTA * TOPK;
    const int k = threadIdx.x;
    const int e = (k < n) ? __ldg(idx + v0 + k) : -1;
    ex[k] = e;
    __syncthreads();
    int p = -1;
    if (k < n) {
        if (e < 0 || e >= E) {
            atomicOr(flag, FLAG_BAD_INDEX);
        } else {
            int rank = 0;
            for (int j = 0; j < k; ++j)
                rank += (ex[j] == e);
            p = __ldg(base + (size_t)blockIdx.x * E + e) + rank;
            list[p] = v0 + k;
        }
    }
    if (k < n)
        inv[v0 + k] = p;                               // the list row of (token, choice), -1 if invalid
}

// xs[r] = src[list[r] / TOPK]: every listed (token, choice) row copied to its
// list row, 16 bytes per thread and eight copies in flight per thread.  Only
// the offsets[E] listed rows are copied (fewer than T * TOPK when a selection
// was invalid), and a token index outside [0, T) is skipped.
__global__ void __launch_bounds__(256) moe_grouped_gather_kernel(const int32_t *list, const int32_t *offsets, int T,
                                                                 const uint16_t *src, uint16_t *xs)
{
    griddep_wait();
    griddep_launch();
    constexpr int Q = H / 8;                           // 16-byte pieces per row
    const int nrows = min(__ldg(offsets + E), T * TOPK);
    const size_t n = (size_t)max(nrows, 0) * Q, stride = (size_t)gridDim.x * blockDim.x;
    for (size_t q0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q0 < n; q0 += 8 * stride) {
        uint4 v[8];
        size_t dq[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const size_t q = q0 + u * stride;
            dq[u] = q;
            if (q < n) {
                const size_t r = q / Q, c = q % Q;
                const int t = __ldg(list + r) / TOPK;
                if ((unsigned)t < (unsigned)T)
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(src) + (size_t)t * Q + c);
                else
                    dq[u] = n;                         // skipped
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (dq[u] < n)
                __stcs(reinterpret_cast<uint4 *>(xs) + dq[u], v[u]);
    }
}

// h rows (bf16) rescaled in place to f16 times 2^shift[row] (one warp per
// row of I = 512 values).
__global__ void __launch_bounds__(256) moe_grouped_hscale_kernel(uint16_t *h, int rows, int32_t *shift)
{
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < rows; r += gridDim.x * 8) {
        uint4 *row = reinterpret_cast<uint4 *>(h + (size_t)r * I);
        uint4 v[I / 256];
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < I / 256; ++i) {
            v[i] = row[lane + 32 * i];
            const uint32_t q4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_float(q4[j] & 0xFFFFu)), fabsf(bf16_bits_to_float(q4[j] >> 16))));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const int sh = row_shift(m);
        const float p = pow2f(sh);
#pragma unroll
        for (int i = 0; i < I / 256; ++i) {
            const uint32_t q4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t o4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                o4[j] = bf16x2_to_f16x2_scaled(q4[j], p);
            row[lane + 32 * i] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
        if (lane == 0)
            shift[r] = sh;
    }
}

// out[t] = sum over choices of the choice's ybuf row (choice order; ybuf is
// in list order, inv[6 t + i] its row), then + ysh[t] (the shared expert's
// down projection, when there is one), rounded once to bf16.  Four
// consecutive features per thread (16-byte loads).
__global__ void __launch_bounds__(256) moe_grouped_combine_kernel(const float *ybuf, const int32_t *inv,
                                                                  const float *ysh, int T, __nv_bfloat16 *out)
{
    griddep_wait();
    griddep_launch();
    const size_t n4 = (size_t)T * (H / 4);
    for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < n4; o += (size_t)gridDim.x * blockDim.x) {
        const size_t t = o / (H / 4), f = 4 * (o % (H / 4));
        int r[TOPK];
#pragma unroll
        for (int i = 0; i < TOPK; ++i)
            r[i] = __ldg(inv + t * TOPK + i);
        float4 y[TOPK + 1];
#pragma unroll
        for (int i = 0; i < TOPK; ++i)
            y[i] = r[i] >= 0 ? __ldcs(reinterpret_cast<const float4 *>(ybuf + (size_t)r[i] * H + f))
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (ysh)
            y[TOPK] = __ldcs(reinterpret_cast<const float4 *>(ysh + t * H + f));
        float4 acc = y[0];
#pragma unroll
        for (int i = 1; i < TOPK; ++i) {
            acc.x += y[i].x;
            acc.y += y[i].y;
            acc.z += y[i].z;
            acc.w += y[i].w;
        }
        if (ysh) {
            acc.x += y[TOPK].x;
            acc.y += y[TOPK].y;
            acc.z += y[TOPK].z;
            acc.w += y[TOPK].w;
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(out + t * H + f) = pk;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

GWsLayout gws_layout(int T)
{
    const size_t nc = (size_t)(T + G_TOK_PER_CTA - 1) / G_TOK_PER_CTA;
    GWsLayout L;
    // ctrl is the decode workspace's flag word; the routing (idx, w, logits)
    // sits where the chunked decode path copies its routing out, after the
    // decode workspace, so moe_read_routing reads one place for either path
    const ChunkRouteLayout C = chunk_route_layout(T);
    L.ctrl = 0;
    L.idx = C.idx;
    L.w = C.w;
    L.logits = C.logits;
    size_t o = C.total;
    L.counts = o;    o = align256(o + (size_t)E * 4);
    L.offsets = o;   o = align256(o + (size_t)(E + 1) * 4);
    L.list = o;      o = align256(o + (size_t)T * TOPK * 4);
    L.hist = o;      o = align256(o + nc * E * 4);
    L.base = o;      o = align256(o + nc * E * 4);
    L.x16 = o;       o = align256(o + (size_t)T * H * 2);
    L.xs = o;        o = align256(o + (size_t)T * TOPK * H * 2);
    L.xshift = o;    o = align256(o + (size_t)T * 4);
    L.hshift = o;    o = align256(o + (size_t)T * (TOPK + 1) * 4);
    L.h_routed = o;  o = o + (size_t)T * TOPK * I * 2;          // h_shared follows directly
    L.h_shared = o;  o = align256(o + (size_t)T * I * 2);
    L.ybuf = o;      o = align256(o + (size_t)T * TOPK * H * 4);
    L.ysh = o;       o = align256(o + (size_t)T * H * 4);
    L.inv = o;       o = align256(o + (size_t)T * TOPK * 4);
    L.total = o;
    return L;
}

static cudaError_t launch_ex(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void **args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

size_t grouped_smem_bytes() { return sizeof(GSmem) + 1024; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); looked up once (a thread-safe static).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    }();
    return fn;
}

// A 2D map over rows x cols 16-bit values (row pitch cols * 2 bytes), box
// 64 columns x box_rows rows, 128-byte swizzle.
static bool make_map(CUtensorMap *m, const void *base, int cols, size_t rows, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)TC_KCHUNK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One grouped GEMM launch; B rows come from `routed` (list rows of the
// routed groups) and `shared` (token rows of the shared group / router), both
// `cols` 16-bit values wide.
static cudaError_t launch_gemm(const GArgs &ga, const void *routed, size_t routed_rows, const void *shared,
                               size_t shared_rows, int cols, int nsm, cudaStream_t st)
{
    static PerDevice configured;
    if (per_device(configured, [](int) {
            return cudaFuncSetAttribute(moe_grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)grouped_smem_bytes()) == cudaSuccess
                       ? 1
                       : -1;
        }) <= 0)
        return cudaErrorInvalidValue;
    alignas(64) CUtensorMap mr64, mr16, ms64, ms16;
    const void *r = routed ? routed : shared, *s = shared ? shared : routed;
    const size_t rr = routed ? routed_rows : shared_rows, sr = shared ? shared_rows : routed_rows;
    if (!make_map(&mr64, r, cols, rr, 64) || !make_map(&mr16, r, cols, rr, 16) || !make_map(&ms64, s, cols, sr, 64) ||
        !make_map(&ms16, s, cols, sr, 16))
        return cudaErrorInvalidValue;
    GArgs copy = ga;
    void *args[] = {&copy, &mr64, &mr16, &ms64, &ms16};
    return launch_ex((const void *)moe_grouped_gemm_kernel, dim3(nsm), dim3(G_THREADS), grouped_smem_bytes(), st, args);
}

cudaError_t launch_grouped_route(const GroupedArgs &a, int nsm, cudaStream_t st)
{
    const GWsLayout L = gws_layout(a.T);
    uint8_t *ws = a.ws;
    GArgs g{};
    g.mode = GM_ROUTER;
    g.T = a.T;
    g.nmax = 128;
    g.a_bf16 = 1;
    g.f16 = 0;
    g.K = H;
    g.mtiles = E / 128;
    g.wr = a.wr;
    g.flag = reinterpret_cast<uint32_t *>(ws + L.ctrl);
    g.logits = reinterpret_cast<float *>(ws + L.logits);
    cudaError_t e = launch_gemm(g, nullptr, 0, a.x, (size_t)a.T, H, nsm, st);
    if (e != cudaSuccess)
        return e;
    float *logits = g.logits;
    int T = a.T;
    int32_t *idx = reinterpret_cast<int32_t *>(ws + L.idx);
    float *w = reinterpret_cast<float *>(ws + L.w);
    int32_t *hist = reinterpret_cast<int32_t *>(ws + L.hist);
    const __nv_bfloat16 *x = a.x;
    __half *x16 = a.convert_x ? reinterpret_cast<__half *>(ws + L.x16) : nullptr;
    int32_t *xshift = reinterpret_cast<int32_t *>(ws + L.xshift);
    uint32_t *flag = g.flag;
    void *targs[] = {&logits, &T, &idx, &w, &hist, &x, &x16, &xshift, &flag};
    return launch_ex((const void *)moe_grouped_topk_kernel, dim3((a.T + G_TOK_PER_CTA - 1) / G_TOK_PER_CTA), dim3(G_TOPK_WARPS * 32),
                     0, st, targs);
}

cudaError_t launch_grouped_layer(const GroupedArgs &a0, int nsm, cudaStream_t st)
{
    GroupedArgs a = a0;
    a.convert_x = a.bf16w ? 0 : 1;
    cudaError_t e = launch_grouped_route(a, nsm, st);
    if (e != cudaSuccess)
        return e;
    const GWsLayout L = gws_layout(a.T);
    uint8_t *ws = a.ws;
    uint32_t *flag = reinterpret_cast<uint32_t *>(ws + L.ctrl);
    int32_t *idx = reinterpret_cast<int32_t *>(ws + L.idx);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *list = reinterpret_cast<int32_t *>(ws + L.list);
    int32_t *hist = reinterpret_cast<int32_t *>(ws + L.hist);
    int32_t *base = reinterpret_cast<int32_t *>(ws + L.base);
    int T = a.T;
    int nc = (a.T + G_TOK_PER_CTA - 1) / G_TOK_PER_CTA;
    {
        void *sargs[] = {&hist, &nc, &base, &counts, &offsets};
        e = launch_ex((const void *)moe_grouped_scan_kernel, dim3(1), dim3(E / 4 * G_SCAN_PARTS), 0, st, sargs);
        if (e != cudaSuccess)
            return e;
        const uint16_t *src = reinterpret_cast<const uint16_t *>(a.bf16w ? (const void *)a.x : (const void *)(ws + L.x16));
        uint16_t *xs = reinterpret_cast<uint16_t *>(ws + L.xs);
        int32_t *inv = reinterpret_cast<int32_t *>(ws + L.inv);
        void *cargs[] = {&idx, &T, &base, &list, &inv, &flag};
        e = launch_ex((const void *)moe_grouped_scatter_kernel, dim3(nc), dim3(G_TOK_PER_CTA * TOPK), 0, st, cargs);
        if (e != cudaSuccess)
            return e;
        void *gargs[] = {&list, &offsets, &T, &src, &xs};
        e = launch_ex((const void *)moe_grouped_gather_kernel, dim3(nsm * 8), dim3(256), 0, st, gargs);
        if (e != cudaSuccess)
            return e;
    }
    const bool f16 = !a.bf16w;
    GArgs g{};
    g.T = a.T;
    g.nmax = G_NMAX;
    g.a_bf16 = a.bf16w;
    g.f16 = f16 ? 1 : 0;
    g.n_shared = a.n_shared;
    g.flag = flag;
    g.counts = counts;
    g.offsets = offsets;
    g.list = list;
    g.topk_w = reinterpret_cast<const float *>(ws + L.w);
    g.h_routed = reinterpret_cast<__nv_bfloat16 *>(ws + L.h_routed);
    g.h_shared = reinterpret_cast<__nv_bfloat16 *>(ws + L.h_shared);
    g.ybuf = reinterpret_cast<float *>(ws + L.ybuf);
    g.ysh = reinterpret_cast<float *>(ws + L.ysh);
    g.out = a.out;
    int32_t *hshift = reinterpret_cast<int32_t *>(ws + L.hshift);
    if (f16) {
        g.xshift = reinterpret_cast<const int32_t *>(ws + L.xshift);
        g.hshift_r = hshift;
        g.hshift_s = hshift + (size_t)T * TOPK;
    }
    const void *xb = f16 ? (const void *)(ws + L.x16) : (const void *)a.x;
    const size_t nrows = (size_t)T * TOPK;
    // gate/up: routed experts (listed tokens) and the shared expert (all tokens)
    g.mode = GM_GATE_UP;
    g.K = H;
    g.mtiles = 2 * I / 128;
    g.ra = a.r_w13;
    g.sa = a.s_w13;
    g.rts = a.r_ts13;
    g.sts = a.s_ts13;
    g.a_stride = a.bf16w ? W13_BYTES_BF : W13_BYTES;
    if ((e = launch_gemm(g, ws + L.xs, nrows, xb, (size_t)T, H, nsm, st)) != cudaSuccess)
        return e;
    if (f16) {
        // h_routed and h_shared are consecutive: one pass over all rows
        uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h_routed);
        int rows = T * TOPK + (a.n_shared ? T : 0);
        void *hargs[] = {&h, &rows, &hshift};
        if ((e = launch_ex((const void *)moe_grouped_hscale_kernel, dim3(nsm * 8), dim3(256), 0, st, hargs)) !=
            cudaSuccess)
            return e;
    }
    // down: routed experts -> weighted rows of ybuf
    g.mode = GM_DOWN;
    g.K = I;
    g.mtiles = H / 128;
    g.ra = a.r_w2;
    g.sa = a.s_w2;
    g.rts = a.r_ts2;
    g.sts = a.s_ts2;
    g.a_stride = a.bf16w ? W2_BYTES_BF : W2_BYTES;
    if ((e = launch_gemm(g, ws + L.h_routed, nrows, nullptr, 0, I, nsm, st)) != cudaSuccess)
        return e;
    if (a.n_shared) {
        g.mode = GM_SHARED_DOWN;
        if ((e = launch_gemm(g, nullptr, 0, ws + L.h_shared, (size_t)T, I, nsm, st)) != cudaSuccess)
            return e;
    }
    const float *yb = g.ybuf;
    const float *ys = a.n_shared ? g.ysh : nullptr;
    __nv_bfloat16 *out = a.out;
    const int32_t *inv = reinterpret_cast<const int32_t *>(ws + L.inv);
    void *cargs[] = {&yb, &inv, &ys, &T, &out};
    return launch_ex((const void *)moe_grouped_combine_kernel, dim3(nsm * 8), dim3(256), 0, st, cargs);
}

}  // namespace moe

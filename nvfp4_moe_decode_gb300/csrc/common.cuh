// common.cuh -- shared constants, the packed NVFP4 layout and inline-PTX
// helpers of the sm_103a kernels behind libnvfp4moe.so.
//
// Packed NVFP4 layout (ours; a lossless permutation of the canonical bytes,
// repacked at load time as the Flint page, "A 40B MoE that activates 2.5B
// parameters", describes for its checkpoint):
//
//   A matrix W[N][K] is cut into N/16 bands of 16 rows.  Band b is 9*K bytes
//   made of K/128 super-chunks of 1152 bytes; super-chunk q covers columns
//   [128q, 128q+128): 1024 bytes of e2m1 codes followed by 128 bytes of e4m3
//   scales, so any run of whole super-chunks is one contiguous copy.
//   Codes: the two 512-byte chunks j = 2q, 2q+1 (64 columns each).  In a
//   chunk, lane l = 4*g + c (g = l/4, c = l%4) owns 16 bytes = four 32-bit
//   words, word s for the k16 step s of the chunk (k0 = 64*j + 16*s).  Byte r
//   of a word is register r of the mma.m16n8k16 A fragment: band row
//   g + 8*(r & 1), columns k0 + 2*c + 8*(r >> 1) + {0 (low nibble),
//   1 (high nibble)}.
//   Scales: the 16 bytes at 1024 + 16*g hold, at byte 2*sb + h, the scale of
//   band row g + 8*h for the 16-column block 8*q + sb.
//   Band rows: PLAIN band b row i = matrix row 16*b + i.  GATE_UP (a W13
//   matrix, N = 2*I): row i < 8 is gate row 8*b + i, row i >= 8 is up row
//   N/2 + 8*b + (i - 8), so that one mma accumulator tile holds matching gate
//   and up rows for the SiLU*up epilogue.
//
// In-register decode: cvt.rn.f16x2.e2m1x2 turns one code byte into the two
// exact e2m1 values of an A register.  The activations (bf16) enter the
// tensor cores as fp16 after an exact per-token power-of-two rescale that puts
// the token's largest magnitude in [2^14, 2^15): bf16's 8-bit significand
// fits fp16's 11 bits, so every element within 2^28 of the largest (the
// normal f16 range after the rescale) is exact; smaller ones become f16
// subnormals, still exact down to 2^-31 of the largest, and only elements
// below that (whose products lie far below the fp32 rounding of the sum)
// are rounded.  Products are exact and accumulate in fp32; the e4m3
// block scale is applied to each k16 step's fp32 partial, the tensor scale
// and the power of two at the end.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4moe.h"

namespace moe {

constexpr int H = MOE_HIDDEN;            // 2048
constexpr int I = MOE_INTER;             // 512
constexpr int E = MOE_EXPERTS;           // 256
constexpr int TOPK = MOE_TOPK;           // 6
constexpr int MAXT = MOE_MAX_DECODE_T;   // 8
constexpr int MAX_SHARED = 1;                        // shared experts inside the layer kernel
constexpr int MAX_SLOTS = MAX_SHARED + MAXT * TOPK;  // 49
// Shared experts computed ahead of the layer kernel by the dense GEMV (two
// at most: a pair of expert sinks, or shared experts of another weight type
// than the routed bank); their router rows follow the routed ones.
constexpr int MAX_EXT = 2;
constexpr int LE = E + MAX_EXT;                      // router rows the tagged logits have room for

__host__ __device__ constexpr size_t band_bytes(int K) { return (size_t)9 * K; }
constexpr int W13_BANDS = 2 * I / 16;                       // 64
constexpr int W2_BANDS = H / 16;                            // 128
constexpr size_t W13_BAND_BYTES = band_bytes(H);            // 18432
constexpr size_t W2_BAND_BYTES = band_bytes(I);             // 4608
constexpr size_t W13_BYTES = W13_BANDS * W13_BAND_BYTES;    // 1179648
constexpr size_t W2_BYTES = W2_BANDS * W2_BAND_BYTES;       // 589824
constexpr size_t W13_BYTES_BF = (size_t)2 * I * H * 2;     // 4194304: bf16 W13 of one expert
constexpr size_t W2_BYTES_BF = (size_t)H * I * 2;          // 2097152: bf16 W2 of one expert

constexpr int SC_BYTES = 1152;            // one 128-column super-chunk of a band
constexpr int ACT_EXP = 14;               // activations scaled so max|v| is in [2^14, 2^15)

// Device flag bits (mirrors of the public MOE_FLAG_*).
constexpr uint32_t FLAG_NONFINITE = MOE_FLAG_NONFINITE_LOGIT;
constexpr uint32_t FLAG_TIMEOUT = MOE_FLAG_WAIT_TIMEOUT;
constexpr uint32_t FLAG_BAD_INDEX = MOE_FLAG_BAD_INDEX;

// Bounded spin: a wait that has not completed after this many polls gives up,
// sets FLAG_TIMEOUT and lets the kernel finish.
constexpr uint32_t SPIN_LIMIT = 1u << 20;

// ---------------------------------------------------------------------------
// Workspace layout (bytes from the workspace base; 256-byte aligned regions).
// ---------------------------------------------------------------------------
struct WsLayout {
    size_t ctrl;       // u32[64]: [0] device flag, [1] routing-kernel arrivals,
                       //   [4] layer-kernel CTAs that have read the launch tag, [5] layer-kernel launches
    size_t logits;     // f32[MAXT][E]
    size_t tlogits;    // u64[MAXT][LE]: layer kernel, (launch tag << 32) | fp32 logit bits
    size_t topk_idx;   // i32[MAXT][TOPK]
    size_t topk_w;     // f32[MAXT][TOPK]
    size_t slots;      // SlotTable
    size_t htag;       // u64[MAX_SLOTS][W13_BANDS][MAXT][4]: (launch tag << 32) | the bf16 SiLU*up
                       //   values of h rows 8 b + 2 w (low half) and 8 b + 2 w + 1 of token t
    size_t ptag;       // u64[MAX_SLOTS][W2_BANDS][16][MAXT]: (launch tag << 32) | fp32 weighted
                       //   down output of row 16 b + r, token t
    size_t ext_h;      // bf16[MAX_EXT][MAXT][I]: SiLU*up of the shared experts run ahead
    size_t ext_y;      // f32[MAX_EXT][MAXT][H]: their down outputs (unweighted)
    size_t sinkw;      // f32[MAXT][MAX_EXT]: the weight of each of them per token
    size_t total;
};

struct SlotTable {
    int32_t n_slots;                  // shared slots first, then sorted distinct experts
    int32_t n_shared;
    int32_t expert[MAX_SLOTS];        // routed expert id, or -1 - s for shared expert s
    float wts[MAX_SLOTS][MAXT];       // routing weight of token t for the slot (0 if unused)
};

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

__host__ __device__ inline WsLayout ws_layout()
{
    WsLayout L;
    size_t o = 0;
    L.ctrl = o;      o = align256(o + 64 * 4);
    L.logits = o;    o = align256(o + (size_t)MAXT * E * 4);
    L.tlogits = o;   o = align256(o + (size_t)MAXT * LE * 8);
    L.topk_idx = o;  o = align256(o + (size_t)MAXT * TOPK * 4);
    L.topk_w = o;    o = align256(o + (size_t)MAXT * TOPK * 4);
    L.slots = o;     o = align256(o + sizeof(SlotTable));
    L.htag = o;      o = align256(o + (size_t)MAX_SLOTS * W13_BANDS * MAXT * 4 * 8);
    L.ptag = o;      o = align256(o + (size_t)MAX_SLOTS * W2_BANDS * 16 * MAXT * 8);
    L.ext_h = o;     o = align256(o + (size_t)MAX_EXT * MAXT * I * 2);
    L.ext_y = o;     o = align256(o + (size_t)MAX_EXT * MAXT * H * 4);
    L.sinkw = o;     o = align256(o + (size_t)MAXT * MAX_EXT * 4);
    L.total = o;
    return L;
}

// ---------------------------------------------------------------------------
// Packed-layout index maps (host and device).
// ---------------------------------------------------------------------------

// Band row i (0..15) of band b -> matrix row.
__host__ __device__ inline int band_row_to_matrix_row(int kind, int N, int b, int i)
{
    if (kind == MOE_PACK_GATE_UP)
        return (i < 8) ? 8 * b + i : N / 2 + 8 * b + (i - 8);
    return 16 * b + i;
}

// Matrix row n -> (band, band row).
__host__ __device__ inline void matrix_row_to_band(int kind, int N, int n, int &b, int &i)
{
    if (kind == MOE_PACK_GATE_UP) {
        if (n < N / 2) { b = n / 8; i = n % 8; }
        else { int m = n - N / 2; b = m / 8; i = 8 + m % 8; }
    } else {
        b = n / 16; i = n % 16;
    }
}

// Packed code nibble of element (band row i, column k) within its band:
// byte offset from the band start and nibble (0 = low, 1 = high).
__host__ __device__ inline void code_position(int i, int k, int &byte_off, int &nib)
{
    int j = k / 64, s = (k % 64) / 16, kk = k % 16;
    int hi = kk & 1, c = (kk & 7) >> 1, rhi = kk >> 3;
    int g = i & 7, rlo = i >> 3;
    int r = rlo + 2 * rhi;
    int lane = 4 * g + c;
    byte_off = (j >> 1) * SC_BYTES + (j & 1) * 512 + lane * 16 + s * 4 + r;
    nib = hi;
}

// Inverse of code_position: (byte offset of a code byte within the band,
// nibble) -> (band row, column).  The byte must be a code byte.
__host__ __device__ inline void code_element(int byte_off, int nib, int &i, int &k)
{
    int q = byte_off / SC_BYTES, rem0 = byte_off % SC_BYTES;
    int j = 2 * q + rem0 / 512, rem = rem0 % 512;
    int lane = rem / 16, w = rem % 16;
    int s = w / 4, r = w % 4;
    int g = lane >> 2, c = lane & 3;
    i = g + 8 * (r & 1);
    k = 64 * j + 16 * s + 2 * c + 8 * (r >> 1) + nib;
}

__host__ __device__ inline bool is_scale_byte(int byte_off) { return byte_off % SC_BYTES >= 1024; }

// Packed scale byte of (band row i, block bk) within the band.
__host__ __device__ inline int scale_position(int i, int bk)
{
    int q = bk / 8, sb = bk % 8;
    int g = i & 7, h = i >> 3;
    return q * SC_BYTES + 1024 + g * 16 + 2 * sb + h;
}

__host__ __device__ inline void scale_element(int off, int &i, int &bk)
{
    int q = off / SC_BYTES, rem = off % SC_BYTES - 1024;
    int g = rem / 16, w = rem % 16;
    int sb = w / 2, h = w % 2;
    i = g + 8 * h;
    bk = 8 * q + sb;
}

#ifdef __CUDACC__

// ---------------------------------------------------------------------------
// Decode: byte r of a packed code word -> the f16x2 A-fragment register r.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t decode_reg(uint32_t w, int r)
{
    uint32_t h2;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(h2) : "r"(w >> (8 * r)));
    return h2;
}

// Two e4m3 scale bytes (low byte -> .x) to fp32 (exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_bytes)
{
    uint32_t h2;
    asm("{\n\t.reg .b16 b;\n\tcvt.u16.u32 b, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, b;\n\t}"
        : "=r"(h2) : "r"(two_bytes));
    __half2 hh = *reinterpret_cast<__half2 *>(&h2);
    return __half22float2(hh);
}

// ---------------------------------------------------------------------------
// Tensor core: D = A(16x16 f16, row) * B(16x8 f16, col), fp32, C = 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier + bulk async copy (TMA, non-tensor).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: returns false (after setting the timeout flag) if the phase
// did not complete within SPIN_LIMIT polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t *flag)
{
    for (uint32_t it = 0; it < SPIN_LIMIT; ++it)
        if (mbar_try_wait(bar, parity))
            return true;
    atomicOr(flag, FLAG_TIMEOUT);
    return false;
}

// Global -> shared bulk copy completing on `bar` (bytes % 16 == 0, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Exponent e such that 2^e <= v < 2^(e+1) for a finite v > 0 (0 for v = 0).
__device__ __forceinline__ int exponent_of(float v)
{
    if (!(v > 0.0f) || !isfinite(v))
        return 0;
    return ((int)((__float_as_uint(v) >> 23) & 0xFF)) - 127;
}

// Two bf16 values (low first) times 2^sh, as an f16x2 (exact in the range
// described at the top of this file).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t v, float pow2)
{
    const float lo = __uint_as_float(v << 16) * pow2;
    const float hi = __uint_as_float(v & 0xFFFF0000u) * pow2;
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ __nv_bfloat162 u32_as_bf162(uint32_t v)
{
    __nv_bfloat162 r;
    *reinterpret_cast<uint32_t *>(&r) = v;
    return r;
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16)
{
    return __uint_as_float(bits16 << 16);
}

#endif  // __CUDACC__

}  // namespace moe

// stage.cuh -- the per-stage tensor-core steps shared by the decode layer
// and the dense GEMV: in-register NVFP4 decode into mma.sync A fragments,
// BF16 ring stages, and the activation power-of-two rescale.
//
// A stage is the unit of one ring slot of a streaming warp: NVFP4, two
// consecutive super-chunks of a band (16 rows x 256 columns, 2304 bytes, one
// bulk copy); BF16, 16 rows x 64 columns (2048 bytes, 32 lanes x four 16-byte
// cp.async, swizzled so that the fragment reads do not conflict).
#pragma once

#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float pow2i(int k) { return __int_as_float((127 + k) << 23); }

__device__ __forceinline__ int act_shift(float maxabs)
{
    int sh = ACT_EXP - exponent_of(maxabs);
    return sh < -100 ? -100 : (sh > 100 ? 100 : sh);
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

// The same with the B fragments read from activations staged row-major in
// shared memory, token t's row at word t * rpw (rpw = K / 2 + 4: rows 16
// bytes apart, so that the 32 lanes' words fall in 32 different banks):
// lane (g, c) takes words 8 step + c and 8 step + 4 + c of token g's row
// (columns 16 step + 2 c, +1 and 16 step + 8 + 2 c, +1).
__device__ __forceinline__ void mma_stage_xs(const uint8_t *stage, const uint32_t *xs, int rpw, int step0, int lane,
                                             float acc[4])
{
    const int g = lane >> 2, c = lane & 3;
    const uint32_t *xrow = xs + g * rpw + c;
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
                uint32_t a0, a1, a2, a3;
                decode4(words[s], a0, a1, a2, a3);
                float d[4];
                mma_f16_16816(d, a0, a1, a2, a3, xrow[8 * step], xrow[8 * step + 4]);
                const int sb = half * 4 + s;
                const uint32_t sw = sws[sb >> 1];
                const float2 sf = e4m3x2_to_float2((sb & 1) ? (sw >> 16) : (sw & 0xFFFFu));
                ffma2(acc[0], acc[1], sf.x, d[0], d[1]);
                ffma2(acc[2], acc[3], sf.y, d[2], d[3]);
            }
        }
    }
}

// BF16: one 64-column ring stage (see bf16_stage) with the B fragments of
// k16 steps step0 .. step0 + 3 read from the row-major staging (the four
// columns of lane (g, c) at bf16_bcol(step, c)).
__device__ __forceinline__ void bf16_stage_xs(const uint8_t *stage, const uint32_t *xs, int rpw, int step0, int lane,
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
        const uint2 b = *reinterpret_cast<const uint2 *>(xs + g * rpw + bf16_bcol(step0 + s, c) / 2);
        mma_bf16_16816(acc, wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1], b.x, b.y);
    }
}

}  // namespace
}  // namespace moe

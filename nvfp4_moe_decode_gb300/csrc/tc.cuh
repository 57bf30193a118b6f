// tc.cuh -- inline-PTX helpers for the fifth-generation tensor cores
// (tcgen05: MMAs with operands in shared memory and the accumulator in tensor
// memory) and the asynchronous copies that feed them, for sm_103a.
//
// Operand layout used by every tcgen05 GEMM in this library: K-major tiles
// of 64 bf16 (128 bytes) per row with the 128-byte swizzle: row r of a tile
// (1024-byte aligned base) occupies bytes [128 r, 128 r + 128), and its
// 16-byte chunk c (columns 8c .. 8c+7 of the 64) is stored at chunk position
// c ^ (r % 8).  Eight rows form one 1024-byte swizzle atom; atoms follow each
// other along M (or N) at 1024 bytes.
#pragma once

#include "common.cuh"

namespace moe {

#ifdef __CUDACC__

constexpr int TC_KCHUNK = 64;                 // K per swizzled tile row (bf16)
constexpr int TC_ROW_BYTES = 128;

// Byte offset of (row r, 16-byte chunk c) in a 128B-swizzled K-major tile.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int c)
{
    return (uint32_t)(r * TC_ROW_BYTES + ((c ^ (r & 7)) << 4));
}

// Shared-memory matrix descriptor of a 128B-swizzled K-major operand:
// start address >> 4 (bits 0-13), stride between 8-row atoms 1024 B >> 4
// (bits 32-45), the fixed version bits 46-48 = 0b001, swizzle mode 2 =
// 128-byte swizzle (bits 61-63).  The leading-dimension offset is unused
// for swizzled K-major layouts.  Advancing K by 16 elements adds 32 bytes
// to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr)
{
    return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptors of kind::f16, both operands K-major, an fp32
// accumulator (bits 4-5 = 1), M = 128 (bits 24-28 = M / 16) and the given N
// (multiple of 16, <= 256; bits 17-22 = N / 8); operand formats in bits 7-9
// (A) and 10-12 (B): 0 = f16, 1 = bf16.
__host__ __device__ __forceinline__ uint32_t idesc_bf16_m128(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__host__ __device__ __forceinline__ uint32_t idesc_f16_m128(int n)
{
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void tc_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] x B[smem desc]^T (kind::f16: f16 or bf16
// operands as the instruction descriptor says), one thread.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_addr(bar)) : "memory");
}

// 32 lanes x 32 consecutive fp32 columns (lane quarter of the warp).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float v[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// 16-byte global -> shared copy (cp.async); src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void st_shared32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

#endif  // __CUDACC__

}  // namespace moe

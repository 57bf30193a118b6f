// kernels.cuh -- argument blocks and host launchers of the kernels behind
// libnvfp4moe.so (internal; not part of the public C ABI).
#pragma once

#include "common.cuh"

namespace moe {

constexpr int CONSUMER_WARPS = 8;
constexpr int EXPERT_THREADS = (CONSUMER_WARPS + 1) * 32;   // 288
constexpr int CONSUMER_THREADS = CONSUMER_WARPS * 32;       // 256

constexpr int GU_STAGES = 4;
constexpr int GU_STEPS = H / 16;                                  // 128 k16 steps
constexpr int GU_CHUNKS_PER_WARP = (H / 64) / CONSUMER_WARPS;     // 4
constexpr size_t GU_SMEM_STAGES = GU_STAGES * W13_BAND_BYTES;     // 73728
constexpr size_t GU_SMEM_XFRAG = (size_t)GU_STEPS * 32 * 8;       // 32768
constexpr size_t GU_SMEM_RED = CONSUMER_WARPS * 32 * 4 * 4;       // 4096
constexpr size_t GU_SMEM_BARS = 2 * GU_STAGES * 8;
constexpr size_t GU_SMEM = GU_SMEM_STAGES + GU_SMEM_XFRAG + GU_SMEM_RED + GU_SMEM_BARS;
constexpr int DN_STEPS = I / 16;                 // 32 k16 steps
constexpr int DN_MAX_SG = 4;

struct RouterArgs {
    const __nv_bfloat16 *x;        // [T][H]
    const __nv_bfloat16 *wr;       // [E][H]
    int T;
    int n_shared;                  // 0 or 1
    uint8_t *ws;                   // workspace base
    int32_t *user_idx;             // optional [T][TOPK]
    float *user_w;                 // optional [T][TOPK]
    float *user_logits;            // optional [T][E]
};

struct GateUpArgs {
    const __nv_bfloat16 *x;   // [T][H]
    int T;
    const uint8_t *routed_w13;
    const float *routed_ts13;
    const uint8_t *shared_w13;
    const float *shared_ts13;
    int n_shared;
    uint8_t *ws;
};

struct DownArgs {
    int T;
    const uint8_t *routed_w2;
    const float *routed_ts2;
    const uint8_t *shared_w2;
    const float *shared_ts2;
    int n_shared;
    int BG;   // bands per CTA (1, 2, 4 or 8)
    int SG;   // slots per CTA (1..DN_MAX_SG)
    uint8_t *ws;
    __nv_bfloat16 *out;   // [T][H]
};

__host__ __device__ inline size_t down_smem_bytes(int BG, int SG)
{
    return (size_t)SG * BG * W2_BAND_BYTES + (size_t)SG * DN_STEPS * 32 * 8 +
           (size_t)CONSUMER_WARPS * 32 * 4 * 4 + (size_t)DN_MAX_SG * 8;
}

struct PackArgs {
    const uint8_t *codes;    // [count][N][K/2]
    const uint8_t *scales;   // [count][N][K/16]
    uint8_t *packed;         // [count][N/16][9K]
    int N, K, kind, count;
};

struct UnpackArgs {
    const uint8_t *packed;
    uint8_t *codes;
    uint8_t *scales;
    int N, K, kind, count;
};

struct DequantArgs {
    const uint8_t *packed;
    float *out;   // [N][K]
    int N, K, kind;
    float tscale;
};

cudaError_t launch_router(const RouterArgs &a, cudaStream_t stream, bool pdl);
cudaError_t launch_gate_up(const GateUpArgs &a, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_down(const DownArgs &a, int qmax, cudaStream_t stream, bool pdl);
cudaError_t launch_pack(const PackArgs &a, cudaStream_t s);
cudaError_t launch_unpack(const UnpackArgs &a, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs &a, cudaStream_t s);

}  // namespace moe

// kernels.cuh -- argument blocks, tiling constants and host launchers of the
// kernels behind libnvfp4moe.so (internal; not part of the public C ABI).
#pragma once

#include "common.cuh"

namespace moe {

// K2 gate/up: one CTA per SM, 8 warps, each with a private ring of stages.
constexpr int GU_WARPS = 8;
constexpr int GU_RING = 4;                                   // stages per warp
constexpr int GU_SC_PER_STAGE = 2;                           // super-chunks per stage
constexpr int GU_STAGE_BYTES = GU_SC_PER_STAGE * SC_BYTES;   // 2304
constexpr int GU_STEPS = H / 16;                             // 128 k16 steps

// K3 down: one CTA per SM, 8 warps in groups of BG warps (one band each).
constexpr int DN_WARPS = 8;
constexpr int DN_RING = 2;                                   // W2 bands per warp in flight
constexpr int DN_STEPS = I / 16;                             // 32 k16 steps
constexpr int DN_HBUF_ENTRIES = 4096;                        // 32 KB of h fragments per CTA

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
    const __nv_bfloat16 *x;        // [T][H]
    int T;
    int KS;                        // warps that split one band's K (1, 2 or 4)
    const uint8_t *routed_w13;
    const float *routed_ts13;
    const uint8_t *shared_w13;
    const float *shared_ts13;
    int n_shared;
    uint8_t *ws;
};

struct DownArgs {
    int T;
    int BG;                        // bands (warps) per unit: 2, 4 or 8
    const uint8_t *routed_w2;
    const float *routed_ts2;
    const uint8_t *shared_w2;
    const float *shared_ts2;
    int n_shared;
    uint8_t *ws;
};

struct CombineArgs {
    int T;
    uint8_t *ws;
    __nv_bfloat16 *out;            // [T][H]
};

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

size_t gate_up_smem_bytes();
size_t down_smem_bytes();

cudaError_t launch_router(const RouterArgs &a, cudaStream_t stream, bool pdl);
cudaError_t launch_gate_up(const GateUpArgs &a, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_down(const DownArgs &a, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream, bool pdl);
cudaError_t launch_pack(const PackArgs &a, cudaStream_t s);
cudaError_t launch_unpack(const UnpackArgs &a, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs &a, cudaStream_t s);

}  // namespace moe

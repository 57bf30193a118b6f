// kernels.cuh -- argument blocks, tiling constants and host launchers of the
// kernels behind libnvfp4moe.so (internal; not part of the public C ABI).
#pragma once

#include "common.cuh"

namespace moe {

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

struct LayerArgs {
    const __nv_bfloat16 *x;        // [T][H]
    const __nv_bfloat16 *wr;       // [E][H]
    int T;
    const uint8_t *r_w13, *r_w2;   // routed bank (packed NVFP4, or bf16 row-major if bf16w)
    const float *r_ts13, *r_ts2;   // NVFP4 only
    const uint8_t *s_w13, *s_w2;   // shared expert (same weight type), if n_shared
    const float *s_ts13, *s_ts2;   // NVFP4 only
    int n_shared;
    int bf16w;                     // 1: both banks hold bf16 weights
    // pre-norm mode (a layer of a decoder stack): the input is
    // RMSNorm(bf16(x + delta)); x is the residual stream, delta (may be null)
    // the previous layer's output; resid_out / xn_out (may be null) receive
    // bf16(x + delta) and the normalised input
    int prenorm;
    const __nv_bfloat16 *delta;
    __nv_bfloat16 *resid_out;
    __nv_bfloat16 *xn_out;
    float eps;
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

size_t layer_smem_bytes();

cudaError_t launch_router(const RouterArgs &a, cudaStream_t stream, bool pdl);
cudaError_t launch_layer(const LayerArgs &a, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_pack(const PackArgs &a, cudaStream_t s);
cudaError_t launch_unpack(const UnpackArgs &a, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs &a, cudaStream_t s);
cudaError_t launch_residual_add(const __nv_bfloat16 *a, const __nv_bfloat16 *b, __nv_bfloat16 *out, int n,
                                cudaStream_t stream, bool pdl);

}  // namespace moe

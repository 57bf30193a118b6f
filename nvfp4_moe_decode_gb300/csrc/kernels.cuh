// kernels.cuh -- argument blocks, tiling constants and host launchers of the
// kernels behind libnvfp4moe.so (internal; not part of the public C ABI).
#pragma once

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Host: a value computed once per device, safe to use from several host
// threads.  make(dev) runs with that device current and returns the value
// (> 0), or <= 0 on failure (not cached; the next call tries again).
// ---------------------------------------------------------------------------
constexpr int MAX_DEVICES = 64;

struct PerDevice {
    std::atomic<int> v[MAX_DEVICES];   // 0: not computed yet
    std::mutex mu;
};

template <class F>
int per_device(PerDevice &pd, F make)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return -1;
    int v = pd.v[dev].load(std::memory_order_acquire);
    if (v > 0)
        return v;
    std::lock_guard<std::mutex> lock(pd.mu);
    v = pd.v[dev].load(std::memory_order_relaxed);
    if (v > 0)
        return v;
    v = make(dev);
    if (v > 0)
        pd.v[dev].store(v, std::memory_order_release);
    return v;
}

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
    int bf16w;                     // 1: the routed bank (and an inside shared expert) holds bf16 weights
    // shared experts run ahead by the dense GEMV: n_ext (0..MAX_EXT) down
    // outputs in ext_y, added in the combine with weight 1, or, when they are
    // expert sinks (n_sink = n_ext), their sigmoid score over the
    // denominator, which their router rows E.. join
    int n_ext;
    int n_sink;
    const float *ext_y;            // f32 [MAX_EXT][MAXT][H]
    // a chunk of a larger batch: CTA 0 also writes this chunk's selection,
    // weights and fp32 logits at token offset t0 of these arrays (or null)
    int32_t *r_idx;                // [..][TOPK]
    float *r_w;                    // [..][TOPK]
    float *r_logits;               // [..][E]
    int t0;
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

// ---------------------------------------------------------------------------
// Mid-size batches: MAXT < T <= chunk_max_t(weight type) tokens run the
// decode kernel on balanced chunks of at most MAXT tokens (the grouped
// path's fixed cost is higher there).  Measured on GB300, µs per layer:
// NVFP4 decode 326 at 88 tokens (11 chunks) against 341 grouped, 356 at 96
// against 346; BF16 decode 381 at 48 against 419, 508 at 64 against 458.
// Each chunk's routing is kept after the decode workspace, where the grouped
// path keeps its routing too, for moe_read_routing.
// ---------------------------------------------------------------------------
constexpr int CHUNK_MAX_T = MOE_MAX_CHUNKED_T;          // the larger of the two limits
constexpr int CHUNK_MAX_T_BF16 = MOE_MAX_CHUNKED_T_BF16;
inline int chunk_max_t(int wtype) { return wtype == MOE_W_BF16 ? CHUNK_MAX_T_BF16 : CHUNK_MAX_T; }

struct ChunkRouteLayout {
    size_t idx;      // i32 [T][TOPK]
    size_t w;        // f32 [T][TOPK]
    size_t logits;   // f32 [T][E]
    size_t total;
};

__host__ __device__ inline ChunkRouteLayout chunk_route_layout(int T)
{
    ChunkRouteLayout c;
    size_t o = ws_layout().total;
    c.idx = o;     o = align256(o + (size_t)T * TOPK * 4);
    c.w = o;       o = align256(o + (size_t)T * TOPK * 4);
    c.logits = o;  o = align256(o + (size_t)T * E * 4);
    c.total = o;
    return c;
}

// ---------------------------------------------------------------------------
// Dense small-batch GEMV (T <= MAXT): see gemv.cu.
// ---------------------------------------------------------------------------
enum GemvEpi {
    GEMV_OUT_BF16 = 0,   // y[m][t][n] = bf16(sum)
    GEMV_OUT_F32 = 1,    // y[m][t][n] = sum (fp32)
    GEMV_SILU_H = 2,     // GATE_UP bands: y[m][t][i] = bf16(silu(gate_i) * up_i), i < N / 2
};
constexpr int GEMV_MAX_K_RW4 = 4096;   // four ring stages per warp up to here
constexpr int GEMV_MAX_K = 8192;       // two beyond (x takes 16 K bytes of shared memory)

struct GemvArgs {
    const __nv_bfloat16 *x;        // [n_mat][T][K] (x_mat_stride elements apart; 0: one x for all)
    size_t x_mat_stride;
    const uint8_t *w;              // n_mat matrices, w_mat_stride bytes apart: packed NVFP4 or bf16 [N][K]
    size_t w_mat_stride;
    const float *ts_dev;           // NVFP4: per-matrix tensor scales on the device, or null (ts_host)
    float ts_host;
    int N, K, T, n_mat;
    int kind;                      // MOE_PACK_PLAIN or MOE_PACK_GATE_UP (band rows)
    int bf16w;
    int epi;                       // GemvEpi
    void *y;                       // output, y_mat_stride elements apart
    size_t y_mat_stride;
    uint32_t *flag;                // device flag word
    int q;                         // set by launch_gemv: warps per band
    int ctas_per_mat;              // set by launch_gemv
};

// Warps per band for a CTA holding `bands_per_cta` bands of `stages` stages.
int gemv_warps_per_band(int bands_per_cta, int stages, int unit);
// cuTensorMapEncodeTiled (null if the driver does not provide it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
cudaError_t launch_gemv(GemvArgs a, int sm_count, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Grouped path (T > MAXT): see grouped.cu.
// ---------------------------------------------------------------------------
constexpr int G_NMAX = 256;            // tokens per GEMM tile
constexpr int G_TOK_PER_CTA = 32;      // tokens per CTA of the top-k / list kernels (one warp per token)
constexpr int MAX_TOKENS = MOE_MAX_TOKENS;

enum GMode { GM_ROUTER = 0, GM_GATE_UP = 1, GM_DOWN = 2, GM_SHARED_DOWN = 3 };

// Workspace of the grouped path for T tokens (bytes from the base).
struct GWsLayout {
    size_t ctrl;       // u32[64], [0] device flag (same place as the decode layout)
    size_t logits;     // f32[T][E]
    size_t idx;        // i32[T][TOPK]
    size_t w;          // f32[T][TOPK]
    size_t counts;     // i32[E]
    size_t offsets;    // i32[E + 1]
    size_t list;       // i32[T * TOPK]: 6 t + i, grouped by expert, increasing within an expert
    size_t hist;       // i32[ceil(T / G_TOK_PER_CTA)][E] selections per expert of each top-k CTA
    size_t base;       // i32[ceil(T / G_TOK_PER_CTA)][E] first list row of each (CTA, expert)
    size_t x16;        // f16[T][H]: x times 2^xshift[t] (NVFP4 weights)
    size_t xs;         // [T * TOPK][H]: the GEMM operand row (x16 or x) of each list row
    size_t xshift;     // i32[T]
    size_t hshift;     // i32[T * TOPK + T]: power of two of each h row (routed rows, then shared)
    size_t h_routed;   // [T * TOPK][I]: SiLU*up of list row r (bf16; f16 x 2^hshift after the rescale)
    size_t h_shared;   // [T][I], directly after h_routed
    size_t ybuf;       // f32[T * TOPK][H]: weighted down output of (token, choice), in list order
    size_t ysh;        // f32[T][H]: the shared expert's down output
    size_t inv;        // i32[T][TOPK]: list row of (token, choice), -1 if invalid
    size_t total;
};
GWsLayout gws_layout(int T);

// Arguments of one grouped GEMM launch.
struct GArgs {
    int mode;                       // GMode
    int T;
    int nmax;                       // tokens per tile (multiple of 16, <= G_NMAX)
    int a_bf16;                     // A rows are bf16 (else packed NVFP4, dequantised to f16)
    int f16;                        // operands are f16 (else bf16)
    int K;                          // reduction length
    int mtiles;                     // 128-row M tiles per group
    int n_shared;
    const uint8_t *ra, *sa;         // routed bank / shared expert matrix (packed or bf16)
    const float *rts, *sts;         // tensor scales (NVFP4)
    size_t a_stride;                // bytes per routed expert matrix
    const __nv_bfloat16 *wr;        // router weights (router mode)
    const __nv_bfloat16 *x;         // [T][H]
    uint32_t *flag;
    float *logits;
    const int32_t *counts, *offsets, *list;
    const float *topk_w;
    __nv_bfloat16 *h_routed, *h_shared;
    float *ybuf;                    // [T * TOPK][H] weighted routed outputs, in list order
    float *ysh;                     // [T][H] the shared expert's down projection
    __nv_bfloat16 *out;
    const int32_t *xshift;          // per token (f16 operands), or null
    const int32_t *hshift_r, *hshift_s; // per routed / shared h row (f16 operands), or null
};

// Arguments of the grouped layer (host side).
struct GroupedArgs {
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *wr;
    int T;
    int bf16w;
    int n_shared;
    int convert_x;                  // also write x16 / xshift (set by the launcher)
    const uint8_t *r_w13, *r_w2, *s_w13, *s_w2;
    const float *r_ts13, *r_ts2, *s_ts13, *s_ts2;
    uint8_t *ws;
    __nv_bfloat16 *out;
};

cudaError_t launch_grouped_route(const GroupedArgs &a, int nsm, cudaStream_t stream);
cudaError_t launch_grouped_layer(const GroupedArgs &a, int nsm, cudaStream_t stream);

size_t layer_smem_bytes();
// CTAs of the decode layer kernel that one SM can hold at once (its shared
// memory and register needs; sets the kernel's shared-memory attribute on
// first use), or -1 on a CUDA error.
int layer_resident_ctas_per_sm();
// Re-arm a decode workspace after a wait timeout (see moe_workspace_recover).
cudaError_t launch_rearm(uint8_t *ws, cudaStream_t stream, bool pdl);
// moe_layer_forward (sink: moe_layer_forward_sink); with rearm, a decode
// call first enqueues launch_rearm on its workspace (after all host-side
// checks).
moe_status layer_forward(const void *x, const void *router_w, const moe_expert_bank *routed,
                         const moe_expert_bank *shared, void *out, int T, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream, bool rearm, bool sink = false);

cudaError_t launch_router(const RouterArgs &a, cudaStream_t stream, bool pdl);
cudaError_t launch_layer(const LayerArgs &a, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_pack(const PackArgs &a, cudaStream_t s);
cudaError_t launch_unpack(const UnpackArgs &a, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs &a, cudaStream_t s);
cudaError_t launch_residual_add(const __nv_bfloat16 *a, const __nv_bfloat16 *b, __nv_bfloat16 *out, int n,
                                cudaStream_t stream, bool pdl);

}  // namespace moe

// api.cu -- the extern "C" entry points of libnvfp4moe.so: argument checks,
// workspace handling and the launch sequence (declared in nvfp4moe.h).
#include <cstring>

#include "kernels.cuh"

using namespace moe;

namespace {

constexpr int ABI_VERSION = 1;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool disjoint(const void *a, const void *b, size_t n)
{
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa + n <= pb || pb + n <= pa;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

PerDevice g_sm_count;

int sm_count()
{
    const int v = per_device(g_sm_count, [](int dev) {
        int n = 0;
        return cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? n : -1;
    });
    return v > 0 ? v : 0;
}

moe_status check_bank(const moe_expert_bank *b, int expect_n, bool allow_empty)
{
    if (b == nullptr)
        return allow_empty ? MOE_OK : MOE_ERR_INVALID_ARG;
    if (allow_empty && b->n_experts == 0)
        return MOE_OK;
    if (b->n_experts != expect_n)
        return MOE_ERR_UNSUPPORTED;
    if (b->wtype != MOE_W_NVFP4 && b->wtype != MOE_W_BF16)
        return MOE_ERR_UNSUPPORTED;
    if (!b->w13 || !b->w2)
        return MOE_ERR_INVALID_ARG;
    if (b->wtype == MOE_W_NVFP4 && (!b->tscale13 || !b->tscale2))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(b->w13) || !aligned16(b->w2))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return ABI_VERSION; }

const char *moe_status_string(moe_status s)
{
    switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_FLAG: return "MOE_ERR_DEVICE_FLAG";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    }
    return "MOE_UNKNOWN_STATUS";
}

size_t moe_packed_bytes(int N, int K)
{
    if (N <= 0 || K <= 0 || N % 16 != 0 || K % 128 != 0)
        return 0;
    return (size_t)N * K / 2 + (size_t)N * K / 16;
}

static moe_status check_pack_args(const void *a, const void *b, const void *c, int N, int K, int kind,
                                  int count)
{
    if (!a || !b || !c || count < 1 || moe_packed_bytes(N, K) == 0)
        return MOE_ERR_INVALID_ARG;
    if (kind != MOE_PACK_PLAIN && kind != MOE_PACK_GATE_UP)
        return MOE_ERR_INVALID_ARG;
    if (kind == MOE_PACK_GATE_UP && N % 32 != 0)
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status moe_pack_nvfp4(const uint8_t *codes, const uint8_t *scales, int N, int K, int kind,
                          int count, void *packed, moe_stream_t stream)
{
    moe_status s = check_pack_args(codes, scales, packed, N, K, kind, count);
    if (s != MOE_OK)
        return s;
    PackArgs a{codes, scales, static_cast<uint8_t *>(packed), N, K, kind, count};
    return cuda_status(launch_pack(a, (cudaStream_t)stream));
}

moe_status moe_unpack_nvfp4(const void *packed, int N, int K, int kind, int count, uint8_t *codes,
                            uint8_t *scales, moe_stream_t stream)
{
    moe_status s = check_pack_args(packed, codes, scales, N, K, kind, count);
    if (s != MOE_OK)
        return s;
    UnpackArgs a{static_cast<const uint8_t *>(packed), codes, scales, N, K, kind, count};
    return cuda_status(launch_unpack(a, (cudaStream_t)stream));
}

moe_status moe_dequant_nvfp4(const void *packed, int N, int K, int kind, float tscale, float *out,
                             moe_stream_t stream)
{
    moe_status s = check_pack_args(packed, out, out, N, K, kind, 1);
    if (s != MOE_OK)
        return s;
    if (!aligned16(packed))
        return MOE_ERR_INVALID_ARG;
    DequantArgs a{static_cast<const uint8_t *>(packed), out, N, K, kind, tscale};
    return cuda_status(launch_dequant(a, (cudaStream_t)stream));
}

size_t moe_workspace_bytes(int T)
{
    if (T < 1 || T > MAX_TOKENS)
        return 0;
    if (T <= MAXT)
        return ws_layout().total;
    const size_t g = gws_layout(T).total;   // moe_route above MAXT tokens
    const size_t d = chunk_route_layout(T).total;   // the chunked decode path's copy-out
    return g > d ? g : d;
}

moe_status moe_workspace_init(void *workspace, size_t workspace_bytes, moe_stream_t stream)
{
    if (!workspace || !aligned16(workspace))
        return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < ws_layout().total)
        return MOE_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(workspace, 0, ws_layout().total, (cudaStream_t)stream));
}

moe_status moe_workspace_recover(void *workspace, size_t workspace_bytes, moe_stream_t stream)
{
    if (!workspace || !aligned16(workspace))
        return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < ws_layout().total)
        return MOE_ERR_WORKSPACE;
    return cuda_status(launch_rearm(static_cast<uint8_t *>(workspace), (cudaStream_t)stream, true));
}

moe_status moe_read_device_flag(void *workspace, moe_stream_t stream, uint32_t *flag_out)
{
    if (!workspace || !flag_out)
        return MOE_ERR_INVALID_ARG;
    uint32_t v = 0;
    uint8_t *flag = static_cast<uint8_t *>(workspace) + ws_layout().ctrl;
    cudaError_t e = cudaMemcpyAsync(&v, flag, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(flag, 0, sizeof v, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess)
        return MOE_ERR_CUDA;
    *flag_out = v;
    return v ? MOE_ERR_DEVICE_FLAG : MOE_OK;
}

moe_status moe_read_routing(const void *workspace, size_t workspace_bytes, int T, int32_t *idx, float *w,
                            float *logits, moe_stream_t stream)
{
    if (!workspace || !aligned16(workspace))
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > MAX_TOKENS)
        return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < moe_workspace_bytes(T))
        return MOE_ERR_WORKSPACE;
    if (!idx && !w && !logits)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const uint8_t *ws = static_cast<const uint8_t *>(workspace);
    size_t o_idx, o_w, o_lg, lg_pitch;
    if (T <= MAXT) {
        // the decode kernel keeps each logit in the low word of a 64-bit
        // (launch tag, logit) pair
        const WsLayout L = ws_layout();
        o_idx = L.topk_idx;
        o_w = L.topk_w;
        o_lg = L.tlogits;
        lg_pitch = 8;
    } else {
        // the decode kernel's chunks and the grouped path write their routing
        // at the same offsets
        const ChunkRouteLayout C = chunk_route_layout(T);
        o_idx = C.idx;
        o_w = C.w;
        o_lg = C.logits;
        lg_pitch = 4;
    }
    cudaError_t e = cudaSuccess;
    if (idx)
        e = cudaMemcpyAsync(idx, ws + o_idx, (size_t)T * TOPK * 4, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && w)
        e = cudaMemcpyAsync(w, ws + o_w, (size_t)T * TOPK * 4, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && logits) {
        if (T <= MAXT) {
            // token t's row: E of its LE (launch tag, logit) words
            for (int t = 0; t < T && e == cudaSuccess; ++t)
                e = cudaMemcpy2DAsync(logits + (size_t)t * E, 4, ws + o_lg + (size_t)t * LE * 8, lg_pitch, 4, E,
                                      cudaMemcpyDeviceToDevice, st);
        } else {
            e = cudaMemcpyAsync(logits, ws + o_lg, (size_t)T * E * 4, cudaMemcpyDeviceToDevice, st);
        }
    }
    return cuda_status(e);
}

static moe_status check_route_args(const void *x, const void *router_w, int T, void *workspace,
                                   size_t workspace_bytes)
{
    if (!x || !router_w || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(router_w) || !aligned16(workspace))
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > MAX_TOKENS)
        return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < moe_workspace_bytes(T))
        return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status moe_route(const void *x, const void *router_w, int T, int n_experts, int top_k,
                     int32_t *idx, float *w, float *logits, void *workspace, size_t workspace_bytes,
                     moe_stream_t stream)
{
    moe_status s = check_route_args(x, router_w, T, workspace, workspace_bytes);
    if (s != MOE_OK)
        return s;
    if (n_experts != E || top_k != TOPK)
        return MOE_ERR_UNSUPPORTED;
    if (!idx || !w)
        return MOE_ERR_INVALID_ARG;
    if (T > MAXT) {
        // router GEMM on the tensor cores, top-k per token, then the results
        // copied out of the workspace
        const int nsm = sm_count();
        if (nsm <= 0)
            return MOE_ERR_CUDA;
        cudaStream_t st = (cudaStream_t)stream;
        GroupedArgs ga{};
        ga.x = static_cast<const __nv_bfloat16 *>(x);
        ga.wr = static_cast<const __nv_bfloat16 *>(router_w);
        ga.T = T;
        ga.ws = static_cast<uint8_t *>(workspace);
        cudaError_t e = launch_grouped_route(ga, nsm, st);
        const GWsLayout L = gws_layout(T);
        const uint8_t *ws = static_cast<const uint8_t *>(workspace);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(idx, ws + L.idx, (size_t)T * TOPK * 4, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(w, ws + L.w, (size_t)T * TOPK * 4, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && logits)
            e = cudaMemcpyAsync(logits, ws + L.logits, (size_t)T * E * 4, cudaMemcpyDeviceToDevice, st);
        return cuda_status(e);
    }
    RouterArgs a{static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(router_w),
                 T, 0, static_cast<uint8_t *>(workspace), idx, w, logits};
    return cuda_status(launch_router(a, (cudaStream_t)stream, true));
}

// Host checks of one layer's weights (nothing is launched): E routed
// experts, and 0..MAX_EXT shared experts of either weight type.
static moe_status check_layer_weights(const void *router_w, const moe_expert_bank *routed,
                                      const moe_expert_bank *shared)
{
    if (!router_w || !aligned16(router_w))
        return MOE_ERR_INVALID_ARG;
    moe_status s;
    if ((s = check_bank(routed, E, false)) != MOE_OK)
        return s;
    const int ns = shared ? shared->n_experts : 0;
    if (ns < 0 || ns > MAX_EXT)
        return MOE_ERR_UNSUPPORTED;
    if (ns > 0 && (s = check_bank(shared, ns, false)) != MOE_OK)
        return s;
    return MOE_OK;
}

// The shared experts run ahead of the layer kernel on the dense GEMV (two
// launches) when the kernel cannot take them as its own slot 0: expert
// sinks, two of them, or another weight type than the routed bank.
static bool shared_ahead(const moe_expert_bank *routed, const moe_expert_bank *shared, bool sink)
{
    const int ns = shared ? shared->n_experts : 0;
    return ns > 0 && (sink || ns > MAX_SHARED || shared->wtype != routed->wtype);
}

// Gate/up (SiLU*up into the workspace's ext_h) and down (fp32 into ext_y) of
// the shared experts for T <= MAXT tokens of x.
static cudaError_t launch_shared_ahead(const void *x, const moe_expert_bank *shared, int T, uint8_t *ws,
                                       int nsm, cudaStream_t st)
{
    const WsLayout L = ws_layout();
    const bool bw = shared->wtype == MOE_W_BF16;
    GemvArgs g{};
    g.x = static_cast<const __nv_bfloat16 *>(x);
    g.x_mat_stride = 0;
    g.w = static_cast<const uint8_t *>(shared->w13);
    g.w_mat_stride = bw ? W13_BYTES_BF : W13_BYTES;
    g.ts_dev = bw ? nullptr : shared->tscale13;
    g.N = 2 * I;
    g.K = H;
    g.T = T;
    g.n_mat = shared->n_experts;
    g.kind = MOE_PACK_GATE_UP;
    g.bf16w = bw ? 1 : 0;
    g.epi = GEMV_SILU_H;
    g.y = ws + L.ext_h;
    g.y_mat_stride = (size_t)MAXT * I;
    g.flag = reinterpret_cast<uint32_t *>(ws + L.ctrl);
    cudaError_t e = launch_gemv(g, nsm, st);
    if (e != cudaSuccess)
        return e;
    g.x = reinterpret_cast<const __nv_bfloat16 *>(ws + L.ext_h);
    g.x_mat_stride = (size_t)MAXT * I;
    g.w = static_cast<const uint8_t *>(shared->w2);
    g.w_mat_stride = bw ? W2_BYTES_BF : W2_BYTES;
    g.ts_dev = bw ? nullptr : shared->tscale2;
    g.N = H;
    g.K = I;
    g.kind = MOE_PACK_PLAIN;
    g.epi = GEMV_OUT_F32;
    g.y = ws + L.ext_y;
    g.y_mat_stride = (size_t)MAXT * H;
    return launch_gemv(g, nsm, st);
}

// Fill the layer kernel's arguments (weights, workspace, output); the
// caller sets the input fields.
static void fill_layer_args(LayerArgs &la, const void *router_w, const moe_expert_bank *routed,
                            const moe_expert_bank *shared, void *out, int T, void *workspace, bool sink = false)
{
    const bool ahead = shared_ahead(routed, shared, sink);
    const int n_shared = (!ahead && shared && shared->n_experts > 0) ? 1 : 0;
    if (ahead) {
        la.n_ext = shared->n_experts;
        la.n_sink = sink ? shared->n_experts : 0;
        la.ext_y = reinterpret_cast<const float *>(static_cast<uint8_t *>(workspace) + ws_layout().ext_y);
    }
    la.wr = static_cast<const __nv_bfloat16 *>(router_w);
    la.T = T;
    la.r_w13 = static_cast<const uint8_t *>(routed->w13);
    la.r_w2 = static_cast<const uint8_t *>(routed->w2);
    la.r_ts13 = routed->tscale13;
    la.r_ts2 = routed->tscale2;
    if (n_shared) {
        la.s_w13 = static_cast<const uint8_t *>(shared->w13);
        la.s_w2 = static_cast<const uint8_t *>(shared->w2);
        la.s_ts13 = shared->tscale13;
        la.s_ts2 = shared->tscale2;
    }
    la.n_shared = n_shared;
    la.bf16w = routed->wtype == MOE_W_BF16 ? 1 : 0;
    la.ws = static_cast<uint8_t *>(workspace);
    la.out = static_cast<__nv_bfloat16 *>(out);
}

// The decode layer kernel's CTAs wait on one another, so its whole grid (one
// CTA per SM, at least 128 for the router phase) must be resident at once:
// the grid, or a status when that cannot hold (nothing is launched).
static moe_status layer_grid(int &grid)
{
    const int nsm = sm_count();
    if (nsm <= 0)
        return MOE_ERR_CUDA;
    grid = nsm >= 128 ? nsm : 128;
    const int per_sm = layer_resident_ctas_per_sm();
    if (per_sm < 0)
        return MOE_ERR_CUDA;
    if ((long)per_sm * nsm < grid)
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// Launch the decode layer kernel on every SM (after layer_grid's checks).
// With rearm set, the workspace's re-arm kernel runs first; with `shared`
// (shared experts run ahead), their two dense GEMV launches before that.
static moe_status launch_layer_on_all_sms(const LayerArgs &la, cudaStream_t st, bool rearm = false,
                                          const moe_expert_bank *shared = nullptr)
{
    int grid = 0;
    const moe_status s = layer_grid(grid);
    if (s != MOE_OK)
        return s;
    if (shared && launch_shared_ahead(la.x, shared, la.T, la.ws, sm_count(), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (rearm && launch_rearm(la.ws, st, true) != cudaSuccess)
        return MOE_ERR_CUDA;
    return cuda_status(launch_layer(la, grid, st, true));
}

}  // extern "C"

// MAXT < T <= chunk_max_t(weight type): the decode kernel on ceil(T / MAXT) balanced
// chunks (each token's output depends only on that token), every chunk's
// routing copied out for moe_read_routing.
static moe_status layer_forward_chunked(const void *x, const void *router_w, const moe_expert_bank *routed,
                                        const moe_expert_bank *shared, void *out, int T, void *workspace,
                                        cudaStream_t st)
{
    int grid = 0;
    const moe_status s = layer_grid(grid);
    if (s != MOE_OK)
        return s;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const ChunkRouteLayout C = chunk_route_layout(T);
    const int n = (T + MAXT - 1) / MAXT;
    for (int c = 0; c < n; ++c) {
        const int t0 = (int)((long)T * c / n), t1 = (int)((long)T * (c + 1) / n);
        LayerArgs la{};
        fill_layer_args(la, router_w, routed, shared, static_cast<__nv_bfloat16 *>(out) + (size_t)t0 * H,
                        t1 - t0, workspace);
        la.x = static_cast<const __nv_bfloat16 *>(x) + (size_t)t0 * H;
        la.r_idx = reinterpret_cast<int32_t *>(ws + C.idx);
        la.r_w = reinterpret_cast<float *>(ws + C.w);
        la.r_logits = reinterpret_cast<float *>(ws + C.logits);
        la.t0 = t0;
        const cudaError_t e = launch_layer(la, grid, st, true);
        if (e != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

// moe_layer_forward; with rearm (decode path only) the workspace's re-arm
// kernel runs ahead of the layer kernel.
moe_status moe::layer_forward(const void *x, const void *router_w, const moe_expert_bank *routed,
                              const moe_expert_bank *shared, void *out, int T, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream, bool rearm, bool sink)
{
    moe_status s = check_route_args(x, router_w, T, workspace, workspace_bytes);
    if (s != MOE_OK)
        return s;
    if (!out || !aligned16(out) || out == x)
        return MOE_ERR_INVALID_ARG;
    if ((s = check_layer_weights(router_w, routed, shared)) != MOE_OK)
        return s;
    const bool ahead = shared_ahead(routed, shared, sink);
    if (sink && !ahead)
        return MOE_ERR_INVALID_ARG;   // expert sinks need at least one shared expert
    if (T > MAXT && ahead)
        return MOE_ERR_UNSUPPORTED;   // the grouped path takes one shared expert of the routed type
    if (ahead && !disjoint(out, x, (size_t)T * H * 2))
        return MOE_ERR_INVALID_ARG;
    const int nsm = sm_count();
    if (nsm <= 0)
        return MOE_ERR_CUDA;
    if (T > MAXT && T <= chunk_max_t(routed->wtype)) {
        if (!disjoint(out, x, (size_t)T * H * 2))
            return MOE_ERR_INVALID_ARG;
        return layer_forward_chunked(x, router_w, routed, shared, out, T, workspace, (cudaStream_t)stream);
    }
    if (T > MAXT) {
        if (!disjoint(out, x, (size_t)T * H * 2))
            return MOE_ERR_INVALID_ARG;
        const bool has_shared = shared && shared->n_experts > 0;
        GroupedArgs ga{};
        ga.x = static_cast<const __nv_bfloat16 *>(x);
        ga.wr = static_cast<const __nv_bfloat16 *>(router_w);
        ga.T = T;
        ga.bf16w = routed->wtype == MOE_W_BF16 ? 1 : 0;
        ga.n_shared = has_shared ? 1 : 0;
        ga.r_w13 = static_cast<const uint8_t *>(routed->w13);
        ga.r_w2 = static_cast<const uint8_t *>(routed->w2);
        ga.r_ts13 = routed->tscale13;
        ga.r_ts2 = routed->tscale2;
        if (has_shared) {
            ga.s_w13 = static_cast<const uint8_t *>(shared->w13);
            ga.s_w2 = static_cast<const uint8_t *>(shared->w2);
            ga.s_ts13 = shared->tscale13;
            ga.s_ts2 = shared->tscale2;
        }
        ga.ws = static_cast<uint8_t *>(workspace);
        ga.out = static_cast<__nv_bfloat16 *>(out);
        return cuda_status(launch_grouped_layer(ga, nsm, (cudaStream_t)stream));
    }
    LayerArgs la{};
    fill_layer_args(la, router_w, routed, shared, out, T, workspace, sink);
    la.x = static_cast<const __nv_bfloat16 *>(x);
    return launch_layer_on_all_sms(la, (cudaStream_t)stream, rearm, ahead ? shared : nullptr);
}



extern "C" {

moe_status moe_layer_forward(const void *x, const void *router_w, const moe_expert_bank *routed,
                             const moe_expert_bank *shared, void *out, int T, void *workspace,
                             size_t workspace_bytes, moe_stream_t stream)
{
    return layer_forward(x, router_w, routed, shared, out, T, workspace, workspace_bytes, (cudaStream_t)stream,
                         false, false);
}

moe_status moe_layer_forward_sink(const void *x, const void *router_w, const moe_expert_bank *routed,
                                  const moe_expert_bank *shared, void *out, int T, void *workspace,
                                  size_t workspace_bytes, moe_stream_t stream)
{
    return layer_forward(x, router_w, routed, shared, out, T, workspace, workspace_bytes, (cudaStream_t)stream,
                         false, true);
}

moe_status moe_read_shared_weights(const void *workspace, size_t workspace_bytes, int T, int n_shared, float *sw,
                                   moe_stream_t stream)
{
    if (!workspace || !aligned16(workspace) || !sw)
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > MAXT || n_shared < 1 || n_shared > MAX_EXT)
        return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < moe_workspace_bytes(T))
        return MOE_ERR_WORKSPACE;
    const uint8_t *ws = static_cast<const uint8_t *>(workspace);
    return cuda_status(cudaMemcpy2DAsync(sw, (size_t)n_shared * 4, ws + ws_layout().sinkw, MAX_EXT * 4,
                                         (size_t)n_shared * 4, (size_t)T, cudaMemcpyDeviceToDevice,
                                         (cudaStream_t)stream));
}

moe_status moe_layer_forward_prenorm(const void *resid, const void *delta, void *resid_out, void *xn_out,
                                     float eps, const void *router_w, const moe_expert_bank *routed,
                                     const moe_expert_bank *shared, void *out, int T, void *workspace,
                                     size_t workspace_bytes, moe_stream_t stream)
{
    moe_status s = check_route_args(resid, router_w, T, workspace, workspace_bytes);
    if (s != MOE_OK)
        return s;
    if (T > MAXT)
        return MOE_ERR_UNSUPPORTED;
    const size_t nb = (size_t)T * H * 2;
    if (!out || !aligned16(out) || !disjoint(out, resid, nb))
        return MOE_ERR_INVALID_ARG;
    if (delta && (!aligned16(delta) || !disjoint(out, delta, nb)))
        return MOE_ERR_INVALID_ARG;
    for (const void *p : {resid_out, xn_out}) {
        if (!p)
            continue;
        if (!aligned16(p) || !disjoint(p, out, nb) || !disjoint(p, resid, nb) ||
            (delta && !disjoint(p, delta, nb)))
            return MOE_ERR_INVALID_ARG;
    }
    if (resid_out && xn_out && !disjoint(resid_out, xn_out, nb))
        return MOE_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !(eps < 1.0f))
        return MOE_ERR_INVALID_ARG;
    if ((s = check_layer_weights(router_w, routed, shared)) != MOE_OK)
        return s;
    if (shared_ahead(routed, shared, false))
        return MOE_ERR_UNSUPPORTED;   // the pre-norm input exists only inside the layer kernel
    if (sm_count() <= 0)
        return MOE_ERR_CUDA;
    LayerArgs la{};
    fill_layer_args(la, router_w, routed, shared, out, T, workspace);
    la.x = static_cast<const __nv_bfloat16 *>(resid);
    la.prenorm = 1;
    la.delta = static_cast<const __nv_bfloat16 *>(delta);
    la.resid_out = static_cast<__nv_bfloat16 *>(resid_out);
    la.xn_out = static_cast<__nv_bfloat16 *>(xn_out);
    la.eps = eps;
    return launch_layer_on_all_sms(la, (cudaStream_t)stream);
}

// Stack workspace: the layer workspace, then the residual ping-pong buffers
// R0, R1 and the layer-output buffers D0, D1 (bf16 [T][H] each).
static size_t stack_buf_bytes(int T) { return align256((size_t)T * H * 2); }

size_t moe_stack_workspace_bytes(int T)
{
    if (T < 1 || T > MAXT)
        return 0;
    return ws_layout().total + 4 * stack_buf_bytes(T);
}

moe_status moe_stack_forward(void *x, const moe_layer_weights *layers, int n_layers, int T, float eps,
                             void *workspace, size_t workspace_bytes, moe_stream_t stream)
{
    if (!x || !aligned16(x) || !layers || n_layers < 1 || !workspace || !aligned16(workspace))
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > MAXT)
        return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < moe_stack_workspace_bytes(T))
        return MOE_ERR_WORKSPACE;
    if (!(eps >= 0.0f) || !(eps < 1.0f))
        return MOE_ERR_INVALID_ARG;
    moe_status s;
    for (int l = 0; l < n_layers; ++l) {
        s = check_layer_weights(layers[l].router_w, &layers[l].routed, &layers[l].shared);
        if (s == MOE_OK && shared_ahead(&layers[l].routed, &layers[l].shared, false))
            s = MOE_ERR_UNSUPPORTED;   // a layer's shared expert must fit the layer kernel's slot 0
        if (s != MOE_OK)
            return s;
    }
    if (sm_count() <= 0)
        return MOE_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(workspace) + ws_layout().total;
    __nv_bfloat16 *R[2], *D[2];
    for (int i = 0; i < 2; ++i) {
        R[i] = reinterpret_cast<__nv_bfloat16 *>(base + (size_t)i * stack_buf_bytes(T));
        D[i] = reinterpret_cast<__nv_bfloat16 *>(base + (size_t)(2 + i) * stack_buf_bytes(T));
    }
    __nv_bfloat16 *x0 = static_cast<__nv_bfloat16 *>(x);
    // layer l reads the residual x_l and the previous output D[(l-1)&1]
    // (none for l = 0), writes x_l's successor's residual part R[l&1] and
    // its own output D[l&1]
    for (int l = 0; l < n_layers; ++l) {
        LayerArgs la{};
        const moe_layer_weights &w = layers[l];
        const moe_expert_bank *sh = w.shared.n_experts > 0 ? &w.shared : nullptr;
        fill_layer_args(la, w.router_w, &w.routed, sh, D[l & 1], T, workspace);
        la.prenorm = 1;
        la.eps = eps;
        if (l == 0) {
            la.x = x0;
        } else {
            la.x = (l == 1) ? x0 : R[(l - 1) & 1];
            la.delta = D[(l - 1) & 1];
            la.resid_out = R[l & 1];
        }
        const moe_status e = launch_layer_on_all_sms(la, st);
        if (e != MOE_OK)
            return e;
    }
    // x_L = x_{L-1} + D[(L-1)&1]
    const __nv_bfloat16 *last = (n_layers == 1) ? x0 : R[(n_layers - 1) & 1];
    return cuda_status(launch_residual_add(last, D[(n_layers - 1) & 1], x0, T * H, st, true));
}

}  // extern "C"

extern "C" {

moe_status moe_dense_gemv_nvfp4(const void *x, const void *w_packed, float tscale, int N, int K, int T, void *y,
                                void *workspace, size_t workspace_bytes, moe_stream_t stream)
{
    if (!x || !w_packed || !y || !workspace || !aligned16(x) || !aligned16(w_packed) || !aligned16(y) ||
        !aligned16(workspace))
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > MAXT || N < 16 || N % 16 != 0 || K < 256 || K % 256 != 0 || K > GEMV_MAX_K)
        return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < 256)
        return MOE_ERR_WORKSPACE;
    const uintptr_t px = (uintptr_t)x, py = (uintptr_t)y;
    if (px < py + (size_t)T * N * 2 && py < px + (size_t)T * K * 2)
        return MOE_ERR_INVALID_ARG;
    const int nsm = sm_count();
    if (nsm <= 0)
        return MOE_ERR_CUDA;
    GemvArgs ga{};
    ga.x = static_cast<const __nv_bfloat16 *>(x);
    ga.w = static_cast<const uint8_t *>(w_packed);
    ga.ts_host = tscale;
    ga.N = N;
    ga.K = K;
    ga.T = T;
    ga.n_mat = 1;
    ga.kind = MOE_PACK_PLAIN;
    ga.bf16w = 0;
    ga.epi = GEMV_OUT_BF16;
    ga.y = y;
    ga.flag = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + ws_layout().ctrl);
    return cuda_status(launch_gemv(ga, nsm, (cudaStream_t)stream));
}

}  // extern "C"

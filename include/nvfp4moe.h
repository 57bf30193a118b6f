/*
 * nvfp4moe.h -- C ABI of libnvfp4moe.so, the GB300 (sm_103a) small-batch
 * weight-only NVFP4 (W4A16) mixture-of-experts layer.
 *
 * The operation (sources are web pages, cited by title and section):
 *
 *  [FLINT]  "vLLM adds day-0 support for Recursive's Flint, hitting about 485
 *           tokens/s on one GB200", section "A 40B MoE that activates 2.5B
 *           parameters": hidden size 2048, 256 routed experts, sigmoid top-6
 *           routing plus one shared expert; the NVFP4 checkpoint is repacked
 *           losslessly at load time and runs weight-only (W4A16) with BF16
 *           activations.  Section "From 1,096 kernels to 346": router and
 *           expert GEMVs read only the selected experts' weights; routing and
 *           the expert combine are fused into the neighbouring GEMVs; each
 *           kernel uses programmatic dependent launch.
 *  [MOET]   "Frontier MoE on consumer Blackwell (SM120)", section
 *           "GLM-5.2 (753B) - the headline model": NVFP4 = e2m1 code x e4m3
 *           scale per block of 16 x per-tensor fp32 scale.
 *  [INKLING] "TML Inkling on vLLM", section "MoE": two shared experts that
 *           act as expert sinks; only the routed experts are NVFP4.
 *
 * For T tokens x[T][H] (bf16) the layer computes
 *     logit[t][e] = sum_k x[t][k] * router_w[e][k]
 *     sel[t]      = the top_k experts by logit (lower index wins a tie)
 *     w[t][i]     = sigmoid(logit[t][sel_i]) / sum_j sigmoid(logit[t][sel_j])
 *     FFN_e(v)    = W2_e ( silu(W1_e v) * (W3_e v) )      (W13 = [W1; W3])
 *     out[t]      = sum_i w[t][i] * FFN_{sel_i}(x[t]) + FFN_shared(x[t])
 * with NVFP4 weights dequantised exactly (e2m1 * e4m3 * tensor scale), fp32
 * accumulation, the SiLU*up activation rounded to bf16 (the activations are
 * BF16), and out rounded once to bf16.
 *
 * Shapes this build supports: H = 2048, I = 512 (W13 is [2I][H], W2 is
 * [H][I]), E = 256 routed experts, top_k = 6, 0 or 1 shared expert (up to
 * 2, of either weight type, for 1..MOE_MAX_DECODE_T tokens), and
 * 1 <= T <= MOE_MAX_TOKENS tokens per call (the decode kernel up to
 * MOE_MAX_DECODE_T tokens, on chunks of at most MOE_MAX_DECODE_T tokens up to
 * MOE_MAX_CHUNKED_T (BF16 weights: MOE_MAX_CHUNKED_T_BF16), the grouped
 * tensor-core path above; the stack and
 * pre-norm calls take 1..MOE_MAX_DECODE_T).
 *
 * Conventions for every entry point:
 *  - All data pointers are DEVICE pointers (cudaMalloc / torch memory) on the
 *    current device, 16-byte aligned, unless a comment says "host".
 *  - The caller owns every buffer; the library allocates and frees nothing.
 *  - Calls enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and return without synchronising, except where stated.
 *  - Argument errors are detected on the host before anything is enqueued
 *    and return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED; launch failures
 *    return MOE_ERR_CUDA.  Conditions found on the device (a non-finite
 *    router logit, an expired bounded wait) set bits of a flag word in the
 *    workspace, read back by moe_read_device_flag.  Kernels never trap.
 *  - Apart from the fixed scratch of moe_layer_forward_static, the library
 *    keeps no mutable global state, so calls with different workspaces are
 *    independent.  But the decode layer kernel (1..MOE_MAX_DECODE_T tokens:
 *    moe_layer_forward, moe_layer_forward_prenorm, moe_stack_forward) needs
 *    one CTA on every SM at the same time, so two of them must not overlap
 *    on one GPU, nor run beside other kernels that hold SMs: order them on
 *    one stream (or with events).  Before each launch the library checks
 *    that one CTA of the kernel fits on an SM (its shared memory and
 *    registers) and that the device has at least 128 SMs, and returns
 *    MOE_ERR_UNSUPPORTED otherwise; if SMs are nonetheless held by other
 *    work (another process, a partitioned device) the bounded waits expire
 *    and set MOE_FLAG_WAIT_TIMEOUT.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* a cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size */
    MOE_ERR_UNSUPPORTED = 2, /* shape or mode this build does not implement */
    MOE_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE_FLAG = 4, /* moe_read_device_flag found a device-side error */
    MOE_ERR_WORKSPACE = 5    /* workspace too small */
} moe_status;

/* Weight storage of an expert bank. */
enum { MOE_W_NVFP4 = 0, MOE_W_BF16 = 1 };

/* Row order of a packed NVFP4 matrix.  GATE_UP interleaves the gate rows
 * [0, N/2) and up rows [N/2, N) of a W13 matrix so that one 16-row band
 * holds gate rows 8b..8b+7 and the matching up rows. */
enum { MOE_PACK_PLAIN = 0, MOE_PACK_GATE_UP = 1 };

/* Device-side error bits reported by moe_read_device_flag. */
enum {
    MOE_FLAG_NONFINITE_LOGIT = 1, /* a router logit was NaN/Inf; routing used index order */
    MOE_FLAG_WAIT_TIMEOUT = 2,    /* a bounded wait on a barrier expired; output invalid */
    MOE_FLAG_BAD_INDEX = 4        /* an expert index out of range was seen; skipped */
};

#define MOE_HIDDEN 2048
#define MOE_INTER 512
#define MOE_EXPERTS 256
#define MOE_TOPK 6
#define MOE_MAX_DECODE_T 8
#define MOE_MAX_CHUNKED_T 88        /* largest T of moe_layer_forward's chunked decode path (NVFP4 weights) */
#define MOE_MAX_CHUNKED_T_BF16 56   /* the same for BF16 weights */
#define MOE_MAX_TOKENS 65536   /* largest T of moe_route / moe_layer_forward */

/*
 * A bank of experts with identical shapes, stored back to back.
 *  wtype == MOE_W_NVFP4: w13 holds n_experts packed W13 matrices (gate/up,
 *     [2I][H], packed with MOE_PACK_GATE_UP), each moe_packed_bytes(2I, H)
 *     bytes; w2 holds n_experts packed W2 matrices ([H][I], MOE_PACK_PLAIN),
 *     each moe_packed_bytes(H, I) bytes; tscale13/tscale2 are device float
 *     arrays [n_experts] of per-tensor scales.
 *  wtype == MOE_W_BF16: w13 is bf16 [n_experts][2I][H] row-major, w2 is bf16
 *     [n_experts][H][I]; tscale13/tscale2 are ignored (may be NULL).
 * The struct itself is host memory; the pointers in it are device pointers.
 */
typedef struct {
    int32_t wtype;
    int32_t n_experts;
    const void *w13;
    const void *w2;
    const float *tscale13;
    const float *tscale2;
} moe_expert_bank;

/* ABI version of this header (bumped on any incompatible change). */
int moe_abi_version(void);

/* Human-readable name of a status (static storage; never NULL). */
const char *moe_status_string(moe_status s);

/* ----------------------------------------------------------------------- */
/* Packing (load time).  [FLINT, "A 40B MoE ...": the NVFP4 blocks are     */
/* repacked losslessly at load time.]                                      */
/* ----------------------------------------------------------------------- */

/* Bytes of one packed NVFP4 matrix [N][K]: N*K/2 code bytes + N*K/16 scale
 * bytes (the same as the canonical form; packing permutes bytes and nibbles
 * only).  Returns 0 when N is not a multiple of 16 or K not a multiple of
 * 128. */
size_t moe_packed_bytes(int N, int K);

/*
 * Pack `count` canonical NVFP4 matrices [N][K] into the kernel layout.
 *  codes:  device u8 [count][N][K/2]; byte (n, j) holds element (n, 2j) in
 *          its low nibble and (n, 2j+1) in its high nibble (e2m1 codes).
 *  scales: device u8 [count][N][K/16]; e4m3 (E4M3FN) scale of elements
 *          (n, 16b .. 16b+15) at (n, b).
 *  kind:   MOE_PACK_PLAIN or MOE_PACK_GATE_UP (needs N % 32 == 0).
 *  packed: device, count * moe_packed_bytes(N, K) bytes, 16-byte aligned.
 * The result is a pure permutation of the input nibbles and scale bytes.
 * Errors: MOE_ERR_INVALID_ARG for null pointers, count < 1 or unsupported
 * N/K; nothing is enqueued then.
 */
moe_status moe_pack_nvfp4(const uint8_t *codes, const uint8_t *scales, int N, int K, int kind,
                          int count, void *packed, moe_stream_t stream);

/* Exact inverse of moe_pack_nvfp4 (same arguments, opposite direction). */
moe_status moe_unpack_nvfp4(const void *packed, int N, int K, int kind, int count,
                            uint8_t *codes, uint8_t *scales, moe_stream_t stream);

/*
 * Dequantise one packed NVFP4 matrix to fp32 in canonical row order:
 * out[n][k] = fp32(e2m1 * e4m3 * tscale) (the e2m1*e4m3 product is exact;
 * one rounding when tscale is applied).  out: device float [N][K].
 * Used to check the packed layout and the in-register decode.
 * [MOET, "GLM-5.2": e2m1 x e4m3 block-16 x per-tensor scale_2]
 */
moe_status moe_dequant_nvfp4(const void *packed, int N, int K, int kind, float tscale,
                             float *out, moe_stream_t stream);

/* ----------------------------------------------------------------------- */
/* Workspace.                                                              */
/* ----------------------------------------------------------------------- */

/* Workspace bytes for moe_route / moe_layer_forward with T tokens (0 unless
 * 1 <= T <= MOE_MAX_TOKENS).  The workspace holds routing results, the
 * SiLU*up activations, combine partials, arrival counters and the device
 * flag; above MOE_MAX_DECODE_T tokens also the routing of every token
 * (either path), the grouped path's expert lists, the tokens' rows sorted
 * by expert and the per-(token, choice) down outputs (about 93 KB per token;
 * the grouped router of moe_route uses them at any T above
 * MOE_MAX_DECODE_T). */
size_t moe_workspace_bytes(int T);

/* Zero a workspace (enqueued memset).  Required once before the first use of
 * a workspace; every call leaves its counters re-armed for the next call (the
 * layer kernel's launch tag, which starts at zero, advances by one per call).
 * After a call that reported MOE_FLAG_WAIT_TIMEOUT, zero the workspace again
 * or call moe_workspace_recover before its next use. */
moe_status moe_workspace_init(void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Re-arm a decode workspace after a wait timeout, without losing its flag
 * word: one small kernel, enqueued on `stream` (it waits for the preceding
 * kernel), that does nothing unless the flag word holds
 * MOE_FLAG_WAIT_TIMEOUT; then it clears the arrival counters a timed-out
 * call may have left behind and advances the launch tag, so that the next
 * layer call ignores router logits tagged by the failed one.  The flag bits
 * stay until moe_read_device_flag reads them.  Allocates nothing.
 * Errors: MOE_ERR_INVALID_ARG (null or misaligned workspace),
 * MOE_ERR_WORKSPACE (smaller than moe_workspace_bytes(1)), MOE_ERR_CUDA.
 */
moe_status moe_workspace_recover(void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Read and clear the device flag word of a workspace.  SYNCHRONISES the
 * stream.  *flag_out (host) receives the MOE_FLAG_* bits.  Returns MOE_OK when
 * no bit was set, MOE_ERR_DEVICE_FLAG when one was, MOE_ERR_CUDA on a CUDA
 * error.
 */
moe_status moe_read_device_flag(void *workspace, moe_stream_t stream, uint32_t *flag_out);

/* ----------------------------------------------------------------------- */
/* Routing.  [FLINT, "A 40B MoE ...": sigmoid top-6 routing]               */
/* ----------------------------------------------------------------------- */

/*
 * Router GEMV + sigmoid + top-k + renormalisation for T tokens.
 *  x:        device bf16 [T][H];  router_w: device bf16 [E][H].
 *  idx:      device int32 [T][top_k] (selection order: best first).
 *  w:        device float [T][top_k], renormalised to sum to 1 per token.
 *  logits:   device float [T][E] fp32 logits, or NULL.
 * T <= MOE_MAX_DECODE_T: logits are fp32 sums of exact bf16*bf16 products
 * (fixed summation tree of depth <= 24).  Larger T: a tcgen05 GEMM computes
 * them (bf16 operands, fp32 accumulation in tensor memory, 128 MMAs of
 * K = 16 in sequence).  The selection is taken on the fp32 logits, a tie
 * going to the lower index.  A non-finite logit sets MOE_FLAG_NONFINITE_LOGIT.
 * Errors: MOE_ERR_UNSUPPORTED unless H, E, top_k match this build and
 * 1 <= T <= MOE_MAX_TOKENS; MOE_ERR_WORKSPACE if workspace_bytes is below
 * moe_workspace_bytes(T).
 */
moe_status moe_route(const void *x, const void *router_w, int T, int n_experts, int top_k,
                     int32_t *idx, float *w, float *logits, void *workspace,
                     size_t workspace_bytes, moe_stream_t stream);

/*
 * Copy out the routing that the last layer call on `workspace` used: the
 * most recent moe_layer_forward, moe_layer_forward_prenorm or (its last
 * layer) moe_stack_forward with the same T.  The layer kernels route
 * internally; this exposes their own selection so that it can be checked
 * against a reference.  [FLINT, "A 40B MoE ...": sigmoid top-6 routing]
 *  idx:    device int32 [T][top_k], selection order (best first), or NULL.
 *  w:      device float [T][top_k], renormalised weights, or NULL.
 *  logits: device float [T][E] fp32 router logits, or NULL.
 *  Where the decode kernel ran (T up to MOE_MAX_CHUNKED_T, or
 *  MOE_MAX_CHUNKED_T_BF16 for BF16 weights): logits are fp32 sums of exact
 *  bf16*bf16 products along a fixed tree of depth 15.  Larger T: the
 *  grouped path's router GEMM (see moe_route).
 * At least one output must be non-NULL.  Enqueued device-to-device copies;
 * the result is undefined if no layer call with this T preceded it.
 * Errors: MOE_ERR_INVALID_ARG (null or misaligned workspace, all outputs
 * NULL), MOE_ERR_UNSUPPORTED (T outside 1..MOE_MAX_TOKENS), MOE_ERR_WORKSPACE
 * (workspace_bytes below moe_workspace_bytes(T)), MOE_ERR_CUDA.
 */
moe_status moe_read_routing(const void *workspace, size_t workspace_bytes, int T, int32_t *idx, float *w,
                            float *logits, moe_stream_t stream);

/* ----------------------------------------------------------------------- */
/* The layer.  [FLINT, "From 1,096 kernels to 346": router and expert GEMVs */
/* that read only the selected experts' weights, routing and the combine   */
/* fused into the neighbouring kernels, chained by programmatic dependent  */
/* launch.]                                                                */
/* ----------------------------------------------------------------------- */

/*
 * out = MoE(x) for 1 <= T <= MOE_MAX_TOKENS tokens (see the top of this
 * header).
 * From MOE_MAX_DECODE_T + 1 to MOE_MAX_CHUNKED_T tokens (NVFP4 weights;
 * MOE_MAX_CHUNKED_T_BF16 for BF16) the decode kernel below runs on
 * ceil(T / MOE_MAX_DECODE_T) balanced chunks of consecutive tokens, one
 * launch per chunk (each token's output depends only on that token; a chunk
 * reads the weights of its own selected experts).  On GB300 this beats the
 * grouped path up to those sizes (measured, NVFP4: the grouped path 122 us
 * at 9 tokens, 341 at 88, 346 at 96; the decode kernel about 30 us per 8
 * tokens).
 * Above those sizes the grouped path runs instead [FLINT,
 * "From 1,096 kernels to 346": the same packed layout serves the grouped
 * GEMMs of large batches]: a router GEMM, top-k, per-expert token lists in
 * token order, then tcgen05 tensor-core GEMMs per expert (weights dequantised
 * to f16 in shared memory; each token row of x and of h scaled by a power of
 * two into f16, exactly for every element within 2^28 of the row's largest),
 * h rounded to bf16 as in the decode path, and a combine that adds the six
 * weighted expert outputs in choice order and the shared expert's (fp32,
 * rounded once to bf16; deterministic).  With BF16 weights the grouped GEMMs
 * use the bf16 values directly.
 * Up to MOE_MAX_DECODE_T tokens: one persistent kernel (one CTA per SM, launched with
 * programmatic dependent launch so that its weight prefetch overlaps the
 * preceding kernel) runs the router GEMV and the top-k of every token, builds
 * the union of the selected experts with per-token weights, streams each
 * selected expert's W13 once for all tokens (SiLU*up fused into the epilogue),
 * then its W2 (routing weight fused), and adds the per-expert partials of
 * every output row in a fixed order (deterministic, bit-identical between
 * calls).  The routing results stay readable in the workspace.
 *  x:        device bf16 [T][H]; must not alias out.
 *  router_w: device bf16 [E][H].
 *  routed:   host struct describing E = 256 routed experts.
 *  shared:   host struct with n_experts 0, 1 or 2 (NULL = no shared expert);
 *            each shared expert is added with weight 1.
 *  out:      device bf16 [T][H].
 *  workspace: device, >= moe_workspace_bytes(T), initialised once with
 *            moe_workspace_init; one workspace per concurrently running call.
 * Weight types: both banks NVFP4 (W4A16), or both BF16 (the W16A16 variant
 * [FLINT, "From 1,096 kernels to 346": BF16 decode]: same routing, same
 * combine, bf16 weights read row-major).  Up to MOE_MAX_DECODE_T tokens the
 * shared bank may also hold 2 experts, or be of the other type than the
 * routed one (TML Inkling's NVFP4 checkpoint: BF16 shared experts beside
 * NVFP4 routed ones [INKLING, "MoE"]): those shared experts then run ahead of
 * the layer kernel as two dense GEMV launches (gate/up with SiLU*up, then
 * down, see moe_dense_gemv_nvfp4; h rounded to bf16, their fp32 outputs kept
 * in the workspace), and the layer kernel adds them in its combine, after
 * the routed experts, before the one rounding to bf16.  Above
 * MOE_MAX_DECODE_T tokens such a shared bank gives MOE_ERR_UNSUPPORTED.
 * Activations must be finite; with NVFP4 weights also max|x[t]| < 2^114 per
 * token: each token is scaled by a power of two into f16 for the tensor cores
 * (see csrc/common.cuh).  With BF16 weights the activations and h enter the
 * tensor cores as bf16 unchanged.
 * Every SM must be able to host one CTA at the same time (the kernel's CTAs
 * wait on each other's counters, with bounded waits that set
 * MOE_FLAG_WAIT_TIMEOUT if that ever fails).
 */
moe_status moe_layer_forward(const void *x, const void *router_w, const moe_expert_bank *routed,
                             const moe_expert_bank *shared, void *out, int T, void *workspace,
                             size_t workspace_bytes, moe_stream_t stream);

/* ----------------------------------------------------------------------- */
/* Dense small-batch GEMV.  [FLINT, "From 1,096 kernels to 346": the       */
/* small-batch dense GEMV (dense MLP layers, projections) runs on the same */
/* packed NVFP4 weights as the large-batch kernel.]                        */
/* ----------------------------------------------------------------------- */

/*
 * y[t][n] = bf16( tscale * sum_k W[n][k] x[t][k] ) for 1 <= T <= MOE_MAX_DECODE_T
 * tokens, W[n][k] = e2m1 * e4m3 (exact) of one packed NVFP4 matrix.
 *  x:        device bf16 [T][K], row-major; must not overlap y.
 *  w_packed: device, moe_packed_bytes(N, K) bytes from moe_pack_nvfp4 with
 *            kind MOE_PACK_PLAIN (row n of y is row n of W).
 *  tscale:   the matrix's per-tensor fp32 scale (host value).
 *  y:        device bf16 [T][N], row-major.
 *  workspace: device, >= 256 bytes, zeroed once (moe_workspace_init on a
 *            layer workspace, or a plain memset); only its device flag word
 *            (read by moe_read_device_flag) is used, so a layer workspace
 *            may be shared with this call when the two do not overlap.
 * Arithmetic: as the decode layer's gate/up GEMV -- each token scaled by a
 * power of two into f16 (exact for every element within 2^28 of the
 * token's largest), e2m1 x f16 products exact in fp32 mma accumulation,
 * the e4m3 block scale applied to each 16-column partial, the K partials
 * added in a fixed order (deterministic, bit-identical between calls), the
 * tensor scale and the power of two applied at the end, one rounding to
 * bf16.  Activations must be finite with max|x[t]| < 2^114.
 * One kernel, one CTA per SM (each CTA streams a contiguous range of 16-row
 * bands), launched with programmatic dependent launch: it starts reading W
 * while the preceding kernel finishes and waits for it only before reading x.
 * So W must not be written by a kernel that may still be running when this
 * call starts (one that signals programmatic completion early); the packing
 * kernel of moe_pack_nvfp4 never does.
 * Errors: MOE_ERR_INVALID_ARG (null or misaligned pointer, x and y overlap),
 * MOE_ERR_UNSUPPORTED (T outside 1..MOE_MAX_DECODE_T, N not a positive
 * multiple of 16, K not a multiple of 256 in 256..8192), MOE_ERR_WORKSPACE
 * (workspace_bytes < 256), MOE_ERR_CUDA.
 */
moe_status moe_dense_gemv_nvfp4(const void *x, const void *w_packed, float tscale, int N, int K, int T,
                                void *y, void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * The layer with expert-sink routing [INKLING, "MoE": 256 routed experts
 * (top-6) plus 2 shared experts that take part in the routing-score
 * computation, absorbing probability mass, but are never candidates for the
 * top-6].  This library reads it as: router_w has E + S rows, the last S
 * being the S shared experts'; every row's score is sigmoid(logit); the
 * top_k are chosen among the E routed experts as in moe_layer_forward; with
 * D = (sum of the selected scores) + (sum of the S shared scores), selected
 * expert e gets the weight s_e / D and shared expert j the weight
 * s_{E+j} / D:
 *     out[t] = sum_i w[t][i] FFN_{sel_i}(x[t]) + sum_j sw[t][j] FFN_shared_j(x[t])
 *  router_w: device bf16 [E + S][H].
 *  shared:   host struct with n_experts S = 1 or 2, NVFP4 or BF16 (the routed
 *            bank may be either type): run ahead of the layer kernel as in
 *            moe_layer_forward.
 *  The logits (all E + S per token, fp32 as in moe_layer_forward), the
 *  selection and the denominator are computed in the layer kernel; the
 *  fp32 denominator adds the selected scores in selection order, then the
 *  shared ones in order.  moe_read_routing returns the routed part
 *  (selection, weights, the E routed logits); moe_read_shared_weights the
 *  shared experts' weights.
 *  The other arguments are those of moe_layer_forward.
 * Errors: as moe_layer_forward; MOE_ERR_INVALID_ARG without a shared expert;
 * MOE_ERR_UNSUPPORTED for T > MOE_MAX_DECODE_T.
 */
moe_status moe_layer_forward_sink(const void *x, const void *router_w, const moe_expert_bank *routed,
                                  const moe_expert_bank *shared, void *out, int T, void *workspace,
                                  size_t workspace_bytes, moe_stream_t stream);

/*
 * Copy out the weights of the shared experts that the last decode-path call
 * on `workspace` with this T used: sw (device float [T][n_shared]) receives
 * s_{E+j} / D per token for moe_layer_forward_sink, 1 for shared experts run
 * ahead by moe_layer_forward.  Undefined unless such a call with S >= n_shared
 * shared experts run ahead preceded it.  Enqueued device-to-device copy.
 * Errors: MOE_ERR_INVALID_ARG (null or misaligned workspace, null sw),
 * MOE_ERR_UNSUPPORTED (T outside 1..MOE_MAX_DECODE_T, n_shared outside 1..2),
 * MOE_ERR_WORKSPACE (workspace_bytes below moe_workspace_bytes(T)), MOE_ERR_CUDA.
 */
moe_status moe_read_shared_weights(const void *workspace, size_t workspace_bytes, int T, int n_shared, float *sw,
                                   moe_stream_t stream);

/* ----------------------------------------------------------------------- */
/* Decoder stacks.  [FLINT, "A 40B MoE that activates 2.5B parameters": a  */
/* 47-layer pre-norm decoder.]  The pages give only "pre-norm"; this       */
/* library reads a layer of the stack as x <- x + MoE(RMSNorm(x)) with a   */
/* unit-weight RMSNorm, the residual stream kept in bf16.                   */
/* ----------------------------------------------------------------------- */

/* The weights of one layer of a stack (host struct; device pointers).  A
 * shared bank with n_experts == 0 means no shared expert. */
typedef struct {
    const void *router_w;          /* device bf16 [E][H] */
    moe_expert_bank routed;
    moe_expert_bank shared;
} moe_layer_weights;

/*
 * One pre-norm layer: v = bf16(resid + delta) (v = resid when delta is
 * NULL), xn = bf16(v / sqrt(mean_k(v_k^2) + eps)) per token (fp32 sum of
 * squares in a fixed order, IEEE sqrt and divide), out = MoE(xn) exactly as
 * moe_layer_forward computes it from xn.  The add and the norm run inside
 * the layer kernel (every CTA forms xn from resid and delta in shared
 * memory); no extra launch.
 *  resid, delta: device bf16 [T][H] (delta may be NULL).
 *  resid_out:    device bf16 [T][H] receiving v, or NULL.
 *  xn_out:       device bf16 [T][H] receiving xn, or NULL.
 *  eps:          0 <= eps < 1.
 *  The other arguments are those of moe_layer_forward; the shared bank must
 *  be one expert of the routed bank's type (MOE_ERR_UNSUPPORTED otherwise).
 *  out must not overlap resid, delta, resid_out or xn_out; resid_out and
 *  xn_out must not overlap any other buffer (MOE_ERR_INVALID_ARG).
 */
moe_status moe_layer_forward_prenorm(const void *resid, const void *delta, void *resid_out, void *xn_out,
                                     float eps, const void *router_w, const moe_expert_bank *routed,
                                     const moe_expert_bank *shared, void *out, int T, void *workspace,
                                     size_t workspace_bytes, moe_stream_t stream);

/* Workspace bytes of moe_stack_forward with T tokens (0 if unsupported):
 * a layer workspace plus four bf16 [T][H] buffers. */
size_t moe_stack_workspace_bytes(int T);

/*
 * x <- layer_{n-1}(... layer_0(x)) with layer_l(x) = x + MoE_l(RMSNorm(x)),
 * each layer as moe_layer_forward_prenorm; n_layers + 1 launches chained by
 * programmatic dependent launch (each layer kernel also adds the previous
 * layer's output to the residual stream; a last small kernel adds the final
 * layer's output into x).
 *  x:         device bf16 [T][H], input x_0, overwritten by x_n.
 *  layers:    host array [n_layers] (n_layers >= 1); every layer is checked
 *             before anything is launched.
 *  workspace: device, >= moe_stack_workspace_bytes(T), initialised with
 *             moe_workspace_init (its first moe_workspace_bytes(T) bytes are
 *             the layers' shared workspace; the device flag lives there).
 * Errors: as moe_layer_forward_prenorm, for the first failing layer; nothing
 * is enqueued on a host-side error.
 */
moe_status moe_stack_forward(void *x, const moe_layer_weights *layers, int n_layers, int T, float eps,
                             void *workspace, size_t workspace_bytes, moe_stream_t stream);

/* ----------------------------------------------------------------------- */
/* The layer without a caller-provided workspace.  The pages describe no   */
/* such entry point; it exists for callers that cannot allocate.           */
/* ----------------------------------------------------------------------- */

/* Bytes of the library's fixed per-device scratch: the workspace of
 * moe_layer_forward at T = MOE_MAX_DECODE_T. */
#define MOE_STATIC_SCRATCH_BYTES 7400448u

/*
 * moe_layer_forward with the workspace replaced by a fixed device array of
 * MOE_STATIC_SCRATCH_BYTES inside the library, for callers that cannot own or
 * allocate device memory (a plugin interface that passes only inputs and
 * outputs, a process whose device memory is fixed at start-up).  Computes
 * exactly what moe_layer_forward computes (same kernel, same results).
 *  Arguments: as moe_layer_forward, without workspace / workspace_bytes.
 *  Allocation: none; no cudaMalloc / cudaFree and no allocating library call.
 *  First call on each device: looks up the array's device address with
 *    cudaGetSymbolAddress (that device current) and zeroes the array on
 *    `stream`; make that first call before any stream capture.  Every call
 *    then launches two kernels: the re-arm kernel of moe_workspace_recover
 *    on the scratch, then the layer.
 *  Zero state: the setup zeroes the scratch; every call leaves its counters
 *    re-armed for the next call (the launch tag advances by one), and after a
 *    call that gave up on a bounded wait the next call's re-arm kernel
 *    restores them.  moe_static_read_device_flag reports the scratch's
 *    device flag.
 *  Concurrency: one scratch per device.  Calls on the same device must not
 *    overlap (serialise them on one stream or with events); overlapping calls
 *    race on the scratch and give wrong results.
 *  Errors: MOE_ERR_UNSUPPORTED for T outside 1..MOE_MAX_DECODE_T (the
 *    scratch's maximum), before any CUDA call; MOE_ERR_CUDA if the setup
 *    fails; otherwise the statuses of moe_layer_forward.
 */
moe_status moe_layer_forward_static(const void *x, const void *router_w,
                                    const moe_expert_bank *routed,
                                    const moe_expert_bank *shared, void *out, int T,
                                    moe_stream_t stream);

/*
 * moe_read_device_flag for the fixed scratch of moe_layer_forward_static on
 * the current device: SYNCHRONISES `stream`, returns the MOE_FLAG_* bits in
 * *flag_out (host) and clears them.  A MOE_FLAG_WAIT_TIMEOUT means the call
 * that set it returned invalid output; the following calls are valid again
 * (their re-arm kernel restored the scratch).  The first use on a device
 * does the scratch's set-up (see above) and reports 0.
 * Errors: MOE_ERR_INVALID_ARG (flag_out NULL), MOE_ERR_DEVICE_FLAG (a bit
 * was set), MOE_ERR_CUDA.
 */
moe_status moe_static_read_device_flag(moe_stream_t stream, uint32_t *flag_out);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */

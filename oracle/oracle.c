/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.  Not part of the product path.
 *
 * A plain, slow, fp64 CPU restatement of the small-batch weight-only NVFP4
 * (W4A16) mixture-of-experts layer.  Only tests/, __graft_entry__.smoke() and
 * the cpu_baseline / reference legs of bench.py may load this library.  It
 * shares no code, header, table or constant with the CUDA path
 * (nvfp4_moe_decode_gb300/csrc), and neither side includes the other.
 *
 * Sources (web pages, cited by title and section):
 *  [FLINT]  "vLLM adds day-0 support for Recursive's Flint, hitting about 485
 *           tokens/s on one GB200", section "A 40B MoE that activates 2.5B
 *           parameters": 256 experts, sigmoid top-6 routing plus a shared
 *           expert; NVFP4 weights run weight-only (W4A16) with BF16
 *           activations.
 *  [FLINT-ZH] the Chinese mirror of the same post, section 模型架构 (model
 *           architecture): 256 experts, sigmoid top-6, plus one shared expert.
 *  [INKLING] "TML Inkling on vLLM", section "MoE": 256 routed experts
 *           (top-6) plus 2 shared experts that act as expert sinks; only the
 *           routed experts are NVFP4, the shared experts BF16.
 *  [MOET]   "Frontier MoE on consumer Blackwell (SM120)", section
 *           "GLM-5.2 (753B) - the headline model": an NVFP4 weight is an e2m1
 *           code times an e4m3 scale per block of 16 times a per-tensor fp32
 *           scale ("scale_2").
 *
 * Readings where the pages are silent:
 *  - canonical byte layout: codes [N][K/2], element (n, 2j) in the LOW nibble
 *    of byte (n, j), element (n, 2j+1) in the HIGH nibble; scales [N][K/16],
 *    block b covers k in [16b, 16b+16) along the reduction (input) axis;
 *  - e4m3 is the OCP E4M3FN flavour (no infinity, S.1111.111 is NaN);
 *  - gate/up matrix W13 is [2I][H]: rows [0, I) are the gate, [I, 2I) the up
 *    projection; the down matrix W2 is [H][I];
 *  - expert MLP: h = silu(W_gate x) * (W_up x), y = W2 h, no clamp;
 *  - routing: s_e = sigmoid(logit_e); the k experts with the largest logits
 *    are selected (sigmoid is monotone), a tie goes to the lower index; the
 *    selected weights are renormalised to sum to 1; the shared expert is
 *    always added with weight 1;
 *  - the selection (an integer decided by floating point) is taken on the
 *    logits rounded to fp32, the precision the kernels decide in; the weights
 *    are computed from the fp64 logits.
 *
 * Everything else is evaluated in fp64 with no intermediate rounding.
 *
 * Mutation hooks: building with -DORACLE_MUTANT=n plants one deliberate
 * mistake (see the ORACLE_MUTANT blocks).  The pin tests compile such
 * variants to prove that each planted mistake is caught.  A normal build
 * defines none of them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ------------------------------------------------------------------------ */
/* Scalar decoders, by the format definitions.                               */
/* ------------------------------------------------------------------------ */

/* e2m1 (FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value = mantissa * 0.5.
 * Otherwise value = 2^(E-1) * (1 + M/2).  [MOET, "GLM-5.2": e2m1 codes] */
double oracle_e2m1_value(int code)
{
    int sign = (code >> 3) & 1;
    int E = (code >> 1) & 3;
    int M = code & 1;
    double mag;
    if (E == 0)
        mag = M * 0.5;
    else
        mag = ldexp(1.0 + M / 2.0, E - 1);
#if ORACLE_MUTANT == 1 /* planted: subnormal code read as 1.0 */
    if (E == 0 && M == 1)
        mag = 1.0;
#endif
    return sign ? -mag : mag;
}

/* e4m3 (OCP E4M3FN): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa.  Exponent 0 is subnormal: (M/8) * 2^-6.  S.1111.111 is NaN;
 * there is no infinity, so the largest finite value is 448.
 * [MOET, "GLM-5.2": e4m3 block-16 scales] */
double oracle_e4m3_value(int code)
{
    int sign = (code >> 7) & 1;
    int E = (code >> 3) & 15;
    int M = code & 7;
    double mag;
    if (E == 15 && M == 7)
        return NAN;
    if (E == 0)
        mag = ldexp(M / 8.0, -6);
    else
        mag = ldexp(1.0 + M / 8.0, E - 7);
#if ORACLE_MUTANT == 2 /* planted: exponent bias off by one */
    if (E != 0)
        mag = ldexp(1.0 + M / 8.0, E - 8);
#endif
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_value(int bits)
{
    uint32_t u = ((uint32_t)(bits & 0xFFFF)) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element (n, k) of a canonical NVFP4 matrix [N][K]. */
static int canonical_code(const uint8_t *codes, int K, int n, int k)
{
    uint8_t byte = codes[(size_t)n * (K / 2) + (size_t)(k / 2)];
#if ORACLE_MUTANT == 3 /* planted: nibble order swapped */
    return (k % 2 == 0) ? (byte >> 4) & 15 : byte & 15;
#else
    return (k % 2 == 0) ? byte & 15 : (byte >> 4) & 15;
#endif
}

static int canonical_scale(const uint8_t *scales, int K, int n, int k)
{
#if ORACLE_MUTANT == 4 /* planted: scale taken from the neighbouring block */
    return scales[(size_t)n * (K / 16) + (size_t)((k / 16 + 1) % (K / 16))];
#else
    return scales[(size_t)n * (K / 16) + (size_t)(k / 16)];
#endif
}

/* Dequantise a canonical NVFP4 matrix: W[n][k] = e2m1 * e4m3 * tscale.
 * [MOET, "GLM-5.2": e2m1 x e4m3 block-16 x per-tensor scale_2] */
void oracle_dequant_nvfp4(const uint8_t *codes, const uint8_t *scales, float tscale,
                          int N, int K, double *W)
{
    for (int n = 0; n < N; n++)
        for (int k = 0; k < K; k++)
            W[(size_t)n * K + k] = oracle_e2m1_value(canonical_code(codes, K, n, k)) *
                                   oracle_e4m3_value(canonical_scale(scales, K, n, k)) *
                                   (double)tscale;
}

/* A bf16 row-major matrix [N][K] to fp64. */
void oracle_dequant_bf16(const uint16_t *w, int N, int K, double *W)
{
    for (size_t i = 0; i < (size_t)N * K; i++)
        W[i] = oracle_bf16_value(w[i]);
}

/* ------------------------------------------------------------------------ */
/* Dense GEMV.  [FLINT, "From 1,096 kernels to 346": the small-batch dense  */
/* GEMV on the same packed NVFP4 weights]  Its plain definition:            */
/*   y[t][n] = sum_k W[n][k] * x[t][k],  W dequantised as above, x bf16.    */
/* fp64 products (exact) and an fp64 sum in k order; no rounding of y.      */
/* ------------------------------------------------------------------------ */

void oracle_dense_gemv_nvfp4(const uint8_t *codes, const uint8_t *scales, float tscale, int N, int K,
                             const uint16_t *x, int T, double *y)
{
    double *W = (double *)malloc(sizeof(double) * (size_t)N * K);
#if ORACLE_MUTANT == 15 /* planted: the tensor scale left out */
    tscale = 1.0f;
#endif
    oracle_dequant_nvfp4(codes, scales, tscale, N, K, W);
    int kend = K;
#if ORACLE_MUTANT == 16 /* planted: the last column dropped from the sum */
    kend = K - 1;
#endif
    for (int t = 0; t < T; t++)
        for (int n = 0; n < N; n++) {
            double acc = 0.0;
            for (int k = 0; k < kend; k++)
                acc += W[(size_t)n * K + k] * oracle_bf16_value(x[(size_t)t * K + k]);
            y[(size_t)t * N + n] = acc;
        }
    free(W);
}

/* ------------------------------------------------------------------------ */
/* Router: logits, sigmoid, top-k, renormalise.  [FLINT, "A 40B MoE ..."]    */
/* ------------------------------------------------------------------------ */

/* logits[t][e] = sum_k x[t][k] * Wr[e][k]; bf16 inputs, fp64 products (exact)
 * and an fp64 sum in k order. */
void oracle_router_logits(const uint16_t *x, const uint16_t *wr, int T, int H, int E,
                          double *logits)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++)
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int k = 0; k < H; k++)
#if ORACLE_MUTANT == 10 /* planted: router matrix read transposed */
                acc += oracle_bf16_value(x[(size_t)t * H + k]) *
                       oracle_bf16_value(wr[(size_t)k * E + e]);
#else
                acc += oracle_bf16_value(x[(size_t)t * H + k]) *
                       oracle_bf16_value(wr[(size_t)e * H + k]);
#endif
            logits[(size_t)t * E + e] = acc;
        }
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* "a ranks before b": larger fp32-rounded logit first, then lower index. */
static int ranks_before(const double *lg, int a, int b)
{
    float fa = (float)lg[a], fb = (float)lg[b];
#if ORACLE_MUTANT == 5 /* planted: tie broken towards the higher index */
    if (fa != fb)
        return fa > fb;
    return a > b;
#else
    if (fa != fb)
        return fa > fb;
    return a < b;
#endif
}

/* For each token pick the top_k experts (selection order: best first) and
 * their renormalised sigmoid weights.  Returns 0, or -1 on a NaN logit. */
int oracle_select_topk(const double *logits, int T, int E, int top_k, int32_t *idx, double *w)
{
    for (int t = 0; t < T; t++) {
        const double *lg = logits + (size_t)t * E;
        for (int e = 0; e < E; e++)
            if (isnan(lg[e]))
                return -1;
        int32_t *sel = idx + (size_t)t * top_k;
        /* selection by repeated scan: the best expert not yet chosen */
        for (int i = 0; i < top_k; i++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                int taken = 0;
                for (int j = 0; j < i; j++)
                    if (sel[j] == e)
                        taken = 1;
                if (taken)
                    continue;
                if (best < 0 || ranks_before(lg, e, best))
                    best = e;
            }
            sel[i] = best;
        }
        double denom = 0.0;
        for (int i = 0; i < top_k; i++)
            denom += sigmoid(lg[sel[i]]);
        for (int i = 0; i < top_k; i++) {
#if ORACLE_MUTANT == 6 /* planted: weights not renormalised */
            w[(size_t)t * top_k + i] = sigmoid(lg[sel[i]]);
#else
            w[(size_t)t * top_k + i] = sigmoid(lg[sel[i]]) / denom;
#endif
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Expert MLP and the layer.                                                 */
/* ------------------------------------------------------------------------ */

/* One expert on one token: g = W13[0:I] x, u = W13[I:2I] x,
 * h = g * sigmoid(g) * u, y = W2 h.  W13 is [2I][H], W2 is [H][I]. */
void oracle_expert_ffn(const double *W13, const double *W2, const double *xt, int H, int I,
                       double *y)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; i++) {
        double g = 0.0, u = 0.0;
        for (int k = 0; k < H; k++) {
            g += W13[(size_t)i * H + k] * xt[k];
            u += W13[(size_t)(I + i) * H + k] * xt[k];
        }
#if ORACLE_MUTANT == 7 /* planted: gate and up swapped */
        h[i] = u * sigmoid(u) * g;
#elif ORACLE_MUTANT == 8 /* planted: SiLU replaced by plain sigmoid */
        h[i] = sigmoid(g) * u;
#else
        h[i] = g * sigmoid(g) * u;
#endif
    }
    for (int n = 0; n < H; n++) {
        double acc = 0.0;
        for (int i = 0; i < I; i++)
#if ORACLE_MUTANT == 11 /* planted: down matrix read transposed */
            acc += W2[(size_t)i * H + n] * h[i];
#else
            acc += W2[(size_t)n * I + i] * h[i];
#endif
        y[n] = acc;
    }
    free(h);
}

/* Weight banks handed to the layer.  wtype 0: NVFP4 canonical (a = codes,
 * b = scales, ts = per-tensor scale); wtype 1: bf16 row-major (a = weights,
 * b and ts unused).  Any pointer of an expert that no token selects may be
 * NULL; selecting such an expert is an error (-2). */
static int dequant_expert(int wtype, const void *a13, const void *b13, float ts13,
                          const void *a2, const void *b2, float ts2, int H, int I,
                          double *W13, double *W2)
{
    if (a13 == NULL || a2 == NULL)
        return -2;
    if (wtype == 0) {
        if (b13 == NULL || b2 == NULL)
            return -2;
        oracle_dequant_nvfp4((const uint8_t *)a13, (const uint8_t *)b13, ts13, 2 * I, H, W13);
        oracle_dequant_nvfp4((const uint8_t *)a2, (const uint8_t *)b2, ts2, H, I, W2);
    } else {
        oracle_dequant_bf16((const uint16_t *)a13, 2 * I, H, W13);
        oracle_dequant_bf16((const uint16_t *)a2, H, I, W2);
    }
    return 0;
}

/* Apply one expert to the tokens in `toks` with weights `gw`, adding
 * gw * y into out (fp64, [T][H]). */
static void apply_expert(const double *W13, const double *W2, const double *xd, int H, int I,
                         const int *toks, const double *gw, int ntok, double *out)
{
#pragma omp parallel
    {
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int j = 0; j < ntok; j++) {
            int t = toks[j];
            oracle_expert_ffn(W13, W2, xd + (size_t)t * H, H, I, y);
            for (int n = 0; n < H; n++)
                out[(size_t)t * H + n] += gw[j] * y[n];
        }
        free(y);
    }
}

/*
 * The full layer for T tokens:
 *   out[t] = sum_{i<top_k} w[t][i] * FFN_{idx[t][i]}(x[t]) + FFN_shared(x[t])
 * (the shared term only when has_shared).  [FLINT, "A 40B MoE ..."]
 *
 * x [T][H] bf16 bits, wr [E][H] bf16 bits.  Routed bank: per-expert pointer
 * arrays of length E (see dequant_expert).  Outputs: out [T][H] fp64,
 * idx [T][top_k], w [T][top_k] (may be NULL), logits [T][E] (may be NULL).
 * Returns 0, -1 on a NaN logit, -2 when a selected expert has no weights,
 * -3 on bad sizes.
 */
int oracle_moe_forward(const uint16_t *x, const uint16_t *wr, int T, int H, int E, int I,
                       int top_k, int wtype, const void *const *a13, const void *const *b13,
                       const float *ts13, const void *const *a2, const void *const *b2,
                       const float *ts2, int has_shared, int shared_wtype, const void *s_a13,
                       const void *s_b13, float s_ts13, const void *s_a2, const void *s_b2,
                       float s_ts2, double *out, int32_t *idx_out, double *w_out,
                       double *logits_out)
{
    if (T < 0 || H <= 0 || E <= 0 || I <= 0 || top_k <= 0 || top_k > E || H % 16 || I % 16)
        return -3;
    int rc = 0;
    double *logits = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * E);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1) * top_k);
    double *w = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * top_k);
    double *xd = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * H);
    double *W13 = (double *)malloc(sizeof(double) * (size_t)2 * I * H);
    double *W2 = (double *)malloc(sizeof(double) * (size_t)H * I);
    int *toks = (int *)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
    double *gw = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));

    for (size_t i = 0; i < (size_t)T * H; i++) {
        xd[i] = oracle_bf16_value(x[i]);
        out[i] = 0.0;
    }
    oracle_router_logits(x, wr, T, H, E, logits);
    if (oracle_select_topk(logits, T, E, top_k, idx, w) != 0) {
        rc = -1;
        goto done;
    }
    for (int e = 0; e < E; e++) {
        int n = 0;
        for (int t = 0; t < T; t++)
            for (int i = 0; i < top_k; i++)
                if (idx[(size_t)t * top_k + i] == e) {
                    toks[n] = t;
                    gw[n] = w[(size_t)t * top_k + i];
                    n++;
                }
        if (n == 0)
            continue;
        rc = dequant_expert(wtype, a13[e], b13 ? b13[e] : NULL, ts13 ? ts13[e] : 1.0f, a2[e],
                            b2 ? b2[e] : NULL, ts2 ? ts2[e] : 1.0f, H, I, W13, W2);
        if (rc != 0)
            goto done;
        apply_expert(W13, W2, xd, H, I, toks, gw, n, out);
    }
#if ORACLE_MUTANT == 9 /* planted: shared expert dropped */
    has_shared = 0;
#endif
    if (has_shared && T > 0) {
        rc = dequant_expert(shared_wtype, s_a13, s_b13, s_ts13, s_a2, s_b2, s_ts2, H, I, W13, W2);
        if (rc != 0)
            goto done;
        for (int t = 0; t < T; t++) {
            toks[t] = t;
            gw[t] = 1.0;
        }
        apply_expert(W13, W2, xd, H, I, toks, gw, T, out);
    }
done:
    if (idx_out)
        memcpy(idx_out, idx, sizeof(int32_t) * (size_t)T * top_k);
    if (w_out)
        memcpy(w_out, w, sizeof(double) * (size_t)T * top_k);
    if (logits_out)
        memcpy(logits_out, logits, sizeof(double) * (size_t)T * E);
    free(logits);
    free(idx);
    free(w);
    free(xd);
    free(W13);
    free(W2);
    free(toks);
    free(gw);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Expert sinks.  [INKLING, "MoE": 256 routed experts (top-6) plus 2 shared  */
/* experts; the shared experts take part in the routing-score computation,   */
/* absorbing probability mass, but are never candidates for the top-6.]      */
/* Readings (the page gives no formula):                                     */
/*  - the router has E + S rows, the last S being the shared experts';      */
/*  - every row gets the score s = sigmoid(logit), as for the routed ones;  */
/*  - the top_k are chosen among the E routed experts exactly as in          */
/*    oracle_select_topk;                                                    */
/*  - with D = (sum of s over the selected) + (sum of s over the S sinks),   */
/*    selected expert e gets the weight s_e / D and shared expert j the      */
/*    weight s_{E+j} / D; nothing else scales them.                          */
/* ------------------------------------------------------------------------ */

/* logits [T][E+S]; idx, w [T][top_k]; sw [T][S].  Returns 0, or -1 on a NaN
 * logit. */
int oracle_select_topk_sink(const double *logits, int T, int E, int S, int top_k, int32_t *idx, double *w,
                            double *sw)
{
    double *row = (double *)malloc(sizeof(double) * (size_t)E);
    int rc = 0;
    for (int t = 0; t < T && rc == 0; t++) {
        const double *lg = logits + (size_t)t * (E + S);
        for (int e = 0; e < E + S; e++)
            if (isnan(lg[e]))
                rc = -1;
        if (rc != 0)
            break;
        int32_t *sel = idx + (size_t)t * top_k;
        double *wt = w + (size_t)t * top_k;
#if ORACLE_MUTANT == 18 /* planted: the sinks are candidates of the top-k */
        {
            int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)top_k);
            double *tw = (double *)malloc(sizeof(double) * (size_t)top_k);
            oracle_select_topk(lg, 1, E + S, top_k, tmp, tw);
            for (int i = 0; i < top_k; i++)
                sel[i] = tmp[i] < E ? tmp[i] : 0;
            free(tmp);
            free(tw);
        }
#else
        memcpy(row, lg, sizeof(double) * (size_t)E);
        oracle_select_topk(row, 1, E, top_k, sel, wt);   /* the selection; weights recomputed below */
#endif
        double denom = 0.0;
        for (int i = 0; i < top_k; i++)
            denom += sigmoid(lg[sel[i]]);
#if ORACLE_MUTANT != 17 /* planted (17): the sinks left out of the denominator */
        for (int j = 0; j < S; j++)
            denom += sigmoid(lg[E + j]);
#endif
        for (int i = 0; i < top_k; i++)
            wt[i] = sigmoid(lg[sel[i]]) / denom;
        for (int j = 0; j < S; j++)
            sw[(size_t)t * S + j] = sigmoid(lg[E + j]) / denom;
    }
    free(row);
    return rc;
}

/*
 * The layer with S shared experts, which may be stored in another weight
 * type than the routed bank (TML Inkling's NVFP4 checkpoint keeps only the
 * routed experts in NVFP4; the shared experts are BF16), optionally as
 * expert sinks:
 *   out[t] = sum_i w[t][i] * FFN_{idx[t][i]}(x[t]) + sum_j sw[t][j] * FFN_shared_j(x[t])
 * with sink = 1: wr has E + S rows and (idx, w, sw) come from
 * oracle_select_topk_sink; sink = 0: wr has E rows, (idx, w) from
 * oracle_select_topk and sw = 1.  Shared expert j: s_a13[j], s_b13[j],
 * s_ts13[j], s_a2[j], s_b2[j], s_ts2[j] (dequant_expert's meaning, type
 * shared_wtype).  Outputs: out [T][H]; idx, w [T][top_k]; sw [T][S];
 * logits [T][E + sink * S] (any output but out may be NULL).  Returns as
 * oracle_moe_forward.
 */
int oracle_moe_forward_sinks(const uint16_t *x, const uint16_t *wr, int T, int H, int E, int I, int top_k,
                             int wtype, const void *const *a13, const void *const *b13, const float *ts13,
                             const void *const *a2, const void *const *b2, const float *ts2, int S, int sink,
                             int shared_wtype, const void *const *s_a13, const void *const *s_b13,
                             const float *s_ts13, const void *const *s_a2, const void *const *s_b2,
                             const float *s_ts2, double *out, int32_t *idx_out, double *w_out, double *sw_out,
                             double *logits_out)
{
    if (T < 0 || H <= 0 || E <= 0 || I <= 0 || top_k <= 0 || top_k > E || H % 16 || I % 16 || S < 0)
        return -3;
    const int R = E + (sink ? S : 0);
    const size_t T1 = (size_t)(T > 0 ? T : 1);
    int rc = 0;
    double *logits = (double *)malloc(sizeof(double) * T1 * R);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * T1 * top_k);
    double *w = (double *)malloc(sizeof(double) * T1 * top_k);
    double *sw = (double *)malloc(sizeof(double) * T1 * (S > 0 ? S : 1));
    double *xd = (double *)malloc(sizeof(double) * T1 * H);
    double *W13 = (double *)malloc(sizeof(double) * (size_t)2 * I * H);
    double *W2 = (double *)malloc(sizeof(double) * (size_t)H * I);
    int *toks = (int *)malloc(sizeof(int) * T1);
    double *gw = (double *)malloc(sizeof(double) * T1);

    for (size_t i = 0; i < (size_t)T * H; i++) {
        xd[i] = oracle_bf16_value(x[i]);
        out[i] = 0.0;
    }
    oracle_router_logits(x, wr, T, H, R, logits);
    if (sink) {
        if (oracle_select_topk_sink(logits, T, E, S, top_k, idx, w, sw) != 0) {
            rc = -1;
            goto done;
        }
    } else {
        if (oracle_select_topk(logits, T, E, top_k, idx, w) != 0) {
            rc = -1;
            goto done;
        }
        for (size_t i = 0; i < (size_t)T * S; i++)
            sw[i] = 1.0;
    }
    for (int e = 0; e < E; e++) {
        int n = 0;
        for (int t = 0; t < T; t++)
            for (int i = 0; i < top_k; i++)
                if (idx[(size_t)t * top_k + i] == e) {
                    toks[n] = t;
                    gw[n] = w[(size_t)t * top_k + i];
                    n++;
                }
        if (n == 0)
            continue;
        rc = dequant_expert(wtype, a13[e], b13 ? b13[e] : NULL, ts13 ? ts13[e] : 1.0f, a2[e],
                            b2 ? b2[e] : NULL, ts2 ? ts2[e] : 1.0f, H, I, W13, W2);
        if (rc != 0)
            goto done;
        apply_expert(W13, W2, xd, H, I, toks, gw, n, out);
    }
    for (int j = 0; j < S && T > 0; j++) {
        rc = dequant_expert(shared_wtype, s_a13[j], s_b13 ? s_b13[j] : NULL, s_ts13 ? s_ts13[j] : 1.0f,
                            s_a2[j], s_b2 ? s_b2[j] : NULL, s_ts2 ? s_ts2[j] : 1.0f, H, I, W13, W2);
        if (rc != 0)
            goto done;
        for (int t = 0; t < T; t++) {
            toks[t] = t;
            gw[t] = sw[(size_t)t * S + j];
        }
        apply_expert(W13, W2, xd, H, I, toks, gw, T, out);
    }
done:
    if (idx_out)
        memcpy(idx_out, idx, sizeof(int32_t) * (size_t)T * top_k);
    if (w_out)
        memcpy(w_out, w, sizeof(double) * (size_t)T * top_k);
    if (sw_out)
        memcpy(sw_out, sw, sizeof(double) * (size_t)T * S);
    if (logits_out)
        memcpy(logits_out, logits, sizeof(double) * (size_t)T * R);
    free(logits);
    free(idx);
    free(w);
    free(sw);
    free(xd);
    free(W13);
    free(W2);
    free(toks);
    free(gw);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Decoder stack: the pre-norm residual step.  [FLINT, "A 40B MoE ...": a    */
/* 47-layer pre-norm decoder.]  Reading (the pages say only "pre-norm"):     */
/* layer l maps the bf16 residual stream x to x + MoE(RMSNorm(x)), RMSNorm   */
/* with unit weight: v / sqrt(mean(v^2) + eps); the normalised activations  */
/* and the residual stream are bf16 tensors (the activations are BF16).     */
/* ------------------------------------------------------------------------ */

/* Nearest bf16 to v (ties to even), as bf16 bits.  bf16 keeps 8 significand
 * bits: with v = m * 2^e, 0.5 <= |m| < 1, the representable neighbours are
 * multiples of 2^(e-8) (2^-133 below the normal range, exponent e < -125).
 * Values past the largest bf16 round to infinity; NaN stays NaN. */
uint16_t oracle_round_bf16(double v)
{
    if (v != v)
        return 0x7FC0;
    if (v == 0.0)
        return signbit(v) ? 0x8000 : 0x0000;
    int e;
    frexp(v, &e);
    if (e < -125)
        e = -125;
    double q = ldexp(v, 8 - e);          /* |q| < 256, exact */
#if ORACLE_MUTANT == 14 /* planted: truncation instead of round-to-nearest-even */
    double r = trunc(q);
#else
    double r = nearbyint(q);             /* default rounding mode: nearest, ties to even */
#endif
    double rv = ldexp(r, e - 8);
    float f = (float)rv;                 /* exact: rv has <= 9 significant bits */
    if (fabs(rv) >= 0x1p128)
        f = (float)(rv > 0 ? INFINITY : -INFINITY);
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return (uint16_t)(bits >> 16);
}

/* One pre-norm step for T tokens of H values: v = bf16(x + delta) (delta may
 * be NULL: v = x), xn = bf16(v / sqrt(mean_k v_k^2 + eps)), both as bf16
 * bits; the sum, mean, root and quotient in fp64. */
void oracle_prenorm(const uint16_t *x, const uint16_t *delta, int T, int H, double eps,
                    uint16_t *v_out, uint16_t *xn_out)
{
    double *v = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    for (int t = 0; t < T; t++) {
        double ss = 0.0;
        for (int k = 0; k < H; k++) {
            size_t i = (size_t)t * H + k;
            double s = oracle_bf16_value(x[i]) + (delta ? oracle_bf16_value(delta[i]) : 0.0);
            v_out[i] = oracle_round_bf16(s);
            v[k] = oracle_bf16_value(v_out[i]);
            ss += v[k] * v[k];
        }
#if ORACLE_MUTANT == 12 /* planted: sum of squares instead of their mean */
        double ms = ss;
#else
        double ms = ss / H;
#endif
#if ORACLE_MUTANT == 13 /* planted: eps added after the root */
        double scale = 1.0 / (sqrt(ms) + eps);
#else
        double scale = 1.0 / sqrt(ms + eps);
#endif
        for (int k = 0; k < H; k++)
            xn_out[(size_t)t * H + k] = oracle_round_bf16(v[k] * scale);
    }
    free(v);
}

/* Threads an OpenMP region in this library uses (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

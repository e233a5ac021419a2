/*
 * mx_oracle.c -- plain single-threaded reference of the routed-MoE FFN block.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).  It
 * shares nothing with the CUDA library.  Build with -ffp-contract=off; every
 * multiply-add of the definition is an explicit fmaf, which is IEEE-exact.
 *
 * Citations are to the pages the method is taken from:
 *   [Mference]   "Mference System design" page;
 *   [TinyTitan]  "TinyTitan_Datacenter Architecture" page.
 * Readings of points the pages leave open are marked READING.
 */
#include "mx_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- dtypes */

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN stays a quiet NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    /* round to nearest, ties to even, on the 16 discarded bits */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static float load_act(const void *x, int dtype, long i)
{
    if (dtype == 1)
        return oracle_bf16_to_f32(((const uint16_t *)x)[i]);
    return ((const float *)x)[i];
}

static void store_act(void *y, int dtype, long i, float v)
{
    if (dtype == 1)
        ((uint16_t *)y)[i] = oracle_f32_to_bf16(v);
    else
        ((float *)y)[i] = v;
}

/* ------------------------------------------------------- quantized values */

/* Quantized integer at column c of one packed row: low nibble / byte first
 * [Mference, "Why the runtime has this shape": packed 4-bit values; 8-bit router]. */
static unsigned qval(const uint32_t *row, int bits, int c)
{
    if (bits == 4)
        return (row[c >> 3] >> (4 * (c & 7))) & 15u;
    return (row[c >> 2] >> (8 * (c & 3))) & 255u;
}

/* Dequantized weight w = s*q + b with the BF16 scale and bias of its group of
 * 64 [Mference, "Why the runtime has this shape": "a BF16 scale and BF16 bias
 * for each group of 64 weights"].  One rounding (fmaf). */
static float dequant(const oracle_qmat *m, int r, int c)
{
    int G = m->cols / 64;
    const uint32_t *row = m->w + (long)r * (m->cols * m->bits / 32);
    float s = oracle_bf16_to_f32(m->s[(long)r * G + c / 64]);
    float b = oracle_bf16_to_f32(m->b[(long)r * G + c / 64]);
    return fmaf(s, (float)qval(row, m->bits, c), b);
}

/* Plain definition of a quantized matrix-vector product: dequantize each
 * weight, then one fp32 dot product in ascending column order. */
void oracle_qmatvec(const oracle_qmat *m, const float *x, float *y)
{
    for (int r = 0; r < m->rows; ++r) {
        float acc = 0.0f;
        for (int c = 0; c < m->cols; ++c)
            acc = fmaf(dequant(m, r, c), x[c], acc);
        y[r] = acc;
    }
}

/* ---------------------------------------------------------------- GELU */

/* GELU, tanh form.  READING: the pages say only "GeGLU" [Mference, "Metal
 * execution"]; the tanh approximation is the Gemma-family convention. */
float oracle_gelu(float z)
{
    const float k0 = 0.7978845608028654f; /* sqrt(2/pi) */
    const float k1 = 0.044715f;
    float inner = k0 * (z + k1 * z * z * z);
    return 0.5f * z * (1.0f + tanhf(inner));
}

/* --------------------------------------------------------------- router */

/* Router logits: logits = int8_affine(x) [Mference, "Decode", router formula].
 *
 * READING (canonical order): the int8 affine projection is written in its
 * group-factored form, which is algebraically the dequantized dot product
 *     logit[t,e] = sum_g  s[e,g] * P[t,e,g]  +  b[e,g] * X[t,g]
 *     P[t,e,g]   = sum_{i in g} q[e,i] * x[t,i],   X[t,g] = sum_{i in g} x[t,i]
 * evaluated in this fixed order, so that the discrete top-k decision is
 * reproducible bit for bit [TinyTitan, "Invariants", items 1-2]:
 *   X: fp32 adds, i ascending, starting from 0;
 *   P: P = fmaf(q_i, x_i, P), i ascending, starting from 0;
 *   acc = fmaf(s, P, acc); acc = fmaf(b, X, acc), g ascending, from 0. */
void oracle_router_logits(const oracle_qmat *router, const float *x, int T, float *logits)
{
    const int D = router->cols, E = router->rows, G = D / 64;
    float *X = (float *)malloc(sizeof(float) * (size_t)G);
    for (int t = 0; t < T; ++t) {
        const float *xt = x + (long)t * D;
        for (int g = 0; g < G; ++g) {
            float a = 0.0f;
            for (int i = 0; i < 64; ++i)
                a = a + xt[64 * g + i];
            X[g] = a;
        }
        for (int e = 0; e < E; ++e) {
            const uint32_t *row = router->w + (long)e * (D * router->bits / 32);
            float acc = 0.0f;
            for (int g = 0; g < G; ++g) {
                float P = 0.0f;
                for (int i = 0; i < 64; ++i)
                    P = fmaf((float)qval(row, router->bits, 64 * g + i), xt[64 * g + i], P);
                float s = oracle_bf16_to_f32(router->s[(long)e * G + g]);
                float b = oracle_bf16_to_f32(router->b[(long)e * G + g]);
                acc = fmaf(s, P, acc);
                acc = fmaf(b, X[g], acc);
            }
            logits[(long)t * E + e] = acc;
        }
    }
    free(X);
}

/* highest_K then softmax(logits[topK]) * per_expert_scale[topK]
 * [Mference, "Decode", router formula].  Order: descending logit, ties to the
 * lower expert index (lowest-index-wins); NaN ranks as -inf, and enters the
 * softmax as -inf.  The softmax is taken over the K selected logits, shifted
 * by the largest, in fp32. */
int oracle_topk_softmax(const float *logits, int T, int E, int K,
                        const float *per_expert_scale, int32_t *topk_idx, float *topk_w)
{
    if (T < 0 || E < 1 || K < 1 || K > E)
        return -1;
    char *taken = (char *)malloc((size_t)E);
    float *ev = (float *)malloc(sizeof(float) * (size_t)K);
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (long)t * E;
        memset(taken, 0, (size_t)E);
        for (int k = 0; k < K; ++k) {
            int best = -1;
            float bv = 0.0f;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                float v = isnan(l[e]) ? -INFINITY : l[e];
                if (best < 0 || v > bv) { /* strict: an equal value keeps the lower index */
                    best = e;
                    bv = v;
                }
            }
            taken[best] = 1;
            topk_idx[(long)t * K + k] = best;
        }
        /* a NaN logit is -inf here too (the reading above), so a selected NaN
         * gets weight 0 */
        const float m0 = l[topk_idx[(long)t * K]];
        const float m = isnan(m0) ? -INFINITY : m0;
        float sum = 0.0f;
        for (int k = 0; k < K; ++k) {
            const float v = l[topk_idx[(long)t * K + k]];
            ev[k] = expf((isnan(v) ? -INFINITY : v) - m);
            sum = sum + ev[k];
        }
        for (int k = 0; k < K; ++k) {
            float w = ev[k] / sum;
            if (per_expert_scale)
                w = w * per_expert_scale[topk_idx[(long)t * K + k]];
            topk_w[(long)t * K + k] = w;
        }
    }
    free(taken);
    free(ev);
    return 0;
}

/* Grouping of token/expert pairs into per-expert work [Mference, "Prefill":
 * "groups token/expert pairs into bounded routed-MoE work"].  READING: slots
 * s = t*K + k are listed expert by expert, ascending s within an expert. */
int oracle_permute(const int32_t *topk_idx, int T, int K, int E,
                   int32_t *counts, int32_t *offsets, int32_t *perm)
{
    long n = (long)T * K;
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (long s = 0; s < n; ++s) {
        if (topk_idx[s] < 0 || topk_idx[s] >= E)
            return -1;
        counts[topk_idx[s]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    long pos = 0;
    for (int e = 0; e < E; ++e)
        for (long s = 0; s < n; ++s)
            if (topk_idx[s] == e)
                perm[pos++] = (int32_t)s;
    return 0;
}

/* ------------------------------------------------------------ expert FFN */

/* GELU-gated expert: h = gelu(W_gate x) * (W_up x); y = W_down h
 * [Mference, "Metal execution": affine decode + GeGLU; gem "Native
 * architecture", GELU-gated FFN].  h stays fp32. */
void oracle_expert_ffn(const oracle_qmat *gate, const oracle_qmat *up, const oracle_qmat *down,
                       const float *x, float *y)
{
    int H = gate->rows;
    float *g = (float *)malloc(sizeof(float) * (size_t)H);
    float *u = (float *)malloc(sizeof(float) * (size_t)H);
    oracle_qmatvec(gate, x, g);
    oracle_qmatvec(up, x, u);
    for (int j = 0; j < H; ++j)
        g[j] = oracle_gelu(g[j]) * u[j];
    oracle_qmatvec(down, g, y);
    free(g);
    free(u);
}

/* View of record r inside the fixed-stride blob [Mference, ".gturbo
 * directory": 128 fixed-stride expert blobs per layer file, each sub-tensor
 * at its own offset]. */
static void record_mats(const oracle_layer *L, int r, oracle_qmat m[3])
{
    const uint8_t *rec = L->blob + (uint64_t)r * L->record_stride;
    const int D = L->d_model, I = L->d_expert;
    for (int j = 0; j < 3; ++j) {
        m[j].w = (const uint32_t *)(rec + L->off_w[j]);
        m[j].s = (const uint16_t *)(rec + L->off_s[j]);
        m[j].b = (const uint16_t *)(rec + L->off_b[j]);
        m[j].bits = 4;
        m[j].rows = (j == 2) ? D : I;
        m[j].cols = (j == 2) ? I : D;
    }
}

/* Record of expert e: the resident-set table when given [Mference, "Load and
 * ownership": a GPU-visible expert-to-slot table, Int16 per expert, -1 for
 * absent; slot n is the n-th fixed-stride blob], else record e.  -1 when the
 * expert is not resident. */
static int expert_record(const oracle_layer *L, int e)
{
    if (!L->expert_slot)
        return e;
    int r = L->expert_slot[e];
    return (r >= 0 && r < L->n_slots) ? r : -1;
}

/* RMSNorm of one fp32 vector with a BF16 weight vector [Mference, "Decode",
 * cb2 row: the layer tail applies the post-FFN norms].  READING: an RMSNorm
 * with weight, as the pre-norms of the same family; canonical order as
 * oracle_rmsnorm_bf16 (per group of 64 an fmaf chain of squares, groups
 * ascending, r = 1/sqrtf(ss/D + eps)); y_d = (y_d * r) * w_d in fp32. */
static void post_norm(float *y, int D, const uint16_t *w, float eps)
{
    float ss = 0.0f;
    for (int g = 0; g < D / 64; ++g) {
        float p = 0.0f;
        for (int i = 0; i < 64; ++i)
            p = fmaf(y[64 * g + i], y[64 * g + i], p);
        ss = ss + p;
    }
    float r = 1.0f / sqrtf(ss / (float)D + eps);
    for (int d = 0; d < D; ++d)
        y[d] = (y[d] * r) * oracle_bf16_to_f32(w[d]);
}

/* Gate of the shared branch [Mference, pinned families: "a gated shared
 * expert" (Qwen 3.6)].  READING: a learned vector g [D]; the gate is
 * sigmoid(g . x) per token, the dot product an fmaf chain in column order,
 * sigmoid(z) = 1 / (1 + expf(-z)). */
static float shared_gate_value(const uint16_t *g, const float *x, int D)
{
    float z = 0.0f;
    for (int i = 0; i < D; ++i)
        z = fmaf(oracle_bf16_to_f32(g[i]), x[i], z);
    return 1.0f / (1.0f + expf(-z));
}

/* The block on T tokens.
 *   router -> top-K -> softmax weights               [Mference, "Decode"]
 *   routed: sum_k w_k * expert_k(x)                   [Mference, "Metal execution"]
 *   shared: added without a routing weight            [Mference, "Why ... shape"]
 *   out = lambda * (shared + routed)                  [Mference, "Decode", cb2 row]
 * Optional parts (each absent unless given): the router reads
 * x * router_scale / sqrt(D) [Mference, "Decode", router formula, second
 * line; READING: router_scale is a vector over the model dimension, the
 * product (x_i * rs_i) * (1 / sqrtf(D)) in fp32 with no rounding to the
 * activation dtype]; the shared branch times its gate; the post-FFN norm of
 * the combined output before the layer scalar.  READING: the residual, when
 * given, is added in fp32 before the one rounding to the activation dtype. */
int oracle_block_forward(const oracle_layer *L, const void *x, int x_dtype, int T,
                         const void *residual, void *out,
                         int32_t *topk_idx, float *topk_w)
{
    const int D = L->d_model, E = L->n_experts, K = L->top_k;
    if (T < 0 || D % 64 || L->d_expert % 64 || K < 1 || K > E)
        return -1;
    float *xf = (float *)malloc(sizeof(float) * (size_t)T * D);
    float *xr = (float *)malloc(sizeof(float) * (size_t)T * D);
    float *logits = (float *)malloc(sizeof(float) * (size_t)T * E);
    float *sh = (float *)malloc(sizeof(float) * (size_t)D);
    float *y = (float *)malloc(sizeof(float) * (size_t)D);
    int rc = 0;
    for (long i = 0; i < (long)T * D; ++i)
        xf[i] = load_act(x, x_dtype, i);
    if (L->router_scale) {
        const float c = 1.0f / sqrtf((float)D);
        for (long i = 0; i < (long)T * D; ++i)
            xr[i] = (xf[i] * oracle_bf16_to_f32(L->router_scale[i % D])) * c;
    } else {
        memcpy(xr, xf, sizeof(float) * (size_t)T * D);
    }

    oracle_router_logits(&L->router, xr, T, logits);
    oracle_topk_softmax(logits, T, E, K, L->per_expert_scale, topk_idx, topk_w);

    for (int t = 0; t < T && rc == 0; ++t) {
        const float *xt = xf + (long)t * D;
        oracle_expert_ffn(&L->shared_gate, &L->shared_up, &L->shared_down, xt, sh);
        if (L->shared_expert_gate) {
            const float gv = shared_gate_value(L->shared_expert_gate, xt, D);
            for (int d = 0; d < D; ++d)
                sh[d] = gv * sh[d];
        }
        float *acc = sh; /* acc starts as the shared branch */
        for (int k = 0; k < K; ++k) {
            const int r = expert_record(L, topk_idx[(long)t * K + k]);
            if (r < 0) {
                rc = -2;
                break;
            }
            oracle_qmat m[3];
            record_mats(L, r, m);
            oracle_expert_ffn(&m[0], &m[1], &m[2], xt, y);
            float w = topk_w[(long)t * K + k];
            for (int d = 0; d < D; ++d)
                acc[d] = acc[d] + w * y[d];
        }
        if (L->post_norm)
            post_norm(acc, D, L->post_norm, L->post_eps);
        for (int d = 0; d < D; ++d) {
            float v = L->layer_scalar * acc[d];
            if (residual)
                v = load_act(residual, x_dtype, (long)t * D + d) + v;
            store_act(out, x_dtype, (long)t * D + d, v);
        }
    }
    free(xf);
    free(xr);
    free(logits);
    free(sh);
    free(y);
    return rc;
}

/* ------------------------------------------------------ RMSNorm and stack */

/* rmsnorm_no_scale [Mference, "Decode", router formula, first line].
 * READING: eps = caller's (1e-6 in the decode stack), no weight; canonical
 * order: per group of 64 a fmaf chain of squares, groups summed in ascending
 * order; r = 1/sqrtf(sum/D + eps) with IEEE division and square root; each
 * output rounded once to BF16. */
void oracle_rmsnorm_bf16(const uint16_t *x, int T, int D, float eps, uint16_t *y)
{
    for (int t = 0; t < T; ++t) {
        const uint16_t *xt = x + (long)t * D;
        float ss = 0.0f;
        for (int g = 0; g < D / 64; ++g) {
            float p = 0.0f;
            for (int i = 0; i < 64; ++i) {
                float v = oracle_bf16_to_f32(xt[64 * g + i]);
                p = fmaf(v, v, p);
            }
            ss = ss + p;
        }
        float r = 1.0f / sqrtf(ss / (float)D + eps);
        for (int i = 0; i < D; ++i)
            y[(long)t * D + i] = oracle_f32_to_bf16(oracle_bf16_to_f32(xt[i]) * r);
    }
}

/* Single-token decode through a stack of MoE blocks (attention omitted):
 * x <- bf16(x + block(rmsnorm(x))) per layer [Mference, "Decode" hidden-state
 * loop over 30 layers; residual and layer scalar in the layer tail]. */
int oracle_stack_forward(const oracle_layer *layers, int n_layers, uint16_t *x_io, int T, float eps,
                         uint16_t *xs_out, int32_t *topk_idx, float *topk_w)
{
    if (n_layers < 1 || T < 0)
        return -1;
    const int D = layers[0].d_model;
    uint16_t *xn = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * D);
    uint16_t *nx = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * D);
    int rc = 0;
    for (int l = 0; l < n_layers && rc == 0; ++l) {
        const int K = layers[l].top_k;
        oracle_rmsnorm_bf16(x_io, T, D, eps, xn);
        rc = oracle_block_forward(&layers[l], xn, 1, T, x_io, nx,
                                  topk_idx + (long)l * T * K, topk_w + (long)l * T * K);
        memcpy(x_io, nx, sizeof(uint16_t) * (size_t)T * D);
        if (xs_out)
            memcpy(xs_out + (long)l * T * D, nx, sizeof(uint16_t) * (size_t)T * D);
    }
    free(xn);
    free(nx);
    return rc;
}

/*
 * mx_oracle.h -- plain, slow, single-threaded CPU reference of the routed
 * Mixture-of-Experts FFN block over MLX-affine group-64 quantized weights.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference legs load this library.  It shares no code,
 * header, table or helper with the CUDA library; the two meet only through
 * the seeded input arrays the generator produces.
 *
 * What it follows ("Mference System design" page):
 *   - section "Why the runtime has this shape": 128 routed experts, top-8 per
 *     token; a dense shared expert added without a routing weight; MLX affine
 *     quantization with a BF16 scale and BF16 bias per group of 64 weights;
 *     an 8-bit router and 4-bit shared / routed experts; parallel shared and
 *     routed FFNs and a learned layer scalar;
 *   - section "Decode": the router formula (rmsnorm, int8 affine projection,
 *     highest-8, softmax over the selected logits times a per-expert scale);
 *   - section "Metal execution": affine decode + GeGLU + weighted expert
 *     reduction.
 * Precision ("TinyTitan_Datacenter Architecture" page, section "Invariants",
 * item 1): fp32 accumulation in a fixed reduction order.  Every multiply-add
 * the definition contains is an explicit IEEE fmaf; the file must be built
 * with -ffp-contract=off so the compiler adds no contraction of its own.
 *
 * Quantized matrix W [rows, cols]: row-major; groups of 64 run along cols
 * (the input dimension).  4-bit: uint32 [rows][cols/8], element c in word c/8
 * at bits 4*(c%8) (low nibble first).  8-bit: uint32 [rows][cols/4], element
 * c in word c/4 at bits 8*(c%4) (low byte first).  scales, biases: BF16 bit
 * patterns [rows][cols/64].  Dequantized value w = s*q + b.
 *
 * Parity: every function here is pinned by the CPU tests (tests/test_oracle_*)
 * against closed forms, brute force, invariants and the by-hand example in
 * tests/golden; none is "parity unpinned".
 */
#ifndef MX_ORACLE_H
#define MX_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One quantized matrix as host pointers. */
typedef struct {
    const uint32_t *w;      /* packed values                      */
    const uint16_t *s;      /* BF16 scales  [rows][cols/64]       */
    const uint16_t *b;      /* BF16 biases  [rows][cols/64]       */
    int32_t rows, cols, bits;
} oracle_qmat;

/* One MoE block: router, shared expert, and a blob of n_experts fixed-stride
 * records, each holding gate [I,D], up [I,D] and down [D,I] 4-bit matrices at
 * the given byte offsets ("packed_experts" layout of the .gturbo directory). */
typedef struct {
    int32_t d_model, d_expert, n_experts, top_k;
    float layer_scalar;
    oracle_qmat router;                          /* bits 8, [E, D]       */
    oracle_qmat shared_gate, shared_up, shared_down; /* [S,D] [S,D] [D,S] */
    const uint8_t *blob;
    uint64_t record_stride;
    uint64_t off_w[3], off_s[3], off_b[3];       /* gate, up, down        */
    const float *per_expert_scale;               /* NULL = all ones       */
    /* Optional parts of the layer (each NULL = absent):
     *   expert_slot   [E]: record of expert e in the blob is expert_slot[e]
     *                 (-1 = not resident), n_slots records; NULL = record e;
     *   router_scale  BF16 [D]: the router reads x * router_scale / sqrt(D);
     *   post_norm     BF16 [D]: the FFN output y becomes rmsnorm(y) * post_norm
     *                 (eps post_eps) before the layer scalar and residual;
     *   shared_expert_gate  BF16 [D]: the shared branch is scaled per token
     *                 by sigmoid(shared_expert_gate . x). */
    const int16_t *expert_slot;
    int32_t n_slots;
    const uint16_t *router_scale;
    const uint16_t *post_norm;
    float post_eps;
    const uint16_t *shared_expert_gate;
} oracle_layer;

/* Activation dtypes: 0 = fp32, 1 = bf16 (uint16 bit patterns). */

float    oracle_bf16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16(float f);          /* round to nearest even */
float    oracle_gelu(float z);                 /* tanh form             */

/* y[r] = sum_c (s*q + b)[r,c] * x[c]  (4- or 8-bit matrix, fp32 x). */
void oracle_qmatvec(const oracle_qmat *m, const float *x, float *y);

/* Router logits in the canonical order (see mx_oracle.c). x: fp32 [T][D]. */
void oracle_router_logits(const oracle_qmat *router, const float *x, int T, float *logits);

/* Top-K by (logit desc, index asc) and softmax over the selected logits.
 * NaN logits rank as -inf.  Returns 0, or -1 on bad arguments. */
int oracle_topk_softmax(const float *logits, int T, int E, int K,
                        const float *per_expert_scale, int32_t *topk_idx, float *topk_w);

/* counts[E], offsets[E+1] (exclusive scan), perm[T*K]: slot ids s = t*K + k
 * sorted by expert, ties in ascending s. */
int oracle_permute(const int32_t *topk_idx, int T, int K, int E,
                   int32_t *counts, int32_t *offsets, int32_t *perm);

/* Gated expert FFN on one token: y = W_down (gelu(W_gate x) * (W_up x)). */
void oracle_expert_ffn(const oracle_qmat *gate, const oracle_qmat *up, const oracle_qmat *down,
                       const float *x, float *y);

/* The block: out[t] = residual[t] + lambda * (shared(x_t) + sum_k w_k * expert_k(x_t)),
 * rounded to the activation dtype (with the optional parts of the layer as
 * above).  residual may be NULL.  Returns 0, -1 on bad arguments, or -2 if a
 * selected expert is not resident in the blob (expert_slot). */
int oracle_block_forward(const oracle_layer *L, const void *x, int x_dtype, int T,
                         const void *residual, void *out,
                         int32_t *topk_idx, float *topk_w);

/* Canonical RMSNorm without weight: y = x / sqrt(mean(x^2) + eps), x and y BF16. */
void oracle_rmsnorm_bf16(const uint16_t *x, int T, int D, float eps, uint16_t *y);

/* Decode stack: for each layer, x <- bf16(x + block(rmsnorm(x))).  x_io is
 * BF16 [T][D], updated in place; xs_out (nullable) receives every layer's
 * output [n_layers][T][D]; topk_idx/topk_w are [n_layers][T][K]. */
int oracle_stack_forward(const oracle_layer *layers, int n_layers, uint16_t *x_io, int T, float eps,
                         uint16_t *xs_out, int32_t *topk_idx, float *topk_w);

#ifdef __cplusplus
}
#endif
#endif /* MX_ORACLE_H */

/*
 * mx_moe.h -- C ABI of the GB300 (sm_103a) routed Mixture-of-Experts FFN block
 * over MLX-affine group-64 quantized weights.
 *
 * The block ("Mference System design" page):
 *   - section "Why the runtime has this shape": each layer has 128 routed
 *     experts, the router selects 8 per token; a dense shared expert is a
 *     separate branch whose output is added without a routing weight; MLX
 *     affine quantization, packed 4-bit values with a BF16 scale and BF16 bias
 *     per group of 64 weights; 8-bit router, 4-bit shared and routed experts;
 *     parallel shared and routed FFNs and a learned layer scalar;
 *   - section "Decode": logits = int8_affine(x); top8 = highest_8(logits);
 *     weights = softmax(logits[top8]) * per_expert_scale[top8];
 *   - section "Metal execution": routed kernels fuse affine decode, GeGLU and
 *     the weighted expert reduction;
 *   - section "The .gturbo directory": one fixed-stride, page-aligned record
 *     per routed expert, each sub-tensor at its own offset; invalid alignment
 *     and unknown format flags are rejected.
 *
 * Per token t:
 *   out[t] = residual[t] + layer_scalar * ( shared(x_t) + sum_k w[t,k] * expert_{idx[t,k]}(x_t) )
 *   expert(x) = W_down ( gelu_tanh(W_gate x) * (W_up x) )
 * with residual = 0 unless given (mx_moe_options), and x optionally replaced by
 * rmsnorm_no_scale(x) rounded to the activation dtype (mx_moe_options).
 *
 * Quantized matrix W [rows, cols] (row-major, groups of 64 along cols, the
 * input dimension):
 *   4-bit: uint32 [rows][cols/8], element c in word c/8 at bits 4*(c%8);
 *   8-bit: uint32 [rows][cols/4], element c in word c/4 at bits 8*(c%4);
 *   scales, biases: BF16 [rows][cols/64]; w[r,c] = s[r,c/64]*q[r,c] + b[r,c/64].
 *
 * Top-k order: descending logit, ties to the lower expert index; NaN logits
 * rank as -inf and enter the softmax as -inf (weight 0).  Routing logits are computed in a fixed fp32 order (per group
 * of 64: P = fma chain of q*x, X = add chain of x; then per group, ascending,
 * acc = fma(s, P, acc), acc = fma(b, X, acc)) so the top-k choice is
 * reproducible bit for bit.
 *
 * Ownership: the caller owns every buffer (inputs, weights, outputs,
 * workspace).  All pointers named "device" are CUDA device pointers; host
 * structs are read only during the call.  Calls are asynchronous on the given
 * stream; outputs are valid after the stream is synchronised.
 * Errors: every argument is validated on the host before anything is
 * launched; on an error nothing is written and the call returns a negative
 * mx_status (mx_last_error_string() gives the reason, per calling thread).
 */
#ifndef MX_MOE_H
#define MX_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MX_API __attribute__((visibility("default")))
#else
#define MX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MX_OK = 0,
    MX_ERR_INVALID_ARG = -1,    /* null pointer, bad size, bad dtype, bad magic/version */
    MX_ERR_ALIGNMENT = -2,      /* pointer, offset or stride misaligned                */
    MX_ERR_UNSUPPORTED = -3,    /* valid but unsupported shape / bit width / group     */
    MX_ERR_WORKSPACE = -4,      /* workspace too small or could not be allocated       */
    MX_ERR_CUDA = -5,           /* a CUDA runtime call failed                          */
    MX_ERR_DEVICE_TIMEOUT = -6, /* a device-side bounded wait gave up                  */
    MX_ERR_RANGE = -7,          /* a device-side range check failed (see below)        */
    MX_ERR_NOT_RESIDENT = -8    /* a selected expert has no record in the blob          */
} mx_status;

typedef enum { MX_F32 = 0, MX_BF16 = 1 } mx_dtype;

/* One quantized matrix (device pointers; each 16-byte aligned). */
typedef struct {
    const void *w;          /* packed uint32 words                   */
    const void *scales;     /* BF16 [rows][cols/64]                  */
    const void *biases;     /* BF16 [rows][cols/64]                  */
    int32_t rows, cols, bits;
} mx_qlinear;

/* The dense shared expert: gate [S,D], up [S,D], down [D,S], 4-bit. */
typedef struct {
    mx_qlinear gate, up, down;
} mx_ffn;

/* Byte offsets of one sub-tensor's packed words, scales and biases inside an
 * expert record. */
typedef struct {
    uint64_t w, s, b;
} mx_sub;

#define MX_MOE_LAYOUT_MAGIC 0x4D584D45u /* "EMXM" little-endian */
#define MX_MOE_LAYOUT_VERSION 3u /* version 1 (ending at per_expert_scale) and 2 (ending at
                                    shared_expert_gate) layouts are accepted too */

/* Layout of one layer's expert blob: n_experts records of record_stride bytes
 * (n_slots records when expert_slot is given).  Record r holds gate [d_expert,
 * d_model], up [d_expert, d_model] and down [d_model, d_expert] matrices
 * (4-bit) at the offsets given.  d_shared is the intermediate width of the
 * layer's shared expert (mx_ffn).
 *
 * Version 2 adds optional parts of the layer, each absent when NULL:
 *   expert_slot   a resident-set table ("Mference System design", section
 *                 "Load and ownership": a GPU-visible expert-to-slot table,
 *                 Int16 per expert, -1 for absent): device int16 [E]; expert
 *                 e's weights are record expert_slot[e] of a blob of n_slots
 *                 records.  A selected expert with no record (-1, or outside
 *                 [0, n_slots)) contributes nothing and the call's error word
 *                 reports it (mx_moe_workspace_check: MX_ERR_NOT_RESIDENT);
 *                 the call's outputs are then not the block's.
 *   router_scale  device BF16 [D]: the router reads x * router_scale / sqrt(D)
 *                 (section "Decode", router formula), each element
 *                 (x_i * router_scale_i) * (1/sqrtf(D)) in fp32; the experts
 *                 still read x.
 *   post_norm     device BF16 [D]: the combined output y = shared + sum_k w_k
 *                 y_k becomes rmsnorm(y) * post_norm before the layer scalar
 *                 and the residual (section "Decode", cb2 row: the post-FFN
 *                 norms), eps post_eps; canonical order as pre_rmsnorm.
 *   shared_expert_gate  device BF16 [D]: the shared branch is scaled per token
 *                 by sigmoid(shared_expert_gate . x) (the page's gated shared
 *                 expert of the Qwen family).
 * router_scale, post_norm and shared_expert_gate are supported by the
 * single-launch decode path (T <= 4) and the grouped-GEMM path (BF16, T > 4);
 * calls that would run the multi-launch decode kernels (fp32 with T > 4, or
 * those paths forced by MX_MOE_SINGLE_LAUNCH=0 / MX_MOE_PREFILL_GEMM=0)
 * return MX_ERR_UNSUPPORTED for them.  expert_slot works on every path.
 *
 * Version 3 adds one optional field, a derived copy of weights already in the
 * layer (so the results do not depend on it):
 *   down_sb       device uint32, 16-byte aligned, nullable: the down
 *                 projections' scale and bias pairs written by
 *                 mx_moe_pack_down_sb for this layout, blob and shared expert,
 *                 one word per (row, group) = scale bits | bias bits << 16,
 *                 column-major: record r, group g, row d at (r * (I/64) + g) *
 *                 D + d for the n records of the blob (n_slots with an
 *                 expert_slot table, else n_experts), then the shared expert's
 *                 group g, row d at n * (I/64) * D + g * D + d.  The group of
 *                 one 64-wide slice of a down projection is then D contiguous
 *                 words, which the single-launch decode path copies in blocks
 *                 instead of gathering 2 D strided 2-byte values per slice;
 *                 the other paths do not read it.  It must be re-packed
 *                 whenever the down scales or biases it was made from change. */
typedef struct {
    uint32_t magic;              /* MX_MOE_LAYOUT_MAGIC                          */
    uint32_t version;            /* MX_MOE_LAYOUT_VERSION                        */
    int32_t d_model;             /* D, multiple of 64                            */
    int32_t d_expert;            /* I, multiple of 64                            */
    int32_t n_experts;           /* E, 1 <= E <= 512                             */
    int32_t top_k;               /* K, 1 <= K <= min(E, 32)                      */
    int32_t d_shared;            /* S, shared-expert width, multiple of 64       */
    int32_t group;               /* 64                                           */
    int32_t bits;                /* 4                                            */
    uint64_t record_stride;      /* bytes, multiple of 4096                      */
    mx_sub gate, up, down;       /* offsets: 16-byte aligned, inside the stride */
    int32_t act_dtype;           /* mx_dtype of x, out and residual              */
    float layer_scalar;          /* lambda                                       */
    const float *per_expert_scale; /* device [E], nullable = all ones            */
    /* version 2 and later */
    const int16_t *expert_slot;  /* device [E], nullable (see above)             */
    int32_t n_slots;             /* records in the blob when expert_slot is set  */
    const uint16_t *router_scale;  /* device BF16 [D], 16-byte aligned, nullable */
    const uint16_t *post_norm;     /* device BF16 [D], 16-byte aligned, nullable */
    float post_eps;                /* eps of post_norm                           */
    const uint16_t *shared_expert_gate; /* device BF16 [D], 16-byte aligned, nullable */
    /* version 3 and later */
    const uint32_t *down_sb;     /* device, 16-byte aligned, nullable (see above)  */
} mx_moe_layout;

/* Per-call options (all optional; pass NULL for the plain block). */
typedef struct {
    const void *residual;        /* device [T][D] act dtype, nullable: out = residual + block  */
    int32_t pre_rmsnorm;         /* 1: the block reads rmsnorm_no_scale(x) rounded to the act
                                    dtype (canonical order: per group of 64 an fma chain of
                                    squares, groups summed ascending, r = 1/sqrtf(ss/D + eps)) */
    float rms_eps;               /* epsilon of pre_rmsnorm                                      */
} mx_moe_options;

/*
 * The block, as in the pages' "Decode"/"Prefill" sections: router GEMV, top-k,
 * softmax, routed gated experts, shared expert, weighted combine, layer scalar.
 *   x          device [T][D], act dtype (layout->act_dtype), 16-byte aligned
 *   T          tokens, >= 1
 *   router     8-bit [E, D]
 *   shared     4-bit gate/up [S, D], down [D, S]
 *   expert_blob device, E * record_stride bytes, 256-byte aligned
 *   out        device [T][D] act dtype (may not alias x)
 *   topk_idx   device int32 [T][K]
 *   topk_w     device fp32  [T][K]
 * Runs on the legacy default stream with a workspace the library allocates
 * and keeps (grown on demand; freed at process exit).  Not for use under CUDA
 * graph capture; use mx_moe_layer_forward_ex there.
 */
MX_API mx_status mx_moe_layer_forward(const void *x, int T, const mx_qlinear *router, const mx_ffn *shared,
                               const void *expert_blob, const mx_moe_layout *layout,
                               void *out, int32_t *topk_idx, float *topk_w);

/*
 * Same block with explicit options, stream and workspace.
 *   opt        nullable
 *   stream     cudaStream_t (NULL = legacy default stream)
 *   ws         device workspace of ws_bytes >= mx_moe_workspace_bytes(layout, T),
 *              256-byte aligned, zero-filled before its first use (see
 *              mx_moe_workspace_init); every call leaves it ready for the next.
 * Allocates nothing.  Calls sharing one workspace must be ordered on the GPU
 * (same stream, or explicit events).
 */
MX_API mx_status mx_moe_layer_forward_ex(const void *x, int T, const mx_qlinear *router, const mx_ffn *shared,
                                  const void *expert_blob, const mx_moe_layout *layout,
                                  void *out, int32_t *topk_idx, float *topk_w,
                                  const mx_moe_options *opt, void *stream, void *ws, size_t ws_bytes);

/* Workspace bytes for up to T_max tokens of this layout (0 on invalid layout). */
MX_API size_t mx_moe_workspace_bytes(const mx_moe_layout *layout, int T_max);

/* Zero-fill a workspace on the stream (cudaMemsetAsync); call once after allocating it. */
MX_API mx_status mx_moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * Device-side error word of a workspace.  Kernels that wait on asynchronous
 * copies give up after a bounded time, record it in the workspace's first word
 * and skip their math; this call synchronises on `stream`, reads the word, and
 * returns MX_ERR_DEVICE_TIMEOUT if a wait gave up, MX_ERR_NOT_RESIDENT if a
 * selected expert had no record in the blob (layout expert_slot),
 * MX_ERR_RANGE if a range check failed, MX_OK otherwise.  The word stays set until the workspace is
 * re-initialised (mx_moe_workspace_init).
 *
 * Range of the single-launch decode path (T <= 4): its down projections are
 * summed over the grid in 64-bit fixed point, so that the sum does not depend
 * on the order of the additions.  With E = floor(log2(max |x|)) over the
 * layer's tokens (x as the block reads it, after the optional rmsnorm), every
 * partial sum v -- one expert slice's contribution to one output element,
 * before the layer scalar -- is scaled by f = 2^(4 - 2E) (clamped to
 * 2^[-100, 100]) and kept to 32 fractional bits at that scale: the absolute
 * resolution is 2^-32 / f, about 2^-32 |y| / |x|^2.  A partial with
 * |v f| >= 2^23 is left out of the sum and sets MX_ERR_RANGE.  For inputs of
 * magnitude 4..8 (f = 1) that is |v| < 8.4e6 at a resolution of 2.3e-10.
 * The other paths accumulate in fp32 and have no such limit.
 */
MX_API mx_status mx_moe_workspace_check(const void *ws, void *stream);

/*
 * The block for 1 <= T <= 4 tokens with no workspace argument and no
 * allocation: the single-launch decode kernel with its scratch (error word,
 * counters, logits, fixed-point sums) in one device array of this library,
 * MX_STATIC_SCRATCH_BYTES long.  The pages have no counterpart to this call;
 * it exists for callers that may not allocate at all while they run -- a
 * serving loop whose device memory is budgeted and owned up front, or code
 * on a path where an allocation's implicit synchronisation or failure under
 * memory pressure is not acceptable -- and that have no workspace to pass.
 *   arguments as mx_moe_layer_forward_ex (opt nullable; stream: cudaStream_t,
 *   NULL = legacy default stream), without ws / ws_bytes.
 * Limits (else MX_ERR_UNSUPPORTED, nothing launched): T <= 4, d_model <= 4096,
 * n_experts <= 256, and the single-launch path usable on this device (its
 * shared-memory plan fits; not disabled by MX_MOE_SINGLE_LAUNCH=0).
 * The first call on each device resolves the array's address
 * (cudaGetSymbolAddress); make that first call outside any stream capture.
 * Every call clears the scratch it uses (cudaMemsetAsync on `stream`) before
 * the kernel.  A call that succeeds (with the stage profiler off) makes no
 * allocation of its own, host or device: no cudaMalloc, cudaFree or malloc,
 * and no thread-local storage (whose first use on a host thread would be
 * allocated lazily); the kernel parameters sit in one static block guarded by
 * a lock, so concurrent host calls serialise on it.  The CUDA runtime itself
 * may load the kernel's code on the first launch on a device, as for any
 * kernel.  A call that fails records its message in the calling thread's
 * message buffer (mx_last_error_string), which that thread's first error may
 * allocate.  There is one scratch
 * array per device: calls that may overlap on the GPU (other streams, other
 * host threads) race on it and must be ordered by the caller.  A device-side
 * wait that gives up is not reported (use mx_moe_layer_forward_ex and
 * mx_moe_workspace_check where that matters).
 */
#define MX_STATIC_SCRATCH_BYTES (144u * 1024u)
MX_API mx_status mx_moe_layer_forward_static(const void *x, int T, const mx_qlinear *router, const mx_ffn *shared,
                                      const void *expert_blob, const mx_moe_layout *layout,
                                      void *out, int32_t *topk_idx, float *topk_w,
                                      const mx_moe_options *opt, void *stream);

/*
 * Routing alone (router GEMV + top-k + softmax + grouping), for exact checks.
 *   topk_idx  device int32 [T][K];  topk_w device fp32 [T][K]
 *   counts    device int32 [E]      tokens per expert
 *   offsets   device int32 [E+1]    exclusive scan of counts
 *   perm      device int32 [T*K]    slot ids s = t*K + k grouped by expert,
 *                                   ascending s within an expert
 *   logits    device fp32 [T][E], nullable: the router logits
 * Grouping follows the "Prefill" section ("groups token/expert pairs into
 * bounded routed-MoE work").  opt may request pre_rmsnorm; residual is ignored.
 * A layout with router_scale returns MX_ERR_UNSUPPORTED here (the block entry
 * points apply it).
 */
MX_API mx_status mx_moe_route(const void *x, int T, const mx_qlinear *router, const mx_moe_layout *layout,
                       int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *offsets,
                       int32_t *perm, float *logits, const mx_moe_options *opt,
                       void *stream, void *ws, size_t ws_bytes);

/*
 * Decode stack without attention: for l in 0..n_layers-1,
 *   x <- round_act(x + block_l(rmsnorm_no_scale(x)))
 * i.e. the block with pre_rmsnorm (eps) and residual = x, ping-ponging between
 * x_io and an internal buffer of the workspace; the final x is written back to
 * x_io.  All per-layer arrays have n_layers entries.
 *   x_io      device [T][D] act dtype (BF16 or fp32), updated in place
 *   topk_idx  device int32 [n_layers][T][K], topk_w device fp32 [n_layers][T][K]
 *   ws        >= mx_moe_stack_workspace_bytes(layouts[0], T), prepared by
 *             mx_moe_workspace_init
 * Every layer must share D, I, E, K, dtype and the shared-expert shape.
 * Allocates nothing; safe to capture into a CUDA graph.
 */
MX_API mx_status mx_moe_stack_forward(void *x_io, int T, int n_layers, const mx_qlinear *routers,
                               const mx_ffn *shareds, const void *const *expert_blobs,
                               const mx_moe_layout *layouts, int32_t *topk_idx, float *topk_w,
                               float rms_eps, void *stream, void *ws, size_t ws_bytes);

MX_API size_t mx_moe_stack_workspace_bytes(const mx_moe_layout *layout, int T);

/*
 * Packed down-projection scale and bias words (layout field down_sb, version
 * 3; format above).  mx_moe_down_sb_bytes returns the size of the table for
 * `layout` (0 if the layout is invalid).  mx_moe_pack_down_sb writes it:
 *   layout       a valid layout (its own down_sb is not read)
 *   blob         device expert blob of that layout
 *   shared_down  the layer's shared down projection [D][S] (its scales and
 *                biases are read)
 *   out          device, 16-byte aligned, mx_moe_down_sb_bytes(layout) bytes,
 *                owned by the caller, not overlapping the blob
 *   stream       CUDA stream (NULL = the legacy default stream); the copy is
 *                asynchronous on it
 * Errors: MX_ERR_INVALID_ARG for null pointers or a bad layout, MX_ERR_ALIGNMENT
 * for a misaligned `out`, MX_ERR_CUDA if the launch fails.  A table is a pure
 * rearrangement of BF16 values the blob already holds (no arithmetic).
 */
MX_API size_t mx_moe_down_sb_bytes(const mx_moe_layout *layout);
MX_API mx_status mx_moe_pack_down_sb(const mx_moe_layout *layout, const void *blob, const mx_qlinear *shared_down,
                                     uint32_t *out, void *stream);

/*
 * Per-stage timing, after the stage-timing profiler of the gem "Native
 * architecture" page (section "profiling": stage-boundary timestamps sampled
 * without changing the ordinary route).  While enabled, every block call
 * records a CUDA event pair around each of its kernels on the call's own
 * stream.  Stages: 0 = routing (router GEMV + top-k + grouping), 1 = gate/up +
 * GeGLU, 2 = down + combine.  The single-launch decode path (T <= 4) records
 * its one launch as stage 1; the grouped-GEMM path (T > 4, BF16) records its
 * gate/up GEMM as stage 1 and its down GEMM + combine as stage 2 (the token
 * gather between routing and gate/up is not timed).  mx_moe_profile_read synchronises on the recorded
 * events and returns, per stage, the summed milliseconds and the number of
 * launches (arrays of MX_PROFILE_STAGES), then clears them if reset != 0.
 * Not for use under CUDA graph capture; off by default; process-wide.
 */
#define MX_PROFILE_STAGES 3
MX_API mx_status mx_moe_profile_enable(int on);
MX_API mx_status mx_moe_profile_read(double *ms, int *launches, int reset);

/* Human-readable status and the last error of the calling thread. */
MX_API const char *mx_status_string(mx_status s);
MX_API const char *mx_last_error_string(void);

/* Library version "major.minor.patch". */
MX_API const char *mx_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MX_MOE_H */

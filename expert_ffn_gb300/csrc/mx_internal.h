// mx_internal.h -- kernel argument blocks and launchers shared by the
// library's translation units (host side).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mx {

// Tokens per FFN work tile of the decode path (one expert's tokens per tile).
constexpr int kTileTokens = 64;
// Largest T one pass of the decode path handles; longer inputs run in chunks.
constexpr int kDecodeChunk = 64;
// BF16 calls with more tokens than this run the grouped tensor-core GEMMs
// (each expert's weights dequantized once per tile of up to 160 of its tokens).
constexpr int kPrefillAbove = 4;
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;
constexpr int kMaxDim = 16384;

struct RouteArgs {
    const void *x;          // [T][D] act dtype
    int x_dtype;            // 0 fp32, 1 bf16
    int T, D, E, K;
    const uint32_t *rw;     // router packed bytes [E][D/4]
    const uint16_t *rs;     // router scales [E][D/64]
    const uint16_t *rb;     // router biases [E][D/64]
    int pre_norm;
    float eps;
    const float *pes;       // per-expert scale, nullable
    int32_t *topk_idx;      // [T][K]
    float *topk_w;          // [T][K]
    float *logits;          // [T][E]
    int32_t *counts;        // [E]
    int32_t *offsets;       // [E+1]
    int32_t *perm;          // [T*K]
    int32_t *tiles;         // [3][n] (expert, begin, end) triples, nullable
    int32_t *n_tiles;       // nullable
    unsigned *tickets;      // [n_token_tiles + 1], zero on entry, zero on exit
    uint16_t *xp;           // FFN operand: [nsplit][T][D] bf16 in operand column order, nullable
    int nsplit;             // 1 (bf16 activations) or 3 (fp32 activations)
    float *xg;              // FFN operand: [T][D/64] per-group sums of x (with xp)
    int ET, GC;             // experts per CTA, groups per chunk
    int logits_only;        // 1: stop after the logits
    int cluster;            // 1: one thread-block cluster; CTA 0 gathers the logits and routes
    unsigned *err;          // device error word (bounded waits that gave up)
    // large router only: its input is x * router_scale * rcoef (XG then holds
    // the group sums of that product); nullable
    const uint16_t *router_scale;
    float rcoef;            // 1 / sqrtf(D), computed on the host
};

// Optional parts of a layer (layout version 2; all absent for version 1).
struct LayerExt {
    const int16_t *slot;         // resident-set table [E], nullable
    int n_slots;                 // records in the blob (E without a table)
    const uint16_t *router_scale, *post_norm, *shared_gate;  // BF16 [D], nullable
    float post_eps;
    float rcoef;                 // 1 / sqrtf(D) (host-rounded, as the oracle's)
    const uint32_t *down_sb;     // packed down (scale | bias << 16) words, nullable
};

struct FfnArgs {
    int T, D, I, S, E, K;
    const int16_t *slot;                    // resident-set table, nullable
    int n_slots;                            // records in the blob
    const uint8_t *blob;
    uint64_t stride;
    uint64_t off_w[3], off_s[3], off_b[3];  // gate, up, down inside a record
    const uint32_t *sw[3];                  // shared gate, up, down packed words
    const uint16_t *ss[3];
    const uint16_t *sb[3];
    const uint16_t *xp;                     // [nsplit][T][D] x operand (operand column order)
    int nsplit;
    const float *xg;                        // [T][D/64] per-group sums of x
    const float *logits;                    // [T][E] router logits
    const float *pes;                       // per-expert scale, nullable
    const int32_t *topk_idx;                // [T][K] routing (written by the router kernel)
    const float *topk_w;                    // [T][K]
    const int32_t *perm;                    // [T*K] slots grouped by expert
    const int32_t *tiles;                   // [3][n] (expert, begin, end)
    const int32_t *n_tiles;
    uint16_t *hr[2];                        // routed hidden, hi/lo [T*K][I]
    uint16_t *hs[2];                        // shared hidden, hi/lo [T][S]
    const void *residual;                   // nullable
    void *out;
    int act_dtype;
    float lam;
    unsigned *err;                          // device error word
};

// Shapes of the weight-streaming kernels (host-computed; byte offsets into
// dynamic shared memory).
struct GuLaunch {
    int stages, slot_bytes, n_shared, tpt, max_tiles;
    int off_meta, off_xs, off_xg, off_ring, off_part;
};
struct DnLaunch {
    int stages, slot_bytes, max_tiles;
    int off_meta, off_ring, off_acc;
};

// TMA tensor maps of one layer's expert weights (mx_tma.cu): routed gate, up,
// down over all experts of the blob, and the shared expert's three matrices.
struct FfnMaps {
    CUtensorMap gate, up, down, sgate, sup, sdown;
    CUtensorMap down1, sdown1;  // down projections, D/16 rows x one 64-column group (single-launch path)
};
cudaError_t get_ffn_maps(const FfnArgs &a, FfnMaps *out);

// Launch configuration of the routing kernel for T tokens.
struct RouteLaunch {
    int TT, ET, GC, n_tt, n_et;
    int cluster;            // cluster mode (T <= kClusterTokens): n_et CTAs form one cluster
    size_t off_gather;      // cluster mode: byte offset of the gathered logits [T][E]
    size_t off_route;       // cluster mode: byte offset of the routing scratch
    size_t smem;
};
constexpr int kClusterTokens = 8;
constexpr int kClusterCtas = 8;
RouteLaunch route_plan(int T, int D, int E, int K);
cudaError_t launch_route(const RouteArgs &a, const RouteLaunch &L, cudaStream_t s);

// Decode-path FFN: gate/up + GeGLU, then down + combine.  The two launches are
// bracketed by prof_begin/prof_end (no-ops unless stage profiling is on).
cudaError_t launch_ffn_decode(const FfnArgs &a, int max_tiles, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------
// Single-launch decode path (mx_decode.cu): the block, or a stack of blocks,
// for T <= kPdMaxT tokens in one persistent cooperative kernel.
constexpr int kPdMaxT = 4;
constexpr int kPdMaxLayers = 30;  // layers per launch (the layer table is a kernel parameter)
constexpr int kPdMaxD = 4096;     // d_model limit of the path (down-slice copies of D/16 rows)

// Byte offsets into the kernel's dynamic shared memory.
struct PdSmem {
    int NR, slot;  // ring depth and slot bytes
    int ring, xraw, xq, xg, xpl, uh, upl, dss, lg, rt, pr, misc, zero;
    int total;
};

// One layer: TMA maps of its routed (over all experts of the blob) and shared
// matrices (the down maps in slices of D/16 rows x one 64-column group), its
// router, the s/b offsets of the expert records, its outputs.
struct PdLayer {
    CUtensorMap gate, up, down, sgate, sup, sdown;
    const uint32_t *rw;
    const uint16_t *rs, *rb;
    const uint8_t *blob;
    uint64_t stride;
    uint32_t off_s[3], off_b[3];  // s / b offsets in a record (the path requires < 2^32)
    const uint16_t *ss[3], *sb[3];
    const uint32_t *dsb, *dsb_s;  // packed down (scale | bias << 16) words: records, shared (nullable)
    const float *pes;
    int32_t *topk_idx;
    float *topk_w;
    const void *x_in;      // the launch's first layer: its input x
    void *x_out;           // nullable: where this layer's output goes (else it stays on chip)
    const void *residual;  // res_mode 2
    float lam;
    int res_mode;          // 0 none, 1 the layer's input x, 2 `residual`
    // optional parts (LayerExt): resident-set table, router input scale,
    // post-FFN norm weight, shared-branch gate
    const int16_t *slot;
    int n_slots;
    const uint16_t *router_scale, *post_norm, *shared_gate;
    float post_eps, rcoef;
};

struct PdParams {
    int T, D, I, S, E, K, n_layers, act, pre_norm, n_cta;
    float eps;
    unsigned *err;         // workspace error word
    int *ctr;              // [n_layers][cstride] counters, then done, abort (zero on entry)
    int cstride;           // 3 + E
    float *logits;         // [T][E]
    long long *ybuf;       // [n_layers][T][D] fixed-point sums of the down projections
    unsigned long long wait_ns;  // bound of every wait on another CTA
    int hold_cta;          // -1, or a CTA that does not arrive at the first logit exchange
    PdSmem sm;
    PdLayer L[kPdMaxLayers];
};
static_assert(sizeof(PdParams) <= 32764, "the layer table must fit the kernel parameter space");

bool pd_plan(int T, int D, int I, int S, int E, int K, int act, int n_cta, int smem_max, PdSmem *out);
size_t pd_ctr_ints(int E, int n_layers);
cudaError_t launch_pd(const PdParams &p, cudaStream_t s);

// ---------------------------------------------------------------------------
// Prefill path (mx_prefill.cu): T > kPrefillAbove tokens with BF16 activations;
// grouped GEMMs on tcgen05 tensor cores.

// Arguments of the grouped-GEMM kernel (one per launch: gate/up or down).
struct PfArgs {
    int mode;               // 0 gate/up, 1 down
    int T, D, I, S, E, K;
    int FT, FTs;            // weight-row tiles: routed, shared
    int KT, KTs;            // K tiles of 64 columns: routed, shared
    int GK, GK_s;           // scale groups per weight row: routed, shared
    int rows, rows_s;       // weight rows: routed, shared
    const int32_t *tt_off;  // [E+1] per-expert token-tile offsets
    const int32_t *counts, *offsets, *perm;
    const float *xsc;       // [T] 2^-k of each token's FP16 scale
    const uint8_t *blob;
    uint64_t stride;
    const int16_t *slot;    // resident-set table, nullable
    int n_slots;            // records in the blob
    uint64_t off_s[3], off_b[3];
    const uint16_t *ss[3], *sb[3];
    void *H, *Hs;           // FP16 [T*K][I], [T][S] (operand column order)
    float *Y, *Ys;          // fp32 [T*K][D], [T][D]
    unsigned *err;
    CUtensorMap wa, wb;     // routed packed weights (gate, up) or (down, -)
    CUtensorMap swa, swb;   // shared packed weights
    CUtensorMap xr, xs;     // FP16 operand rows: routed slots, shared tokens
};

// One prefill call, after the router has written counts/offsets/perm/topk.
struct PfCall {
    const void *x;          // BF16 [T][D]
    int T, D, I, S, E, K;
    int pre_norm;
    float eps;
    const int32_t *perm, *counts, *offsets;
    const float *topk_w;
    const uint8_t *blob;
    uint64_t stride;
    uint64_t off_w[3], off_s[3], off_b[3];
    const uint32_t *sw[3];
    const uint16_t *ss[3], *sb[3];
    float lam;
    const void *residual;   // BF16, nullable
    void *out;              // BF16 [T][D]
    unsigned *err;
    uint8_t *ws;            // pf_workspace_bytes(...)
    int n_cta;
    LayerExt ext;           // optional parts of the layer
};

// Buffers the router reads on the prefill path: FP16 activations in operand
// order (scaled per token by xsc^-1), per-group sums of the BF16 values.
struct PfPrepared {
    const void *X16;
    const float *xsc, *XG;
    float *QF;  // route_f32_bytes of scratch for the router
};

size_t pf_workspace_bytes(int T, int D, int I, int S, int E, int K);
// Before routing: (optional rmsnorm) -> FP16 rows, scales, group sums.
cudaError_t launch_prefill_prepare(const PfCall &c, PfPrepared *out, cudaStream_t s);
// After routing: scatter, gate/up GEMM, down GEMM, combine.
cudaError_t launch_prefill(const PfCall &c, cudaStream_t s);
// Routing of many tokens from the prepared activations (same logits, bit for bit).
// QF: route_f32_bytes(T, D, E, K) of workspace: the router's bytes as floats,
// then (reused) the per-block counts of the grouping.
size_t route_f32_bytes(int T, int D, int E, int K);
cudaError_t launch_route_large(const RouteArgs &a, const void *X16, const float *xsc, const float *XG, float *QF,
                               cudaStream_t s);

// Opt kernel `k` into `bytes` of dynamic shared memory on the current device.
// cudaFuncSetAttribute acts on the current device only, so the opt-in is
// remembered per (device, kernel); sizes up to 48 KiB need none.
cudaError_t smem_optin(const void *k, size_t bytes);

// Stage profiler (mx_moe_profile_*): event pair around one launch.
enum Stage { kStageRoute = 0, kStageGateUp = 1, kStageDown = 2 };
void prof_begin(int stage, cudaStream_t s);
void prof_end(int stage, cudaStream_t s);

} // namespace mx

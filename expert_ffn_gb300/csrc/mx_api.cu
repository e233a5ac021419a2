// mx_api.cu -- the C ABI declared in include/mx_moe.h: argument validation,
// workspace plan, and the launch sequence of the block.
//
// Validation follows the reject-don't-guess rule of the "Mference System
// design" page (section "The .gturbo directory": the runtime rejects unknown
// format flags, incompatible architecture values and invalid alignment); it
// runs entirely on the host, before any CUDA call, so a rejected call touches
// neither the device nor the outputs.
#include "mx_moe.h"
#include "mx_internal.h"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

using namespace mx;

namespace {

thread_local char g_err[512] = "";

mx_status fail(mx_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

mx_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(MX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

mx_status check_qlinear(const mx_qlinear *q, const char *name, int rows, int cols, int bits)
{
    if (!q)
        return fail(MX_ERR_INVALID_ARG, "%s is NULL", name);
    if (!q->w || !q->scales || !q->biases)
        return fail(MX_ERR_INVALID_ARG, "%s has a NULL pointer", name);
    if (q->bits != bits)
        return fail(MX_ERR_UNSUPPORTED, "%s: bits=%d, expected %d", name, q->bits, bits);
    if (q->rows != rows || q->cols != cols)
        return fail(MX_ERR_INVALID_ARG, "%s: shape [%d, %d], expected [%d, %d]", name, q->rows, q->cols, rows,
                    cols);
    if (!aligned(q->w, 16) || !aligned(q->scales, 16) || !aligned(q->biases, 16))
        return fail(MX_ERR_ALIGNMENT, "%s: pointers must be 16-byte aligned", name);
    return MX_OK;
}

mx_status check_layout(const mx_moe_layout *L)
{
    if (!L)
        return fail(MX_ERR_INVALID_ARG, "layout is NULL");
    if (L->magic != MX_MOE_LAYOUT_MAGIC)
        return fail(MX_ERR_INVALID_ARG, "layout magic 0x%08x is not 0x%08x", L->magic, MX_MOE_LAYOUT_MAGIC);
    if (L->version < 1u || L->version > MX_MOE_LAYOUT_VERSION)
        return fail(MX_ERR_INVALID_ARG, "layout version %u is not supported", L->version);
    const int D = L->d_model, I = L->d_expert, E = L->n_experts, K = L->top_k, S = L->d_shared;
    if (L->group != 64)
        return fail(MX_ERR_UNSUPPORTED, "group %d: only 64 is supported", L->group);
    if (L->bits != 4)
        return fail(MX_ERR_UNSUPPORTED, "expert bits %d: only 4 is supported", L->bits);
    if (D <= 0 || D % 64 || D > kMaxDim)
        return fail(MX_ERR_UNSUPPORTED, "d_model %d must be a positive multiple of 64 <= %d", D, kMaxDim);
    if (I <= 0 || I % 64 || I > kMaxDim)
        return fail(MX_ERR_UNSUPPORTED, "d_expert %d must be a positive multiple of 64 <= %d", I, kMaxDim);
    if (S <= 0 || S % 64 || S > kMaxDim)
        return fail(MX_ERR_UNSUPPORTED, "d_shared %d must be a positive multiple of 64 <= %d", S, kMaxDim);
    if (E < 1 || E > kMaxExperts)
        return fail(MX_ERR_UNSUPPORTED, "n_experts %d must be in [1, %d]", E, kMaxExperts);
    if (K < 1 || K > E || K > kMaxTopK)
        return fail(MX_ERR_INVALID_ARG, "top_k %d must be in [1, min(n_experts, %d)]", K, kMaxTopK);
    if (L->act_dtype != MX_F32 && L->act_dtype != MX_BF16)
        return fail(MX_ERR_INVALID_ARG, "act_dtype %d is not MX_F32 or MX_BF16", L->act_dtype);
    if (L->record_stride == 0 || L->record_stride % 4096)
        return fail(MX_ERR_ALIGNMENT, "record_stride %llu must be a positive multiple of 4096",
                    (unsigned long long)L->record_stride);
    const uint64_t wsz[3] = {(uint64_t)I * D / 2, (uint64_t)I * D / 2, (uint64_t)D * I / 2};
    const uint64_t ssz[3] = {(uint64_t)I * (D / 64) * 2, (uint64_t)I * (D / 64) * 2, (uint64_t)D * (I / 64) * 2};
    const mx_sub *subs[3] = {&L->gate, &L->up, &L->down};
    const char *names[3] = {"gate", "up", "down"};
    for (int j = 0; j < 3; ++j) {
        const uint64_t offs[3] = {subs[j]->w, subs[j]->s, subs[j]->b};
        const uint64_t sizes[3] = {wsz[j], ssz[j], ssz[j]};
        for (int k = 0; k < 3; ++k) {
            if (offs[k] % 16)
                return fail(MX_ERR_ALIGNMENT, "%s offset %llu is not 16-byte aligned", names[j],
                            (unsigned long long)offs[k]);
            if (offs[k] > L->record_stride || sizes[k] > L->record_stride - offs[k])
                return fail(MX_ERR_INVALID_ARG, "%s sub-tensor [%llu, +%llu) exceeds the record stride %llu",
                            names[j], (unsigned long long)offs[k], (unsigned long long)sizes[k],
                            (unsigned long long)L->record_stride);
        }
    }
    if (L->per_expert_scale && !aligned(L->per_expert_scale, 4))
        return fail(MX_ERR_ALIGNMENT, "per_expert_scale must be 4-byte aligned");
    if (L->version >= 2u) {
        if (L->expert_slot) {
            if (!aligned(L->expert_slot, 2))
                return fail(MX_ERR_ALIGNMENT, "expert_slot must be 2-byte aligned");
            if (L->n_slots < 1 || L->n_slots > 32767)
                return fail(MX_ERR_INVALID_ARG, "n_slots %d must be in [1, 32767] with an expert_slot table",
                            L->n_slots);
        }
        const void *vecs[3] = {L->router_scale, L->post_norm, L->shared_expert_gate};
        const char *vnames[3] = {"router_scale", "post_norm", "shared_expert_gate"};
        for (int j = 0; j < 3; ++j)
            if (vecs[j] && !aligned(vecs[j], 16))
                return fail(MX_ERR_ALIGNMENT, "%s must be 16-byte aligned", vnames[j]);
        if (L->post_norm && !(L->post_eps >= 0.0f))
            return fail(MX_ERR_INVALID_ARG, "post_eps must be >= 0");
    }
    if (L->version >= 3u && L->down_sb && !aligned(L->down_sb, 16))
        return fail(MX_ERR_ALIGNMENT, "down_sb must be 16-byte aligned");
    return MX_OK;
}

// The optional parts of a layout (none for a version-1 layout).
LayerExt ext_of(const mx_moe_layout *L)
{
    LayerExt x{};
    x.n_slots = L->n_experts;
    x.rcoef = 1.0f / sqrtf((float)L->d_model);
    if (L->version >= 2u) {
        x.slot = L->expert_slot;
        if (x.slot)
            x.n_slots = L->n_slots;
        x.router_scale = L->router_scale;
        x.post_norm = L->post_norm;
        x.post_eps = L->post_eps;
        x.shared_gate = L->shared_expert_gate;
    }
    if (L->version >= 3u)
        x.down_sb = L->down_sb;
    return x;
}

// The parts only the single-launch and grouped-GEMM paths implement.
bool ext_needs_new_paths(const LayerExt &x) { return x.router_scale || x.post_norm || x.shared_gate; }

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Workspace plan.  Offsets are 256-byte aligned; the ticket counters come first
// so mx_moe_workspace_init only needs to clear the front.
struct Plan {
    size_t err, tickets, logits, counts, offsets, perm, tiles, ntiles, xp, xg, hr0, hr1, hs0, hs1;
    // single-launch decode path (T <= kPdMaxT)
    size_t pd_ctr, pd_logits, pd_y, pd_x;
    int pd_T;
    // prefill path (T > kPrefillAbove, BF16)
    size_t pf;
    size_t total;
    int max_tiles_route;
};

Plan make_plan(const mx_moe_layout *L, int T_route, int T_ffn)
{
    const size_t D = L->d_model, I = L->d_expert, E = L->n_experts, K = L->top_k, S = L->d_shared;
    Plan p{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += up256(bytes);
        return at;
    };
    p.err = take(sizeof(unsigned));  // offset 0: device error word (bounded waits)
    p.tickets = take(((size_t)T_route + 2) * sizeof(unsigned));
    p.logits = take((size_t)T_route * E * 4);
    p.counts = take(E * 4);
    p.offsets = take((E + 1) * 4);
    p.perm = take((size_t)T_route * K * 4);
    p.max_tiles_route = (int)(E + ((size_t)T_route * K) / kTileTokens + 1);
    p.tiles = take((size_t)3 * p.max_tiles_route * 4);
    p.ntiles = take(4);
    p.xp = take((size_t)3 * T_ffn * D * 2);
    p.xg = take((size_t)T_ffn * (D / 64) * 4);
    p.hr0 = take((size_t)T_ffn * K * I * 2);
    p.hr1 = take((size_t)T_ffn * K * I * 2);
    p.hs0 = take((size_t)T_ffn * S * 2);
    p.hs1 = take((size_t)T_ffn * S * 2);
    // single-launch decode path, sized for min(T, kPdMaxT) tokens
    const size_t Tp = T_ffn < kPdMaxT ? T_ffn : kPdMaxT;
    const size_t es = L->act_dtype == MX_F32 ? 4 : 2;
    p.pd_T = (int)Tp;
    p.pd_ctr = take(pd_ctr_ints((int)E, kPdMaxLayers) * 4);
    p.pd_logits = take(Tp * E * 4);
    p.pd_y = take((size_t)kPdMaxLayers * Tp * D * 8);
    p.pd_x = take(Tp * D * es);
    p.pf = (T_route > kPrefillAbove && L->act_dtype == MX_BF16)
               ? take(pf_workspace_bytes(T_route, (int)D, (int)I, (int)S, (int)E, (int)K))
               : o;
    p.total = o;
    return p;
}

int ffn_tokens(int T) { return T < kDecodeChunk ? T : kDecodeChunk; }

// Number of SMs of the current device (cached per device).
int num_sms()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    std::lock_guard<std::mutex> g(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// Device limits used by the single-launch path (cached per device).
struct DevInfo {
    int sms = 0, smem_optin = 0;
};

DevInfo dev_info()
{
    static std::mutex mu;
    static DevInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return DevInfo{};
    std::lock_guard<std::mutex> g(mu);
    DevInfo &d = cache[dev];
    if (!d.sms) {
        int n = 0, m = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&m, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return DevInfo{};
        d.sms = n;
        d.smem_optin = m;
    }
    return d;
}

// Whether T tokens of this layout take the single-launch path; fills its plan.
// MX_MOE_SINGLE_LAUNCH=0 in the environment turns the path off (the block then
// runs as separate router / gate-up / down launches).
bool pd_usable(const mx_moe_layout *L, int T, PdSmem *sm, int *n_cta)
{
    if (T < 1 || T > kPdMaxT)
        return false;
    const char *env = getenv("MX_MOE_SINGLE_LAUNCH");
    if (env && env[0] == '0')
        return false;
    const DevInfo d = dev_info();
    if (!d.sms)
        return false;
    // the kernel keeps the scale / bias offsets inside an expert record in 32 bits
    const mx_sub *subs[3] = {&L->gate, &L->up, &L->down};
    for (int j = 0; j < 3; ++j)
        if ((subs[j]->s | subs[j]->b) >> 32)
            return false;
    const int act = L->act_dtype == MX_BF16 ? 1 : 0;
    // leave room for the kernel's static shared memory
    if (!pd_plan(T, L->d_model, L->d_expert, L->d_shared, L->n_experts, L->top_k, act, d.sms, d.smem_optin - 1280,
                 sm))
        return false;
    *n_cta = d.sms;
    return true;
}

// One layer of the single-launch path.
struct PdIn {
    const mx_qlinear *router;
    const mx_ffn *shared;
    const void *blob;
    const mx_moe_layout *L;
    const void *x_in;      // used for the launch's first layer
    void *x_out;           // nullable
    const void *residual;  // res_mode 2
    int res_mode;          // 0 none, 1 the layer input, 2 residual
    int32_t *topk_idx;
    float *topk_w;
};

mx_status run_pd(const PdIn *in, int n, int T, int pre_norm, float eps, const PdSmem &sm, int n_cta, const Plan &p,
                 uint8_t *ws, cudaStream_t s)
{
    const mx_moe_layout *L0 = in[0].L;
    // ~31 KB of kernel parameters: one static block (not thread-local, whose
    // lazy per-thread allocation would make a host thread's first call
    // allocate), held under a lock until the launch has copied it
    static PdParams P;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    std::memset(&P, 0, sizeof P);
    P.T = T;
    P.D = L0->d_model;
    P.I = L0->d_expert;
    P.S = L0->d_shared;
    P.E = L0->n_experts;
    P.K = L0->top_k;
    P.n_layers = n;
    P.act = L0->act_dtype == MX_BF16 ? 1 : 0;
    P.pre_norm = pre_norm;
    P.eps = eps;
    P.n_cta = n_cta;
    P.err = reinterpret_cast<unsigned *>(ws + p.err);
    P.ctr = reinterpret_cast<int *>(ws + p.pd_ctr);
    P.cstride = 3 + P.E;
    P.logits = reinterpret_cast<float *>(ws + p.pd_logits);
    P.ybuf = reinterpret_cast<long long *>(ws + p.pd_y);
    // Failure injection on the host, for tests of the bounded waits:
    // MX_MOE_WAIT_LIMIT_US shortens every wait on another CTA (default 2 s),
    // MX_MOE_HOLD_CTA=c keeps CTA c from arriving at the first logit exchange.
    P.wait_ns = 2000000000ull;
    P.hold_cta = -1;
    if (const char *v = getenv("MX_MOE_WAIT_LIMIT_US")) {
        const long long us = atoll(v);
        if (us > 0)
            P.wait_ns = (unsigned long long)us * 1000ull;
    }
    if (const char *v = getenv("MX_MOE_HOLD_CTA"))
        P.hold_cta = atoi(v);
    P.sm = sm;
    for (int l = 0; l < n; ++l) {
        const PdIn &c = in[l];
        const mx_moe_layout *L = c.L;
        PdLayer &d = P.L[l];
        const LayerExt x = ext_of(L);
        FfnArgs f{};
        f.D = L->d_model;
        f.I = L->d_expert;
        f.S = L->d_shared;
        f.E = L->n_experts;
        f.slot = x.slot;
        f.n_slots = x.n_slots;
        f.blob = static_cast<const uint8_t *>(c.blob);
        f.stride = L->record_stride;
        const mx_sub *subs[3] = {&L->gate, &L->up, &L->down};
        const mx_qlinear *sq[3] = {&c.shared->gate, &c.shared->up, &c.shared->down};
        for (int j = 0; j < 3; ++j) {
            f.off_w[j] = subs[j]->w;
            d.off_s[j] = subs[j]->s;
            d.off_b[j] = subs[j]->b;
            f.sw[j] = static_cast<const uint32_t *>(sq[j]->w);
            d.ss[j] = static_cast<const uint16_t *>(sq[j]->scales);
            d.sb[j] = static_cast<const uint16_t *>(sq[j]->biases);
        }
        FfnMaps maps;
        cudaError_t e = get_ffn_maps(f, &maps);
        if (e != cudaSuccess)
            return cuda_fail(e, "encoding the weight tensor maps");
        d.gate = maps.gate;
        d.up = maps.up;
        d.down = maps.down1;
        d.sgate = maps.sgate;
        d.sup = maps.sup;
        d.sdown = maps.sdown1;
        d.rw = static_cast<const uint32_t *>(c.router->w);
        d.rs = static_cast<const uint16_t *>(c.router->scales);
        d.rb = static_cast<const uint16_t *>(c.router->biases);
        d.blob = f.blob;
        d.stride = L->record_stride;
        d.pes = L->per_expert_scale;
        d.topk_idx = c.topk_idx;
        d.topk_w = c.topk_w;
        d.x_in = c.x_in;
        d.x_out = c.x_out;
        d.residual = c.residual;
        d.res_mode = c.res_mode;
        d.lam = L->layer_scalar;
        d.dsb = x.down_sb;
        d.dsb_s = x.down_sb ? x.down_sb + (size_t)x.n_slots * (L->d_expert / 64) * L->d_model : nullptr;
        d.slot = x.slot;
        d.n_slots = x.n_slots;
        d.router_scale = x.router_scale;
        d.post_norm = x.post_norm;
        d.shared_gate = x.shared_gate;
        d.post_eps = x.post_eps;
        d.rcoef = x.rcoef;
    }
    prof_begin(kStageGateUp, s);
    cudaError_t e = launch_pd(P, s);
    prof_end(kStageGateUp, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "single-launch decode kernel");
    return MX_OK;
}

struct Call {
    const void *x;
    int T;
    const mx_qlinear *router;
    const mx_ffn *shared;
    const void *blob;
    const mx_moe_layout *L;
    void *out;
    int32_t *topk_idx;
    float *topk_w;
    const mx_moe_options *opt;
};

mx_status validate_block(const Call &c)
{
    mx_status st = check_layout(c.L);
    if (st != MX_OK)
        return st;
    if (c.T < 0)
        return fail(MX_ERR_INVALID_ARG, "T=%d is negative", c.T);
    const int D = c.L->d_model, E = c.L->n_experts, S = c.L->d_shared;
    if ((st = check_qlinear(c.router, "router", E, D, 8)) != MX_OK)
        return st;
    if (!c.shared)
        return fail(MX_ERR_INVALID_ARG, "shared is NULL");
    if ((st = check_qlinear(&c.shared->gate, "shared.gate", S, D, 4)) != MX_OK)
        return st;
    if ((st = check_qlinear(&c.shared->up, "shared.up", S, D, 4)) != MX_OK)
        return st;
    if ((st = check_qlinear(&c.shared->down, "shared.down", D, S, 4)) != MX_OK)
        return st;
    if (!c.blob)
        return fail(MX_ERR_INVALID_ARG, "expert_blob is NULL");
    if (!aligned(c.blob, 256))
        return fail(MX_ERR_ALIGNMENT, "expert_blob must be 256-byte aligned");
    if (c.T == 0)
        return MX_OK;
    if (!c.x || !c.out || !c.topk_idx || !c.topk_w)
        return fail(MX_ERR_INVALID_ARG, "x, out, topk_idx and topk_w must be non-NULL");
    if (!aligned(c.x, 16) || !aligned(c.out, 16))
        return fail(MX_ERR_ALIGNMENT, "x and out must be 16-byte aligned");
    if (!aligned(c.topk_idx, 4) || !aligned(c.topk_w, 4))
        return fail(MX_ERR_ALIGNMENT, "topk_idx and topk_w must be 4-byte aligned");
    const size_t es = c.L->act_dtype == MX_F32 ? 4 : 2;
    const size_t xbytes = (size_t)c.T * D * es;
    if (overlap(c.x, xbytes, c.out, xbytes))
        return fail(MX_ERR_INVALID_ARG, "out must not overlap x");
    if (c.opt && c.opt->residual && !aligned(c.opt->residual, 16))
        return fail(MX_ERR_ALIGNMENT, "residual must be 16-byte aligned");
    if (c.opt && c.opt->pre_rmsnorm && !(c.opt->rms_eps >= 0.0f))
        return fail(MX_ERR_INVALID_ARG, "rms_eps must be >= 0");
    return MX_OK;
}

RouteArgs route_args(const void *x, int T, const mx_qlinear *router, const mx_moe_layout *L,
                     const mx_moe_options *opt, const Plan &p, uint8_t *ws)
{
    RouteArgs a{};
    a.x = x;
    a.x_dtype = L->act_dtype == MX_BF16 ? 1 : 0;
    a.T = T;
    a.D = L->d_model;
    a.E = L->n_experts;
    a.K = L->top_k;
    a.rw = static_cast<const uint32_t *>(router->w);
    a.rs = static_cast<const uint16_t *>(router->scales);
    a.rb = static_cast<const uint16_t *>(router->biases);
    a.pre_norm = (opt && opt->pre_rmsnorm) ? 1 : 0;
    a.eps = opt ? opt->rms_eps : 0.0f;
    a.pes = L->per_expert_scale;
    a.logits = reinterpret_cast<float *>(ws + p.logits);
    a.counts = reinterpret_cast<int32_t *>(ws + p.counts);
    a.offsets = reinterpret_cast<int32_t *>(ws + p.offsets);
    a.perm = reinterpret_cast<int32_t *>(ws + p.perm);
    a.tiles = reinterpret_cast<int32_t *>(ws + p.tiles);
    a.n_tiles = reinterpret_cast<int32_t *>(ws + p.ntiles);
    a.tickets = reinterpret_cast<unsigned *>(ws + p.tickets);
    a.err = reinterpret_cast<unsigned *>(ws + p.err);
    a.xp = reinterpret_cast<uint16_t *>(ws + p.xp);
    a.xg = reinterpret_cast<float *>(ws + p.xg);
    a.nsplit = L->act_dtype == MX_BF16 ? 1 : 3;
    return a;
}

// One pass of the block over T <= kDecodeChunk tokens.
mx_status run_pass(const void *x, int T, const mx_qlinear *router, const mx_ffn *shared, const void *blob,
                   const mx_moe_layout *L, void *out, int32_t *topk_idx, float *topk_w, const mx_moe_options *opt,
                   const Plan &p, uint8_t *ws, cudaStream_t s)
{
    RouteArgs ra = route_args(x, T, router, L, opt, p, ws);
    ra.topk_idx = topk_idx;
    ra.topk_w = topk_w;
    ra.logits_only = 0;
    const RouteLaunch rl = route_plan(T, L->d_model, L->n_experts, L->top_k);
    ra.ET = rl.ET;
    ra.GC = rl.GC;
    ra.cluster = rl.cluster;
    prof_begin(kStageRoute, s);
    cudaError_t e = launch_route(ra, rl, s);
    prof_end(kStageRoute, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "route kernel launch");

    FfnArgs f{};
    f.T = T;
    f.D = L->d_model;
    f.I = L->d_expert;
    f.S = L->d_shared;
    f.E = L->n_experts;
    f.K = L->top_k;
    const LayerExt ext = ext_of(L);
    f.slot = ext.slot;
    f.n_slots = ext.n_slots;
    f.blob = static_cast<const uint8_t *>(blob);
    f.stride = L->record_stride;
    const mx_sub *subs[3] = {&L->gate, &L->up, &L->down};
    for (int j = 0; j < 3; ++j) {
        f.off_w[j] = subs[j]->w;
        f.off_s[j] = subs[j]->s;
        f.off_b[j] = subs[j]->b;
    }
    const mx_qlinear *sq[3] = {&shared->gate, &shared->up, &shared->down};
    for (int j = 0; j < 3; ++j) {
        f.sw[j] = static_cast<const uint32_t *>(sq[j]->w);
        f.ss[j] = static_cast<const uint16_t *>(sq[j]->scales);
        f.sb[j] = static_cast<const uint16_t *>(sq[j]->biases);
    }
    f.xp = ra.xp;
    f.xg = ra.xg;
    f.nsplit = ra.nsplit;
    f.logits = ra.logits;
    f.pes = L->per_expert_scale;
    f.topk_idx = topk_idx;
    f.topk_w = topk_w;
    f.perm = ra.perm;
    f.tiles = ra.tiles;
    f.n_tiles = ra.n_tiles;
    f.hr[0] = reinterpret_cast<uint16_t *>(ws + p.hr0);
    f.hr[1] = reinterpret_cast<uint16_t *>(ws + p.hr1);
    f.hs[0] = reinterpret_cast<uint16_t *>(ws + p.hs0);
    f.hs[1] = reinterpret_cast<uint16_t *>(ws + p.hs1);
    f.residual = opt ? opt->residual : nullptr;
    f.out = out;
    f.act_dtype = L->act_dtype == MX_BF16 ? 1 : 0;
    f.lam = L->layer_scalar;
    f.err = ra.err;
    const int max_tiles = T * L->top_k < L->n_experts ? T * L->top_k : L->n_experts;
    e = launch_ffn_decode(f, max_tiles, num_sms(), s);
    if (e != cudaSuccess)
        return cuda_fail(e, "ffn kernel launch");
    return MX_OK;
}

// Prefill: prepare the activations, route all T tokens at once from them, then
// the grouped tensor-core GEMMs.
mx_status run_prefill(const Call &c, const Plan &p, uint8_t *ws, cudaStream_t s)
{
    const mx_moe_layout *L = c.L;
    RouteArgs ra = route_args(c.x, c.T, c.router, L, c.opt, p, ws);
    ra.topk_idx = c.topk_idx;
    ra.topk_w = c.topk_w;
    ra.xp = nullptr;
    PfCall f{};
    f.x = c.x;
    f.T = c.T;
    f.D = L->d_model;
    f.I = L->d_expert;
    f.S = L->d_shared;
    f.E = L->n_experts;
    f.K = L->top_k;
    f.pre_norm = (c.opt && c.opt->pre_rmsnorm) ? 1 : 0;
    f.eps = c.opt ? c.opt->rms_eps : 0.0f;
    f.perm = ra.perm;
    f.counts = ra.counts;
    f.offsets = ra.offsets;
    f.topk_w = c.topk_w;
    f.blob = static_cast<const uint8_t *>(c.blob);
    f.stride = L->record_stride;
    const mx_sub *subs[3] = {&L->gate, &L->up, &L->down};
    const mx_qlinear *sq[3] = {&c.shared->gate, &c.shared->up, &c.shared->down};
    for (int j = 0; j < 3; ++j) {
        f.off_w[j] = subs[j]->w;
        f.off_s[j] = subs[j]->s;
        f.off_b[j] = subs[j]->b;
        f.sw[j] = static_cast<const uint32_t *>(sq[j]->w);
        f.ss[j] = static_cast<const uint16_t *>(sq[j]->scales);
        f.sb[j] = static_cast<const uint16_t *>(sq[j]->biases);
    }
    f.lam = L->layer_scalar;
    f.residual = c.opt ? c.opt->residual : nullptr;
    f.out = c.out;
    f.err = ra.err;
    f.ws = ws + p.pf;
    f.n_cta = num_sms();
    f.ext = ext_of(L);
    ra.router_scale = f.ext.router_scale;
    ra.rcoef = f.ext.rcoef;
    PfPrepared pp;
    prof_begin(kStageRoute, s);
    cudaError_t e = launch_prefill_prepare(f, &pp, s);
    if (e == cudaSuccess)
        e = launch_route_large(ra, pp.X16, pp.xsc, pp.XG, pp.QF, s);
    prof_end(kStageRoute, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "prefill routing");
    e = launch_prefill(f, s);  // times its gate/up GEMM and its down GEMM + combine as stages 1 and 2
    if (e != cudaSuccess)
        return cuda_fail(e, "prefill kernels");
    return MX_OK;
}

mx_status forward_impl(const Call &c, cudaStream_t s, void *ws, size_t ws_bytes)
{
    const int D = c.L->d_model, K = c.L->top_k;
    const size_t es = c.L->act_dtype == MX_F32 ? 4 : 2;
    // BF16 with more than kPrefillAbove tokens: the grouped tensor-core GEMMs
    // (MX_MOE_PREFILL_GEMM=0 in the environment keeps such calls on the decode
    // kernels instead)
    const char *pf_env = getenv("MX_MOE_PREFILL_GEMM");
    if (c.T > kPrefillAbove && c.L->act_dtype == MX_BF16 && !(pf_env && pf_env[0] == '0')) {
        const Plan p = make_plan(c.L, c.T, ffn_tokens(c.T));
        if (!ws || ws_bytes < p.total)
            return fail(MX_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, p.total);
        if (!aligned(ws, 256))
            return fail(MX_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
        return run_prefill(c, p, static_cast<uint8_t *>(ws), s);
    }
    const Plan p = make_plan(c.L, ffn_tokens(c.T), ffn_tokens(c.T));
    if (!ws || ws_bytes < p.total)
        return fail(MX_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, p.total);
    if (!aligned(ws, 256))
        return fail(MX_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    uint8_t *w = static_cast<uint8_t *>(ws);
    PdSmem sm;
    int n_cta = 0;
    if (c.T <= p.pd_T && pd_usable(c.L, c.T, &sm, &n_cta)) {
        const void *res = c.opt ? c.opt->residual : nullptr;
        const PdIn in{c.router, c.shared, c.blob, c.L, c.x, c.out, res, res ? 2 : 0, c.topk_idx, c.topk_w};
        const int pre = (c.opt && c.opt->pre_rmsnorm) ? 1 : 0;
        return run_pd(&in, 1, c.T, pre, c.opt ? c.opt->rms_eps : 0.0f, sm, n_cta, p, w, s);
    }
    if (ext_needs_new_paths(ext_of(c.L)))
        return fail(MX_ERR_UNSUPPORTED, "router_scale, post_norm and shared_expert_gate need the single-launch "
                                        "decode path (T <= %d) or the grouped GEMMs (BF16, T > %d); this call "
                                        "(T=%d, %s) would run the multi-launch decode kernels",
                    kPdMaxT, kPrefillAbove, c.T, c.L->act_dtype == MX_BF16 ? "bf16" : "fp32");
    for (int t0 = 0; t0 < c.T; t0 += kDecodeChunk) {
        const int n = c.T - t0 < kDecodeChunk ? c.T - t0 : kDecodeChunk;
        mx_moe_options o{};
        if (c.opt)
            o = *c.opt;
        if (o.residual)
            o.residual = static_cast<const uint8_t *>(o.residual) + (size_t)t0 * D * es;
        mx_status st = run_pass(static_cast<const uint8_t *>(c.x) + (size_t)t0 * D * es, n, c.router, c.shared,
                                c.blob, c.L, static_cast<uint8_t *>(c.out) + (size_t)t0 * D * es,
                                c.topk_idx + (size_t)t0 * K, c.topk_w + (size_t)t0 * K, &o, p, w, s);
        if (st != MX_OK)
            return st;
    }
    return MX_OK;
}

// Library-owned workspace of the 9-argument entry point (per device).
struct OwnedWs {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;
OwnedWs g_ws[64];

} // namespace

// Scratch of mx_moe_layer_forward_static: one per device, zero at load.
static __device__ __align__(256) unsigned char g_static_scratch[MX_STATIC_SCRATCH_BYTES];
static std::mutex g_static_mu;
static void *g_static_ptr[64];  // per device ordinal, resolved on the first call

// Column-major copy of the down projections' (scale | bias << 16) words: one
// thread per output word (record words, then the shared expert's).  A one-off
// rearrangement: the strided reads are not worth tiling.
__global__ void pack_down_sb_kernel(const uint8_t *blob, uint64_t stride, uint64_t off_s, uint64_t off_b, int nrec,
                                    int GI, int D, const uint16_t *ss, const uint16_t *sb, int GS, uint32_t *out)
{
    const size_t n_r = (size_t)nrec * GI * D, n = n_r + (size_t)GS * D;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        uint16_t sv, bv;
        if (i < n_r) {
            const size_t d = i % D, rg = i / D, r = rg / GI;
            const int g = (int)(rg % GI);
            const uint8_t *rec = blob + r * stride;
            sv = reinterpret_cast<const uint16_t *>(rec + off_s)[d * GI + g];
            bv = reinterpret_cast<const uint16_t *>(rec + off_b)[d * GI + g];
        } else {
            const size_t j = i - n_r, d = j % D, g = j / D;
            sv = ss[d * GS + g];
            bv = sb[d * GS + g];
        }
        out[i] = (uint32_t)sv | ((uint32_t)bv << 16);
    }
}

extern "C" {

const char *mx_version(void) { return "0.1.0"; }

const char *mx_status_string(mx_status s)
{
    switch (s) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
    case MX_ERR_ALIGNMENT: return "MX_ERR_ALIGNMENT";
    case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
    case MX_ERR_WORKSPACE: return "MX_ERR_WORKSPACE";
    case MX_ERR_CUDA: return "MX_ERR_CUDA";
    case MX_ERR_DEVICE_TIMEOUT: return "MX_ERR_DEVICE_TIMEOUT";
    case MX_ERR_RANGE: return "MX_ERR_RANGE";
    case MX_ERR_NOT_RESIDENT: return "MX_ERR_NOT_RESIDENT";
    }
    return "MX_ERR_UNKNOWN";
}

const char *mx_last_error_string(void) { return g_err; }

size_t mx_moe_workspace_bytes(const mx_moe_layout *layout, int T_max)
{
    if (check_layout(layout) != MX_OK || T_max < 0)
        return 0;
    const int t = T_max < 1 ? 1 : T_max;
    return make_plan(layout, t, ffn_tokens(t)).total;
}

size_t mx_moe_stack_workspace_bytes(const mx_moe_layout *layout, int T)
{
    if (check_layout(layout) != MX_OK || T < 0)
        return 0;
    const int t = T < 1 ? 1 : T;
    // the per-layer plan, then the ping-pong activation buffer
    return make_plan(layout, t, ffn_tokens(t)).total + up256((size_t)t * layout->d_model * 4);
}

size_t mx_moe_down_sb_bytes(const mx_moe_layout *layout)
{
    if (check_layout(layout) != MX_OK)
        return 0;
    const LayerExt x = ext_of(layout);
    const size_t D = layout->d_model, GI = layout->d_expert / 64, GS = layout->d_shared / 64;
    return ((size_t)x.n_slots * GI + GS) * D * 4;
}

mx_status mx_moe_pack_down_sb(const mx_moe_layout *layout, const void *blob, const mx_qlinear *shared_down,
                              uint32_t *out, void *stream)
{
    mx_status st;
    if ((st = check_layout(layout)) != MX_OK)
        return st;
    if (!blob || !shared_down || !out)
        return fail(MX_ERR_INVALID_ARG, "mx_moe_pack_down_sb: blob, shared_down and out must not be NULL");
    const int D = layout->d_model, I = layout->d_expert, S = layout->d_shared;
    if ((st = check_qlinear(shared_down, "shared.down", D, S, 4)) != MX_OK)
        return st;
    if (!aligned(out, 16))
        return fail(MX_ERR_ALIGNMENT, "mx_moe_pack_down_sb: out must be 16-byte aligned");
    const LayerExt x = ext_of(layout);
    const size_t bytes = mx_moe_down_sb_bytes(layout);
    if (overlap(out, bytes, blob, (size_t)x.n_slots * layout->record_stride))
        return fail(MX_ERR_INVALID_ARG, "mx_moe_pack_down_sb: out overlaps the blob");
    const size_t n = bytes / 4;
    const int blocks = (int)std::min<size_t>((n + 255) / 256, 8192);
    pack_down_sb_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(blob), layout->record_stride, layout->down.s, layout->down.b, x.n_slots, I / 64,
        D, static_cast<const uint16_t *>(shared_down->scales), static_cast<const uint16_t *>(shared_down->biases),
        S / 64, out);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MX_OK : cuda_fail(e, "mx_moe_pack_down_sb");
}

mx_status mx_moe_workspace_init(void *ws, size_t ws_bytes, void *stream)
{
    if (!ws)
        return fail(MX_ERR_INVALID_ARG, "workspace is NULL");
    cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync");
    return MX_OK;
}

mx_status mx_moe_workspace_check(const void *ws, void *stream)
{
    if (!ws)
        return fail(MX_ERR_INVALID_ARG, "workspace is NULL");
    unsigned word = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the workspace error word");
    if (word & 1u)
        return fail(MX_ERR_DEVICE_TIMEOUT, "a device-side wait gave up (error word 0x%x)", word);
    if (word & 4u)
        return fail(MX_ERR_NOT_RESIDENT, "a selected expert has no record in the blob (error word 0x%x)", word);
    if (word != 0)
        return fail(MX_ERR_RANGE, "a partial sum fell outside the fixed-point range of the decode path "
                                  "(error word 0x%x)", word);
    return MX_OK;
}

mx_status mx_moe_layer_forward_ex(const void *x, int T, const mx_qlinear *router, const mx_ffn *shared,
                                  const void *expert_blob, const mx_moe_layout *layout, void *out,
                                  int32_t *topk_idx, float *topk_w, const mx_moe_options *opt, void *stream,
                                  void *ws, size_t ws_bytes)
{
    const Call c{x, T, router, shared, expert_blob, layout, out, topk_idx, topk_w, opt};
    mx_status st = validate_block(c);
    if (st != MX_OK || T == 0)
        return st;
    return forward_impl(c, static_cast<cudaStream_t>(stream), ws, ws_bytes);
}

mx_status mx_moe_layer_forward(const void *x, int T, const mx_qlinear *router, const mx_ffn *shared,
                               const void *expert_blob, const mx_moe_layout *layout, void *out, int32_t *topk_idx,
                               float *topk_w)
{
    const Call c{x, T, router, shared, expert_blob, layout, out, topk_idx, topk_w, nullptr};
    mx_status st = validate_block(c);
    if (st != MX_OK || T == 0)
        return st;
    const size_t need = mx_moe_workspace_bytes(layout, T);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(MX_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> g(g_ws_mu);
    OwnedWs &w = g_ws[dev];
    if (w.bytes < need) {
        if (w.ptr) {
            cudaDeviceSynchronize();
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
        }
        if ((e = cudaMalloc(&w.ptr, need)) != cudaSuccess)
            return fail(MX_ERR_WORKSPACE, "cudaMalloc(%zu): %s", need, cudaGetErrorString(e));
        if ((e = cudaMemset(w.ptr, 0, need)) != cudaSuccess)
            return cuda_fail(e, "cudaMemset");
        w.bytes = need;
    }
    return forward_impl(c, nullptr, w.ptr, w.bytes);
}

// ------------------------------------------------ allocation-free variant

mx_status mx_moe_layer_forward_static(const void *x, int T, const mx_qlinear *router, const mx_ffn *shared,
                                      const void *expert_blob, const mx_moe_layout *layout, void *out,
                                      int32_t *topk_idx, float *topk_w, const mx_moe_options *opt, void *stream)
{
    const Call c{x, T, router, shared, expert_blob, layout, out, topk_idx, topk_w, opt};
    mx_status st = validate_block(c);
    if (st != MX_OK || T == 0)
        return st;
    const int D = layout->d_model, E = layout->n_experts;
    if (T > kPdMaxT || D > kPdMaxD || E > 256)
        return fail(MX_ERR_UNSUPPORTED, "the allocation-free call takes T <= %d, d_model <= %d, n_experts <= 256 "
                                        "(got T=%d, d_model=%d, n_experts=%d)",
                    kPdMaxT, kPdMaxD, T, D, E);
    PdSmem sm;
    int n_cta = 0;
    if (!pd_usable(layout, T, &sm, &n_cta))
        return fail(MX_ERR_UNSUPPORTED, "the single-launch decode path is not usable for this layout on this device");
    // scratch: error word, counters, logits, fixed-point sums (all must start at zero)
    Plan p{};
    p.err = 0;
    p.pd_ctr = 256;
    p.pd_logits = p.pd_ctr + up256(pd_ctr_ints(E, 1) * sizeof(int));
    p.pd_y = p.pd_logits + up256((size_t)T * E * sizeof(float));
    const size_t used = p.pd_y + (size_t)T * D * sizeof(long long);
    if (used > MX_STATIC_SCRATCH_BYTES)
        return fail(MX_ERR_UNSUPPORTED, "scratch of %zu bytes needed, %u available", used, MX_STATIC_SCRATCH_BYTES);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(MX_ERR_UNSUPPORTED, "device ordinal %d", dev);
    void *base;
    {
        std::lock_guard<std::mutex> g(g_static_mu);
        if (!g_static_ptr[dev]) {
            void *ptr = nullptr;
            if ((e = cudaGetSymbolAddress(&ptr, g_static_scratch)) != cudaSuccess)
                return cuda_fail(e, "cudaGetSymbolAddress");
            g_static_ptr[dev] = ptr;
        }
        base = g_static_ptr[dev];
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((e = cudaMemsetAsync(base, 0, used, s)) != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync");
    const void *res = opt ? opt->residual : nullptr;
    const PdIn in{router, shared, expert_blob, layout, x, out, res, res ? 2 : 0, topk_idx, topk_w};
    const int pre = (opt && opt->pre_rmsnorm) ? 1 : 0;
    return run_pd(&in, 1, T, pre, opt ? opt->rms_eps : 0.0f, sm, n_cta, p, static_cast<uint8_t *>(base), s);
}

mx_status mx_moe_route(const void *x, int T, const mx_qlinear *router, const mx_moe_layout *layout,
                       int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *offsets, int32_t *perm,
                       float *logits, const mx_moe_options *opt, void *stream, void *ws, size_t ws_bytes)
{
    mx_status st = check_layout(layout);
    if (st != MX_OK)
        return st;
    if (T < 0)
        return fail(MX_ERR_INVALID_ARG, "T=%d is negative", T);
    if ((st = check_qlinear(router, "router", layout->n_experts, layout->d_model, 8)) != MX_OK)
        return st;
    if (ext_of(layout).router_scale)
        return fail(MX_ERR_UNSUPPORTED, "mx_moe_route does not take a layout with router_scale");
    if (T == 0)
        return MX_OK;
    if (!x || !topk_idx || !topk_w || !counts || !offsets || !perm)
        return fail(MX_ERR_INVALID_ARG, "x, topk_idx, topk_w, counts, offsets and perm must be non-NULL");
    if (!aligned(x, 16))
        return fail(MX_ERR_ALIGNMENT, "x must be 16-byte aligned");
    if (opt && opt->pre_rmsnorm && !(opt->rms_eps >= 0.0f))
        return fail(MX_ERR_INVALID_ARG, "rms_eps must be >= 0");
    const Plan p = make_plan(layout, T, ffn_tokens(T));
    if (!ws || ws_bytes < p.total)
        return fail(MX_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, p.total);
    if (!aligned(ws, 256))
        return fail(MX_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    uint8_t *w = static_cast<uint8_t *>(ws);
    RouteArgs a = route_args(x, T, router, layout, opt, p, w);
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    if (logits)
        a.logits = logits;
    a.xp = nullptr;
    const RouteLaunch rl = route_plan(T, layout->d_model, layout->n_experts, layout->top_k);
    a.ET = rl.ET;
    a.GC = rl.GC;
    a.cluster = rl.cluster;
    prof_begin(kStageRoute, static_cast<cudaStream_t>(stream));
    cudaError_t e = launch_route(a, rl, static_cast<cudaStream_t>(stream));
    prof_end(kStageRoute, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "route kernel launch");
    return MX_OK;
}

mx_status mx_moe_stack_forward(void *x_io, int T, int n_layers, const mx_qlinear *routers, const mx_ffn *shareds,
                               const void *const *expert_blobs, const mx_moe_layout *layouts, int32_t *topk_idx,
                               float *topk_w, float rms_eps, void *stream, void *ws, size_t ws_bytes)
{
    if (n_layers < 1 || !routers || !shareds || !expert_blobs || !layouts)
        return fail(MX_ERR_INVALID_ARG, "n_layers >= 1 and non-NULL per-layer arrays are required");
    if (!(rms_eps >= 0.0f))
        return fail(MX_ERR_INVALID_ARG, "rms_eps must be >= 0");
    const mx_moe_layout *L0 = &layouts[0];
    mx_status st = check_layout(L0);
    if (st != MX_OK)
        return st;
    const size_t es = L0->act_dtype == MX_F32 ? 4 : 2;
    const size_t xbytes = (size_t)T * L0->d_model * es;
    const size_t need = mx_moe_stack_workspace_bytes(L0, T);
    if (!ws || ws_bytes < need)
        return fail(MX_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
    if (!aligned(ws, 256))
        return fail(MX_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    const int t1 = T < 1 ? 1 : T;
    const size_t layer_ws = make_plan(L0, t1, ffn_tokens(t1)).total;
    uint8_t *xbuf = static_cast<uint8_t *>(ws) + layer_ws;
    for (int l = 0; l < n_layers; ++l) {
        const mx_moe_layout *L = &layouts[l];
        if (L->d_model != L0->d_model || L->d_expert != L0->d_expert || L->n_experts != L0->n_experts ||
            L->top_k != L0->top_k || L->d_shared != L0->d_shared || L->act_dtype != L0->act_dtype)
            return fail(MX_ERR_INVALID_ARG, "layer %d: every layer must share D, I, E, K, S and dtype", l);
        const void *xin = (l % 2 == 0) ? x_io : xbuf;
        void *xout = (l % 2 == 0) ? static_cast<void *>(xbuf) : x_io;
        const Call c{xin, T, &routers[l], &shareds[l], expert_blobs[l], L, xout,
                     topk_idx ? topk_idx + (size_t)l * T * L0->top_k : nullptr,
                     topk_w ? topk_w + (size_t)l * T * L0->top_k : nullptr, nullptr};
        if ((st = validate_block(c)) != MX_OK) {
            char why[sizeof g_err];
            memcpy(why, g_err, sizeof why);
            return fail(st, "layer %d: %s", l, why);
        }
    }
    if (T == 0)
        return MX_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        const Plan p = make_plan(L0, ffn_tokens(t1), ffn_tokens(t1));
        PdSmem sm;
        int n_cta = 0;
        if (T <= p.pd_T && pd_usable(L0, T, &sm, &n_cta)) {
            // all layers in launches of up to kPdMaxLayers: x stays on chip
            // inside a launch; between launches it passes through the
            // workspace; the last layer writes x_io
            uint8_t *w = static_cast<uint8_t *>(ws);
            PdIn in[kPdMaxLayers];
            for (int l0 = 0; l0 < n_layers; l0 += kPdMaxLayers) {
                const int n = n_layers - l0 < kPdMaxLayers ? n_layers - l0 : kPdMaxLayers;
                for (int i = 0; i < n; ++i) {
                    const int l = l0 + i;
                    const void *xin = l == 0 ? x_io : static_cast<const void *>(w + p.pd_x);
                    void *xout = nullptr;
                    if (i == n - 1)
                        xout = l == n_layers - 1 ? x_io : static_cast<void *>(w + p.pd_x);
                    in[i] = PdIn{&routers[l], &shareds[l], expert_blobs[l], &layouts[l], xin, xout, nullptr, 1,
                                 topk_idx + (size_t)l * T * L0->top_k, topk_w + (size_t)l * T * L0->top_k};
                }
                if ((st = run_pd(in, n, T, 1, rms_eps, sm, n_cta, p, w, s)) != MX_OK)
                    return st;
            }
            return MX_OK;
        }
    }
    for (int l = 0; l < n_layers; ++l) {
        const void *xin = (l % 2 == 0) ? x_io : xbuf;
        void *xout = (l % 2 == 0) ? static_cast<void *>(xbuf) : x_io;
        mx_moe_options o{};
        o.residual = xin;
        o.pre_rmsnorm = 1;
        o.rms_eps = rms_eps;
        const Call c{xin, T, &routers[l], &shareds[l], expert_blobs[l], &layouts[l], xout,
                     topk_idx + (size_t)l * T * L0->top_k, topk_w + (size_t)l * T * L0->top_k, &o};
        if ((st = forward_impl(c, s, ws, layer_ws)) != MX_OK)
            return st;
    }
    if (n_layers % 2 == 1) {
        cudaError_t e = cudaMemcpyAsync(x_io, xbuf, xbytes, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyAsync");
    }
    return MX_OK;
}

} // extern "C"

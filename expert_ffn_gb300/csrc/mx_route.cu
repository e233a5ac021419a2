// mx_route.cu -- router GEMV (8-bit affine) + top-k + softmax + grouping of
// token/expert pairs, in one launch.
//
// "Mference System design" page, section "Decode": logits = int8_affine(x),
// top8 = highest_8(logits), weights = softmax(logits[top8]) *
// per_expert_scale[top8]; section "Prefill": token/expert pairs are grouped
// into bounded per-expert work.
//
// Logit order (fixed so the discrete top-k decision is reproducible bit for bit;
// "TinyTitan_Datacenter Architecture" page, "Invariants", items 1-2):
//   per group g of 64 columns:  X = ((x0 + x1) + x2) + ...        (fp32 adds)
//                               P = fma(q63, x63, ... fma(q0, x0, 0))
//   over groups, ascending:     acc = fma(s_g, P, acc); acc = fma(b_g, X, acc)
//
// Grid: (expert tiles, token tiles).  Each CTA computes the logits of TT tokens
// x ET experts; the last CTA of a token tile (atomic ticket, no waiting) picks
// the top-k of those tokens; the last token tile groups all T*K slots by
// expert.  Tickets return to zero, so the workspace is ready for the next call.
#include "mx_common.cuh"
#include "mx_cta_route.cuh"
#include "mx_internal.h"

#include <cuda_fp16.h>

#include <climits>
#include <mutex>
#include <type_traits>

namespace mx {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kXPad = 68;  // floats per staged group row (64 + 4): conflict-free 16-byte reads

__device__ __forceinline__ float load_x(const RouteArgs &a, int t, int col)
{
    const size_t i = (size_t)t * a.D + col;
    if (a.x_dtype == 1)
        return bf2f(__ldg(reinterpret_cast<const uint16_t *>(a.x) + i));
    return __ldg(reinterpret_cast<const float *>(a.x) + i);
}

// The 64 activations of group g of token t, with 16-byte loads.
__device__ __forceinline__ void load_group(const RouteArgs &a, int t, int g, float (&v)[kGroup])
{
    const size_t i = (size_t)t * a.D + (size_t)g * kGroup;
    if (a.x_dtype == 1) {
        const uint4 *p = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(a.x) + i);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 w = __ldg(p + j);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[8 * j + 2 * k] = __uint_as_float(u[k] << 16);
                v[8 * j + 2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
            }
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.x) + i);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 w = __ldg(p + j);
            v[4 * j] = w.x;
            v[4 * j + 1] = w.y;
            v[4 * j + 2] = w.z;
            v[4 * j + 3] = w.w;
        }
    }
}

// Top-k of the logits of tokens [t0, t0+nt): one warp per token.
__device__ void topk_tokens(const RouteArgs &a, int t0, int nt, float *sm)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E, K = a.K, nwords = (E + 31) >> 5;
    float *lg = sm + warp * E;
    uint32_t *taken = reinterpret_cast<uint32_t *>(sm + kWarps * E) + warp * nwords;
    for (int t = warp; t < nt; t += kWarps) {
        const size_t row = (size_t)(t0 + t);
        for (int e = lane; e < E; e += 32) {
            const float v = __ldcg(a.logits + row * E + e);
            lg[e] = isnan(v) ? -INFINITY : v;
        }
        for (int j = lane; j < nwords; j += 32)
            taken[j] = 0u;
        __syncwarp();
        int my_idx = 0;
        float my_val = 0.0f;
        for (int k = 0; k < K; ++k) {
            float bv = -INFINITY;
            int bi = INT_MAX;
            for (int e = lane; e < E; e += 32) {
                if ((taken[e >> 5] >> (e & 31)) & 1u)
                    continue;
                const float v = lg[e];
                if (bi == INT_MAX || v > bv) {
                    bv = v;
                    bi = e;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (lane == 0)
                taken[bi >> 5] |= 1u << (bi & 31);
            if (lane == k) {
                my_idx = bi;
                my_val = bv;
            }
            __syncwarp();
        }
        // softmax over the selected logits, shifted by the largest (lane 0's)
        const float m = __shfl_sync(0xffffffffu, my_val, 0);
        float ev = (lane < K) ? expf(my_val - m) : 0.0f;
        float sum = ev;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane < K) {
            float w = ev / sum;
            if (a.pes)
                w = w * __ldg(a.pes + my_idx);
            a.topk_idx[row * K + lane] = my_idx;
            a.topk_w[row * K + lane] = w;
        }
        __syncwarp();
    }
}

// Group all T*K slots by expert, ascending slot id inside an expert; NW warps.
template <int NW>
__device__ void group_slots_nw(const RouteArgs &a, float *sm)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E, n = a.T * a.K;
    int *wc = reinterpret_cast<int *>(sm);   // [NW][E] per-warp counts
    int *base = wc + NW * E;             // [NW][E] per-warp running bases
    int *cnt = base + NW * E;            // [E]
    int *off = cnt + E;                      // [E]
    int *tix = off + E;                      // [E] first tile slot of each expert
    for (int i = threadIdx.x; i < NW * E; i += (32 * NW))
        wc[i] = 0;
    __syncthreads();
    const int chunk = (n + NW - 1) / NW;
    const int lo = min(n, warp * chunk), hi = min(n, lo + chunk);
    // eight 32-slot rows of the warp's range in flight at a time, then counted
    // in order
    constexpr int kB = 8;
    for (int s0 = lo; s0 < hi; s0 += 32 * kB) {
        int ev[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int s = s0 + 32 * j + lane;
            ev[j] = (s < hi) ? __ldcg(a.topk_idx + s) : -1;
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int e = ev[j];
            const unsigned m = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && lane == __ffs(m) - 1)
                wc[warp * E + e] += __popc(m);
            __syncwarp();
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += (32 * NW)) {
        int run = 0;
        for (int w = 0; w < NW; ++w) {
            base[w * E + e] = run;
            run += wc[w * E + e];
        }
        cnt[e] = run;
        a.counts[e] = run;
    }
    __syncthreads();
    // exclusive scans over experts (counts -> offsets, tiles per expert -> tile
    // slots), by warp 0 with a shuffle scan of per-lane partial sums
    if (warp == 0) {
        const int per = (E + 31) / 32, e_lo = lane * per, e_hi = min(E, e_lo + per);
        int sc = 0, st = 0;
        for (int e = e_lo; e < e_hi; ++e) {
            sc += cnt[e];
            st += (cnt[e] + kTileTokens - 1) / kTileTokens;
        }
        int ic = sc, is = st;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vc = __shfl_up_sync(0xffffffffu, ic, o), vs = __shfl_up_sync(0xffffffffu, is, o);
            if (lane >= o) {
                ic += vc;
                is += vs;
            }
        }
        int oc = ic - sc, os = is - st;
        for (int e = e_lo; e < e_hi; ++e) {
            off[e] = oc;
            a.offsets[e] = oc;
            tix[e] = os;
            oc += cnt[e];
            os += (cnt[e] + kTileTokens - 1) / kTileTokens;
        }
        if (lane == 31) {
            a.offsets[E] = ic;
            if (a.n_tiles)
                *a.n_tiles = is;
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int s0 = lo; s0 < hi; s0 += 32 * kB) {
        int ev[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int s = s0 + 32 * j + lane;
            ev[j] = (s < hi) ? __ldcg(a.topk_idx + s) : -1;
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int s = s0 + 32 * j + lane, e = ev[j];
            const unsigned m = __match_any_sync(0xffffffffu, e);
            if (e >= 0)
                a.perm[off[e] + base[warp * E + e] + __popc(m & lt)] = s;
            __syncwarp();
            if (e >= 0 && lane == __ffs(m) - 1)
                base[warp * E + e] += __popc(m);
            __syncwarp();
        }
    }
    if (a.tiles) {
        for (int e = threadIdx.x; e < E; e += (32 * NW)) {
            int t = tix[e];
            for (int b = 0; b < cnt[e]; b += kTileTokens, ++t) {
                a.tiles[3 * t + 0] = e;
                a.tiles[3 * t + 1] = off[e] + b;
                a.tiles[3 * t + 2] = off[e] + min(b + kTileTokens, cnt[e]);
            }
        }
    }
}

__device__ void group_slots(const RouteArgs &a, float *sm) { group_slots_nw<kWarps>(a, sm); }

struct RouteSync {
    __device__ void operator()() const { __syncthreads(); }
};

template <int TT>
__global__ void __launch_bounds__(kThreads) route_kernel(const RouteArgs a, const RouteLaunch RL)
{
    extern __shared__ __align__(16) float sm[];
    __shared__ int s_last;
    const int tid = threadIdx.x;
    const int D = a.D, G = D / kGroup, E = a.E, ET = a.ET, GC = a.GC;
    const int t0 = blockIdx.y * TT, nt = min(TT, a.T - t0);
    const int e0 = blockIdx.x * ET, ne = min(ET, E - e0);
    float *xs = sm;                         // [TT][GC][kXPad]
    float *Ps = xs + TT * GC * kXPad;       // [TT][ET][GC]
    float *Xs = Ps + TT * ET * GC;          // [TT][G]
    float *sS = Xs + TT * G;                // [ET][G]
    float *sB = sS + ET * G;                // [ET][G]
    float *rn = sB + ET * G;                // [TT]
    const bool prep = (blockIdx.x == 0) && a.xp != nullptr;

    // Let the next kernel (gate/up) launch now: its producer streams the shared
    // expert's weights while this kernel runs; it waits for our results itself.
    pdl_trigger();
    // Router scales, biases and the first chunk's packed bytes do not depend on
    // the previous kernel: load them before waiting for it.
    for (int i = tid; i < ne * G; i += kThreads) {
        const size_t j = (size_t)e0 * G + i;
        sS[i] = bf2f(__ldg(a.rs + j));
        sB[i] = bf2f(__ldg(a.rb + j));
    }
    const int my_el = tid % ET, my_gl = tid / ET;
    const bool my_pair = tid < ET * min(GC, G) && my_el < ne;
    uint4 qv[4];
    if (my_pair) {
        const uint32_t *q = a.rw + (size_t)(e0 + my_el) * (D / 4) + (size_t)my_gl * 16;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            qv[j] = ldg_u4(q + 4 * j);
    }
    pdl_wait();

    if (a.pre_norm) {
        // rmsnorm_no_scale, canonical order: per group an fma chain of squares,
        // groups summed ascending, r = 1/sqrtf(ss/D + eps).
        float *tmp = Xs;  // [TT][G]; Xs is filled only after this
        for (int i = tid; i < nt * G; i += kThreads) {
            const int t = i / G, g = i % G;
            float v[kGroup];
            load_group(a, t0 + t, g, v);
            float p = 0.0f;
#pragma unroll
            for (int k = 0; k < kGroup; ++k)
                p = fmaf(v[k], v[k], p);
            tmp[t * G + g] = p;
        }
        __syncthreads();
        if (tid < nt) {
            float ss = 0.0f;
            for (int gb = 0; gb < G; gb += 8) {
                float v8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v8[j] = tmp[tid * G + min(gb + j, G - 1)];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (gb + j < G)
                        ss = ss + v8[j];
            }
            rn[tid] = 1.0f / sqrtf(ss / (float)D + a.eps);
        }
        __syncthreads();
    }

    constexpr int kAcc = 4;  // logit accumulators per thread: TT*ET <= 1024
    float acc[kAcc];
#pragma unroll
    for (int i = 0; i < kAcc; ++i)
        acc[i] = 0.0f;
    const int npairs = nt * ne;
    const size_t TD = (size_t)a.T * D;

    for (int c0 = 0; c0 < G; c0 += GC) {
        const int gc = min(GC, G - c0);
        // stage x (normalised and rounded to the act dtype when asked)
        for (int i = tid; i < nt * gc * kGroup; i += kThreads) {
            const int t = i / (gc * kGroup), r = i % (gc * kGroup), gl = r / kGroup, k = r % kGroup;
            const int col = (c0 + gl) * kGroup + k;
            float v = load_x(a, t0 + t, col);
            if (a.pre_norm) {
                v = v * rn[t];
                if (a.x_dtype == 1)
                    v = bf2f(f2bf(v));
            }
            xs[(t * GC + gl) * kXPad + k] = v;
            if (prep) {
                const size_t o = (size_t)(t0 + t) * D + perm8(col);
                const uint16_t h1 = f2bf(v);
                a.xp[o] = h1;
                if (a.nsplit > 1) {
                    const float r1 = v - bf2f(h1);
                    const uint16_t h2 = f2bf(r1);
                    a.xp[TD + o] = h2;
                    a.xp[2 * TD + o] = f2bf(r1 - bf2f(h2));
                }
            }
        }
        __syncthreads();
        for (int i = tid; i < nt * gc; i += kThreads) {
            const int t = i / gc, gl = i % gc;
            const float4 *xr = reinterpret_cast<const float4 *>(xs + (t * GC + gl) * kXPad);
            float4 v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = xr[j];
            float s = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                s = s + v[j].x;
                s = s + v[j].y;
                s = s + v[j].z;
                s = s + v[j].w;
            }
            Xs[t * G + c0 + gl] = s;
            if (prep)
                a.xg[(size_t)(t0 + t) * G + c0 + gl] = s;
        }
        if (tid < ET * gc) {
            const int el = my_el, gl = my_gl;
            if (el < ne) {
                if (c0 > 0) {
                    const uint32_t *q = a.rw + (size_t)(e0 + el) * (D / 4) + (size_t)(c0 + gl) * 16;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        qv[j] = ldg_u4(q + 4 * j);
                }
                float P[TT];
#pragma unroll
                for (int t = 0; t < TT; ++t)
                    P[t] = 0.0f;
                const float *xr = xs + gl * kXPad;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t w = (j % 4 == 0) ? qv[j / 4].x : (j % 4 == 1) ? qv[j / 4].y
                                     : (j % 4 == 2) ? qv[j / 4].z : qv[j / 4].w;
                    const float q0 = byte_f<0>(w), q1 = byte_f<1>(w), q2 = byte_f<2>(w), q3 = byte_f<3>(w);
#pragma unroll
                    for (int t = 0; t < TT; ++t) {
                        if (t < nt) {
                            const float4 xv = *reinterpret_cast<const float4 *>(xr + t * GC * kXPad + 4 * j);
                            P[t] = fmaf(q0, xv.x, P[t]);
                            P[t] = fmaf(q1, xv.y, P[t]);
                            P[t] = fmaf(q2, xv.z, P[t]);
                            P[t] = fmaf(q3, xv.w, P[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < TT; ++t)
                    if (t < nt)
                        Ps[(t * ET + el) * GC + gl] = P[t];
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kAcc; ++i) {
            const int p = tid + i * kThreads;
            if (p < npairs) {
                const int t = p / ne, el = p % ne;
                float v = acc[i];
                for (int gb = 0; gb < gc; gb += 8) {
                    float ps[8], xs8[8], ss8[8], bs8[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int gl = min(gb + j, gc - 1), g = c0 + gl;
                        ss8[j] = sS[el * G + g];
                        bs8[j] = sB[el * G + g];
                        ps[j] = Ps[(t * ET + el) * GC + gl];
                        xs8[j] = Xs[t * G + g];
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (gb + j < gc) {
                            v = fmaf(ss8[j], ps[j], v);
                            v = fmaf(bs8[j], xs8[j], v);
                        }
                    }
                }
                acc[i] = v;
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < kAcc; ++i) {
        const int p = tid + i * kThreads;
        if (p < npairs) {
            const int t = p / ne, el = p % ne;
            a.logits[(size_t)(t0 + t) * E + e0 + el] = acc[i];
        }
    }

    if (a.cluster) {
        // Deliver this CTA's logits to CTA 0 of the cluster (distributed shared
        // memory), then CTA 0 routes all T tokens and publishes the result.
        float *gather = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(sm) + RL.off_gather);
#pragma unroll
        for (int i = 0; i < kAcc; ++i) {
            const int p = tid + i * kThreads;
            if (p < npairs) {
                const int t = p / ne, el = p % ne;
                uint32_t remote;
                asm volatile("mapa.shared::cluster.u32 %0, %1, 0;"
                             : "=r"(remote)
                             : "r"(smem_u32(gather + t * E + e0 + el)));
                asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(acc[i]) : "memory");
            }
        }
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
        if (blockIdx.x != 0)
            return;
        const CtaRoute rt = cta_route_carve(reinterpret_cast<uint8_t *>(sm) + RL.off_route, a.T, E, a.K);
        cta_route(gather, a.T, E, a.K, a.pes, rt, RouteSync{});
        const int tk = a.T * a.K;
        for (int i = tid; i < tk; i += kThreads) {
            a.topk_idx[i] = rt.topk_idx[i];
            a.topk_w[i] = rt.topk_w[i];
            a.perm[i] = rt.perm[i];
        }
        for (int e = tid; e < E; e += kThreads) {
            a.counts[e] = rt.cnt[e];
            a.offsets[e] = rt.off[e];
        }
        const int nt_tiles = *rt.n_tiles;
        for (int i = tid; i < 3 * nt_tiles; i += kThreads)
            a.tiles[i] = rt.tiles[i];
        if (tid == 0) {
            a.offsets[E] = rt.off[E];
            *a.n_tiles = nt_tiles;
        }
        return;
    }
    if (a.logits_only)
        return;
    // last expert tile of this token tile: top-k
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&a.tickets[blockIdx.y], 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    if (tid == 0)
        a.tickets[blockIdx.y] = 0u;
    topk_tokens(a, t0, nt, sm);

    // last token tile: grouping of all slots
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&a.tickets[gridDim.y], 1u);
        s_last = (prev == gridDim.y - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    if (tid == 0)
        a.tickets[gridDim.y] = 0u;
    group_slots(a, sm);
}

template <int TT>
cudaError_t launch_tt(const RouteArgs &a, const RouteLaunch &L, cudaStream_t s)
{
    auto k = route_kernel<TT>;
    {
        cudaError_t e = smem_optin(reinterpret_cast<const void *>(k), L.smem);
        if (e != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.n_et, L.n_tt);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (L.cluster) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = L.n_et;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, k, a, L);
}

// ---------------------------------------------------------------- large T
//
// For many tokens the logits are a batched product: a register-tiled kernel
// computes a 64-token x 64-expert block, one group of 64 columns at a time.
// Every (token, expert) accumulator still follows the fixed order of the
// header -- within a group an fma chain over the 64 columns in ascending
// order, then acc = fma(s, P, acc), acc = fma(b, X, acc), groups ascending --
// so the logits equal the small-T kernel's bit for bit.  The activations come
// from the prefill gather: FP16 rows scaled by a power of two per token (exact
// for the BF16 values), in operand column order, and their per-group sums in
// the fixed add order.

constexpr int kLE = 64;  // experts per block

// The router's bytes as floats, once per call: QF[(g * 64 + c) * Ep + e] =
// q[e][64 g + c] (Ep = E rounded up to 64, zero padding), so a block's 64 x 64
// tile of one group is 64 rows of 256 contiguous bytes.
__global__ void __launch_bounds__(256) router_to_f32(const uint32_t *__restrict__ rw, int E, int Ep, int D,
                                                     float *__restrict__ QF)
{
    const int wi = blockIdx.x, e = blockIdx.y * 256 + threadIdx.x;  // packed word column, expert
    if (e >= Ep)
        return;
    const uint32_t w = e < E ? __ldg(rw + (size_t)e * (D / 4) + wi) : 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b)
        QF[(size_t)(4 * wi + b) * Ep + e] = (float)((w >> (8 * b)) & 0xFFu);
}

// Block of TT tokens x 64 experts, 256 threads: thread (ty, tx) of 16 x 16
// holds tokens ty*TM .. ty*TM + TM - 1 (TM = TT/16) and experts 4tx .. 4tx+3,
// TM x 4 accumulators.  Each group of 64 columns is staged in shared memory
// (double-buffered; the next group's activations and router floats are loaded
// into registers while the current one is multiplied), so one barrier per
// group separates the buffers.
template <int TT>
__global__ void __launch_bounds__(256, 1) logits_gemm(const __half *__restrict__ X16, const float *__restrict__ xsc,
                                                    const float *__restrict__ XG, const float *__restrict__ QF,
                                                    const uint16_t *__restrict__ rs, const uint16_t *__restrict__ rb,
                                                    int T, int D, int E, int Ep, float *__restrict__ logits,
                                                    const uint16_t *__restrict__ rsc, float rcoef)
{
    constexpr int NT = 256, TM = TT / 16;
    constexpr int XV = TT * 8 / NT;             // 16-byte activation vectors per thread per group
    constexpr int QV = 64 * kLE / 4 / NT;       // 16-byte router vectors per thread per group (= 4)
    static_assert(XV >= 1 && XV * NT == TT * 8 && QV * NT * 4 == 64 * kLE && TM % 2 == 0, "tile shape");
    extern __shared__ __align__(16) float lsm[];
    float *xs0 = lsm;                           // [2][64][TT]   [column][token]
    float *qs0 = xs0 + 2 * 64 * TT;             // [2][64][kLE]  [column][expert]
    float *sS0 = qs0 + 2 * 64 * kLE;            // [2][kLE]
    float *sB0 = sS0 + 2 * kLE;                 // [2][kLE]
    float *sX0 = sB0 + 2 * kLE;                 // [2][TT]
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int t0 = blockIdx.y * TT, e0 = blockIdx.x * kLE, G = D / 64;
    uint4 xr[XV], qr[QV];
    float xscale[XV];
    // activations: vector v of thread tid is 8-column chunk ch of token t, with
    // consecutive threads on consecutive tokens (conflict-free stores below)
    auto fetch = [&](int g) {
#pragma unroll
        for (int v = 0; v < XV; ++v) {
            const int i = tid + v * NT, t = i % TT, ch = i / TT, tt = t0 + t;
            xr[v] = tt < T ? __ldg(reinterpret_cast<const uint4 *>(X16 + (size_t)tt * D + 64 * g) + ch)
                           : make_uint4(0, 0, 0, 0);
            xscale[v] = tt < T ? __ldg(xsc + tt) : 0.f;
        }
#pragma unroll
        for (int v = 0; v < QV; ++v) {
            const int i = tid + v * NT, c = i >> 4, e4 = i & 15;
            qr[v] = __ldg(reinterpret_cast<const uint4 *>(QF + (size_t)(64 * g + c) * Ep + e0) + e4);
        }
    };
    // registers -> shared buffer b: activations back in column order (operand
    // position p of an 8-block holds column [0,4,1,5,2,6,3,7][p])
    auto stage = [&](int g, int b) {
        float *xs = xs0 + b * 64 * TT, *qs = qs0 + b * 64 * kLE;
#pragma unroll
        for (int v = 0; v < XV; ++v) {
            const int i = tid + v * NT, t = i % TT, ch = i / TT;
            const uint32_t u[4] = {xr[v].x, xr[v].y, xr[v].z, xr[v].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 h = *reinterpret_cast<const __half2 *>(&u[j]);
                const float2 f = __half22float2(h);
                float a0 = f.x * xscale[v], a1 = f.y * xscale[v];
                if (rsc) {  // the router's input (x_i * rsc_i) * rcoef
                    a0 = __fmul_rn(__fmul_rn(a0, bf2f(__ldg(rsc + 64 * g + 8 * ch + j))), rcoef);
                    a1 = __fmul_rn(__fmul_rn(a1, bf2f(__ldg(rsc + 64 * g + 8 * ch + j + 4))), rcoef);
                }
                xs[(8 * ch + j) * TT + t] = a0;      // operand position 2j   -> column j
                xs[(8 * ch + j + 4) * TT + t] = a1;  // operand position 2j+1 -> column j+4
            }
        }
#pragma unroll
        for (int v = 0; v < QV; ++v) {
            const int i = tid + v * NT, c = i >> 4, e4 = i & 15;
            *reinterpret_cast<uint4 *>(qs + c * kLE + 4 * e4) = qr[v];
        }
        if (tid < kLE) {
            const int ee = e0 + tid;
            sS0[b * kLE + tid] = ee < E ? bf2f(__ldg(rs + (size_t)ee * G + g)) : 0.f;
            sB0[b * kLE + tid] = ee < E ? bf2f(__ldg(rb + (size_t)ee * G + g)) : 0.f;
        }
        if (tid < TT) {
            const int tt = t0 + tid;
            sX0[b * TT + tid] = tt < T ? __ldg(XG + (size_t)tt * G + g) : 0.f;
        }
    };
    float acc[TM][4];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[i][j] = 0.f;
    fetch(0);
    stage(0, 0);
    if (G > 1)
        fetch(1);
    __syncthreads();
    for (int g = 0; g < G; ++g) {
        const int b = g & 1;
        const float *xs = xs0 + b * 64 * TT, *qs = qs0 + b * 64 * kLE;
        // P[i][j] for token pairs (i, i + 1): one packed two-lane fma per
        // pair and expert, each lane an IEEE fma like fmaf (the same chain)
        uint64_t P2[TM / 2][4];
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                P2[i][j] = 0ull;
#pragma unroll 8
        for (int c = 0; c < 64; ++c) {
            uint64_t xp[TM / 2];
#pragma unroll
            for (int i = 0; i < TM / 2; ++i)
                xp[i] = *reinterpret_cast<const uint64_t *>(xs + c * TT + ty * TM + 2 * i);
            const float4 qv = *reinterpret_cast<const float4 *>(qs + c * kLE + 4 * tx);
            const uint64_t qd[4] = {pair_f32(qv.x, qv.x), pair_f32(qv.y, qv.y), pair_f32(qv.z, qv.z),
                                    pair_f32(qv.w, qv.w)};
#pragma unroll
            for (int i = 0; i < TM / 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    fma_f32x2(P2[i][j], qd[j], xp[i]);
        }
        float P[TM][4];
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                unpair_f32(P2[i][j], P[2 * i][j], P[2 * i + 1][j]);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[i][j] = fmaf(sS0[b * kLE + 4 * tx + j], P[i][j], acc[i][j]);
                acc[i][j] = fmaf(sB0[b * kLE + 4 * tx + j], sX0[b * TT + ty * TM + i], acc[i][j]);
            }
        // the other buffer was last read in group g - 1, before the barrier
        // that ended it: stage group g + 1 there, then fetch group g + 2
        if (g + 1 < G) {
            stage(g + 1, b ^ 1);
            if (g + 2 < G)
                fetch(g + 2);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int tt = t0 + ty * TM + i;
        if (tt >= T)
            continue;
        const int ee = e0 + 4 * tx;
        if ((E & 3) == 0 && ee + 3 < E) {
            *reinterpret_cast<float4 *>(logits + (size_t)tt * E + ee) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (ee + j < E)
                    logits[(size_t)tt * E + ee + j] = acc[i][j];
        }
    }
}

template <int TT>
constexpr size_t logits_smem()
{
    return (size_t)(2 * 64 * TT + 2 * 64 * kLE + 4 * kLE + 2 * TT) * sizeof(float);
}

// Few tokens (up to kPartT): the per-group dot products P[g][t][e] of every
// group in its own block (grid: expert tiles x token tiles x groups), then
// logits_sum adds them in the fixed order.  Each P is the same chain as in
// logits_gemm, so the logits are the same bit for bit; the grid has G times
// more blocks.
constexpr int kPartT = 512;

__global__ void __launch_bounds__(256) logits_part(const __half *__restrict__ X16, const float *__restrict__ xsc,
                                                   const float *__restrict__ QF, int T, int D, int E, int Ep,
                                                   const uint16_t *__restrict__ rsc, float rcoef,
                                                   float *__restrict__ P)
{
    constexpr int TT = 32, TM = 2, NT = 256;
    __shared__ __align__(16) float xs[64 * TT];   // [column][token]
    __shared__ __align__(16) float qs[64 * kLE];  // [column][expert]
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int t0 = blockIdx.y * TT, e0 = blockIdx.x * kLE, g = blockIdx.z;
    {
        // activations: thread tid = 8-column chunk ch of token t (one 16-byte load)
        const int t = tid % TT, ch = tid / TT, tt = t0 + t;
        const uint4 xr = tt < T ? __ldg(reinterpret_cast<const uint4 *>(X16 + (size_t)tt * D + 64 * g) + ch)
                                : make_uint4(0, 0, 0, 0);
        const float xscale = tt < T ? __ldg(xsc + tt) : 0.f;
        const uint32_t u[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&u[j]);
            const float2 f = __half22float2(h);
            float a0 = f.x * xscale, a1 = f.y * xscale;
            if (rsc) {
                a0 = __fmul_rn(__fmul_rn(a0, bf2f(__ldg(rsc + 64 * g + 8 * ch + j))), rcoef);
                a1 = __fmul_rn(__fmul_rn(a1, bf2f(__ldg(rsc + 64 * g + 8 * ch + j + 4))), rcoef);
            }
            xs[(8 * ch + j) * TT + t] = a0;
            xs[(8 * ch + j + 4) * TT + t] = a1;
        }
#pragma unroll
        for (int v = 0; v < 64 * kLE / 4 / NT; ++v) {
            const int i = tid + v * NT, c = i >> 4, e4 = i & 15;
            *reinterpret_cast<uint4 *>(qs + c * kLE + 4 * e4) =
                __ldg(reinterpret_cast<const uint4 *>(QF + (size_t)(64 * g + c) * Ep + e0) + e4);
        }
    }
    __syncthreads();
    uint64_t P2[TM / 2][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        P2[0][j] = 0ull;
#pragma unroll 8
    for (int c = 0; c < 64; ++c) {
        const uint64_t xp = *reinterpret_cast<const uint64_t *>(xs + c * TT + ty * TM);
        const float4 qv = *reinterpret_cast<const float4 *>(qs + c * kLE + 4 * tx);
        fma_f32x2(P2[0][0], pair_f32(qv.x, qv.x), xp);
        fma_f32x2(P2[0][1], pair_f32(qv.y, qv.y), xp);
        fma_f32x2(P2[0][2], pair_f32(qv.z, qv.z), xp);
        fma_f32x2(P2[0][3], pair_f32(qv.w, qv.w), xp);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float p0, p1;
        unpair_f32(P2[0][j], p0, p1);
        const int ee = e0 + 4 * tx + j, tt = t0 + ty * TM;
        if (ee < E) {
            if (tt < T)
                P[((size_t)g * T + tt) * E + ee] = p0;
            if (tt + 1 < T)
                P[((size_t)g * T + tt + 1) * E + ee] = p1;
        }
    }
}

__global__ void __launch_bounds__(256) logits_sum(const float *__restrict__ P, const uint16_t *__restrict__ rs,
                                                  const uint16_t *__restrict__ rb, const float *__restrict__ XG,
                                                  int T, int E, int G, float *__restrict__ logits)
{
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= T * E)
        return;
    const int t = i / E, e = i - t * E;
    float acc = 0.f;
    for (int g = 0; g < G; ++g) {
        acc = fmaf(bf2f(__ldg(rs + (size_t)e * G + g)), __ldg(P + ((size_t)g * T + t) * E + e), acc);
        acc = fmaf(bf2f(__ldg(rb + (size_t)e * G + g)), __ldg(XG + (size_t)t * G + g), acc);
    }
    logits[i] = acc;
}

// Top-k + softmax of 8 tokens per block (one warp per token), from the logits.
__global__ void __launch_bounds__(kThreads) topk_kernel(const RouteArgs a)
{
    extern __shared__ __align__(16) float sm[];
    const int t0 = blockIdx.x * kWarps;
    topk_tokens(a, t0, min(kWarps, a.T - t0), sm);
}

// Grouping of many slots by expert over several blocks (the order of
// group_slots: ascending expert, ascending slot within an expert).  Block b
// takes slots [b kGrpSlots, (b + 1) kGrpSlots); its warp w the w-th quarter.
//   group_count    per-block expert counts bc[b][e]
//   group_scan     counts, offsets, and each block's base bb[b][e] within
//                  its expert (exclusive over blocks)
//   group_scatter  each warp ranks its slots (32 at a time, in order) and
//                  writes perm[offsets[e] + bb[b][e] + (earlier warps' and
//                  rows' count) + rank]
constexpr int kGrpSlots = 1024, kGrpWarps = 4;

__global__ void __launch_bounds__(32 * kGrpWarps) group_count(const int32_t *__restrict__ idx, int n, int E,
                                                              int32_t *__restrict__ bc)
{
    extern __shared__ int h[];  // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        h[e] = 0;
    __syncthreads();
    const int lo = blockIdx.x * kGrpSlots, hi = min(n, lo + kGrpSlots);
    for (int s = lo + threadIdx.x; s < hi; s += blockDim.x)
        atomicAdd(&h[__ldg(idx + s)], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        bc[(size_t)blockIdx.x * E + e] = h[e];
}

__global__ void __launch_bounds__(1024) group_scan(const int32_t *__restrict__ bc, int nb, int E,
                                                   int32_t *__restrict__ bb, int32_t *__restrict__ counts,
                                                   int32_t *__restrict__ offsets)
{
    __shared__ int cnt[kMaxExperts + 1];
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int b = 0; b < nb; ++b) {
            bb[(size_t)b * E + e] = run;
            run += bc[(size_t)b * E + e];
        }
        cnt[e] = run;
        counts[e] = run;
    }
    __syncthreads();
    // exclusive scan of cnt over the experts (E <= 1024: one value per thread)
    const int v = tid < E ? cnt[tid] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int w = lane < nw ? wsum[lane] : 0, wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o)
                wi += y;
        }
        wsum[lane] = wi - w;
    }
    __syncthreads();
    const int ex = incl - v + wsum[warp];
    if (tid < E)
        offsets[tid] = ex;
    if (tid == E - 1)
        offsets[E] = ex + v;
}

__global__ void __launch_bounds__(32 * kGrpWarps) group_scatter(const int32_t *__restrict__ idx, int n, int E,
                                                                const int32_t *__restrict__ bb,
                                                                const int32_t *__restrict__ offsets,
                                                                int32_t *__restrict__ perm)
{
    extern __shared__ int wb[];  // [kGrpWarps][E]: counts, then running positions
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int per = kGrpSlots / kGrpWarps;
    const int lo = min(n, blockIdx.x * kGrpSlots + warp * per), hi = min(n, lo + per);
    for (int i = threadIdx.x; i < kGrpWarps * E; i += blockDim.x)
        wb[i] = 0;
    __syncthreads();
    int *mine = wb + warp * E;
    for (int s0 = lo; s0 < hi; s0 += 32) {
        const int s = s0 + lane, e = s < hi ? __ldg(idx + s) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(m) - 1)
            mine[e] += __popc(m);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = __ldg(offsets + e) + __ldg(bb + (size_t)blockIdx.x * E + e);
        for (int w = 0; w < kGrpWarps; ++w) {
            const int c = wb[w * E + e];
            wb[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int s0 = lo; s0 < hi; s0 += 32) {
        const int s = s0 + lane, e = s < hi ? __ldg(idx + s) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        if (e >= 0)
            perm[mine[e] + __popc(m & lt)] = s;
        __syncwarp();
        if (e >= 0 && lane == __ffs(m) - 1)
            mine[e] += __popc(m);
        __syncwarp();
    }
}


} // namespace

RouteLaunch route_plan(int T, int D, int E, int K)
{
    RouteLaunch L{};
    const int G = D / kGroup;
    if (T <= 1)
        L.TT = 1;
    else if (T <= 4)
        L.TT = 4;
    else if (T <= 128)
        L.TT = 8;
    else
        L.TT = 32;
    L.cluster = T <= kClusterTokens;
    if (L.cluster) {
        // one cluster: the experts split over kClusterCtas CTAs
        int et = (E + kClusterCtas - 1) / kClusterCtas;
        L.ET = et;
        int gc = kThreads / et;
        L.GC = gc < 1 ? 1 : (gc > G ? G : gc);
    } else {
        if (L.TT <= 4)
            L.GC = G;
        else if (L.TT == 8)
            L.GC = G < 32 ? G : 32;
        else
            L.GC = G < 8 ? G : 8;
        int et = kThreads / L.GC;
        if (et * L.TT > 1024)
            et = 1024 / L.TT;
        if (et > E)
            et = E;
        if (et < 1)
            et = 1;
        L.ET = et;
    }
    L.n_tt = (T + L.TT - 1) / L.TT;
    L.n_et = (E + L.ET - 1) / L.ET;
    const size_t main_f = (size_t)L.TT * L.GC * kXPad + (size_t)L.TT * L.ET * L.GC + (size_t)L.TT * G +
                          2 * (size_t)L.ET * G + L.TT;
    const size_t topk_f = (size_t)kWarps * E + (size_t)kWarps * ((E + 31) / 32);
    const size_t group_f = 2 * (size_t)kWarps * E + 3 * (size_t)E;
    size_t f = main_f;
    if (!L.cluster) {
        if (topk_f > f)
            f = topk_f;
        if (group_f > f)
            f = group_f;
    }
    size_t bytes = ((f * sizeof(float)) + 127) & ~size_t(127);
    if (L.cluster) {
        L.off_gather = bytes;
        bytes += (((size_t)T * E * sizeof(float)) + 127) & ~size_t(127);
        L.off_route = bytes;
        bytes += cta_route_bytes(T, E, K);
    }
    L.smem = bytes;
    return L;
}

cudaError_t launch_route(const RouteArgs &a, const RouteLaunch &L, cudaStream_t s)
{
    switch (L.TT) {
    case 1: return launch_tt<1>(a, L, s);
    case 4: return launch_tt<4>(a, L, s);
    case 8: return launch_tt<8>(a, L, s);
    default: return launch_tt<32>(a, L, s);
    }
}

size_t route_f32_bytes(int T, int D, int E, int K)
{
    // the router's bytes as floats, then the per-group products of up to
    // kPartT tokens (reserved for every T, so that the size grows with T)
    const size_t qf = (size_t)D * ((E + kLE - 1) / kLE * kLE) + (size_t)(D / 64) * (T < kPartT ? T : kPartT) * E;
    const size_t nb = ((size_t)T * K + kGrpSlots - 1) / kGrpSlots;
    const size_t grp = 2 * nb * (size_t)E;
    return (qf > grp ? qf : grp) * sizeof(float);
}

cudaError_t launch_route_large(const RouteArgs &a, const void *X16, const float *xsc, const float *XG, float *QF,
                               cudaStream_t s)
{
    const int ne = (a.E + kLE - 1) / kLE, Ep = ne * kLE;
    router_to_f32<<<dim3(a.D / 4, (Ep + 255) / 256), 256, 0, s>>>(a.rw, a.E, Ep, a.D, QF);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    // the largest token block that still gives most SMs a block
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        sms = 148;
    auto run = [&](auto tt_tag) -> cudaError_t {
        constexpr int TT = decltype(tt_tag)::value;
        auto k = logits_gemm<TT>;
        const size_t smem = logits_smem<TT>();
        cudaError_t r = smem_optin(reinterpret_cast<const void *>(k), smem);
        if (r != cudaSuccess)
            return r;
        k<<<dim3(ne, (a.T + TT - 1) / TT), 256, smem, s>>>(static_cast<const __half *>(X16), xsc, XG, QF, a.rs,
                                                            a.rb, a.T, a.D, a.E, Ep, a.logits, a.router_scale,
                                                            a.rcoef);
        return cudaGetLastError();
    };
    const long long need = (long long)sms * 4 / 5;
    if (a.T <= kPartT) {
        const int G = a.D / 64;
        float *P = QF + (size_t)a.D * Ep;
        logits_part<<<dim3(ne, (a.T + 31) / 32, G), 256, 0, s>>>(static_cast<const __half *>(X16), xsc, QF, a.T,
                                                                 a.D, a.E, Ep, a.router_scale, a.rcoef, P);
        if ((e = cudaGetLastError()) == cudaSuccess) {
            logits_sum<<<(a.T * a.E + 255) / 256, 256, 0, s>>>(P, a.rs, a.rb, XG, a.T, a.E, G, a.logits);
            e = cudaGetLastError();
        }
    } else if ((long long)ne * ((a.T + 127) / 128) >= need)
        e = run(std::integral_constant<int, 128>{});
    else if ((long long)ne * ((a.T + 63) / 64) >= need)
        e = run(std::integral_constant<int, 64>{});
    else
        e = run(std::integral_constant<int, 32>{});
    if (e != cudaSuccess)
        return e;
    const size_t topk_smem = ((size_t)kWarps * a.E + (size_t)kWarps * ((a.E + 31) / 32)) * sizeof(float);
    topk_kernel<<<(a.T + kWarps - 1) / kWarps, kThreads, topk_smem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    // grouping over several blocks; its block counts reuse QF (the logits are done)
    const int n = a.T * a.K, nb = (n + kGrpSlots - 1) / kGrpSlots;
    int32_t *bc = reinterpret_cast<int32_t *>(QF), *bb = bc + (size_t)nb * a.E;
    group_count<<<nb, 32 * kGrpWarps, a.E * sizeof(int), s>>>(a.topk_idx, n, a.E, bc);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    group_scan<<<1, 1024, 0, s>>>(bc, nb, a.E, bb, a.counts, a.offsets);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    group_scatter<<<nb, 32 * kGrpWarps, kGrpWarps * a.E * sizeof(int), s>>>(a.topk_idx, n, a.E, bb, a.offsets,
                                                                            a.perm);
    return cudaGetLastError();
}

} // namespace mx

// mx_cta_route.cuh -- top-k, softmax and grouping of token/expert pairs,
// computed by one CTA's consumer warps into shared memory.
//
// "Mference System design" page, section "Decode": top8 = highest_8(logits),
// weights = softmax(logits[top8]) * per_expert_scale[top8]; section "Prefill":
// token/expert pairs are grouped into bounded per-expert work.
//
// The router runs this once per layer: for a few tokens in CTA 0 of a thread-
// block cluster whose CTAs deliver their logits over distributed shared memory.
// Order: descending logit, ties to the lower expert index, NaN ranks as -inf;
// slots s = t*K + k grouped by expert, ascending s within an expert; one tile
// per (expert, up to kTileTokens slots).
#pragma once

#include "mx_common.cuh"
#include "mx_internal.h"

#include <climits>

namespace mx {

constexpr int kRouteWarps = 8;   // the routine runs on 8 warps (256 threads)
constexpr int kRankTokens = 16;  // tokens ranked per pass (bounds the scratch)

// Shared-memory arrays of the routing result.
struct CtaRoute {
    int *topk_idx;  // [T*K]
    float *topk_w;  // [T*K]
    int *cnt;       // [E]
    int *off;       // [E+1]
    int *perm;      // [T*K]
    int *tiles;     // [3][max tiles] (expert, begin, end)
    int *n_tiles;   // [1]
    int *scratch;   // max(min(T, kRankTokens)*E, 2*kRouteWarps*E + E) words
};

// Bytes of shared memory the routine needs for T tokens.
__host__ __device__ inline size_t cta_route_bytes(int T, int E, int K)
{
    const size_t tk = (size_t)T * K;
    const size_t sel = (size_t)(T < kRankTokens ? T : kRankTokens) * E;
    const size_t grp = 2 * (size_t)kRouteWarps * E + E;
    const size_t max_tiles = (size_t)E + tk / kTileTokens + 1;
    return 4 * (tk * 3 + (size_t)E + (E + 1) + 3 * max_tiles + 1 + (sel > grp ? sel : grp));
}

__device__ inline CtaRoute cta_route_carve(void *base, int T, int E, int K)
{
    int *p = static_cast<int *>(base);
    const int tk = T * K, max_tiles = E + tk / kTileTokens + 1;
    CtaRoute r;
    r.topk_idx = p;
    p += tk;
    r.topk_w = reinterpret_cast<float *>(p);
    p += tk;
    r.perm = p;
    p += tk;
    r.cnt = p;
    p += E;
    r.off = p;
    p += E + 1;
    r.tiles = p;
    p += 3 * max_tiles;
    r.n_tiles = p;
    p += 1;
    r.scratch = p;
    return r;
}

// Run by threads 0..255 (8 warps) of the CTA; `sync` synchronises exactly them.
// logits: [T][E], in this CTA's shared memory or in global memory written
// before a barrier that orders it with this CTA.
template <typename Sync>
__device__ void cta_route(const float *logits, int T, int E, int K, const float *pes, const CtaRoute &r, Sync sync)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // ---- top-k by rank: the rank of logit e of token t is the number of
    // logits ahead of it (larger, or equal with a lower index); the top-k are
    // the ranks below K, in rank order.  One thread per (t, e); no sequential
    // rounds.
    for (int t0 = 0; t0 < T; t0 += kRankTokens) {
        const int nt = min(kRankTokens, T - t0);
        float *lg = reinterpret_cast<float *>(r.scratch);  // [nt][E]
        for (int i = threadIdx.x; i < nt * E; i += 32 * kRouteWarps) {
            const float v = logits[(size_t)t0 * E + i];
            lg[i] = isnan(v) ? -INFINITY : v;
        }
        sync();
        for (int i = threadIdx.x; i < nt * E; i += 32 * kRouteWarps) {
            const int tl = i / E, e = i - tl * E, t = t0 + tl;
            const float *row = lg + tl * E;
            const float v = row[e];
            int rank = 0;
            for (int j = 0; j < E; ++j) {
                const float u = row[j];
                rank += (u > v) || (u == v && j < e);
            }
            if (rank < K) {
                r.topk_idx[t * K + rank] = e;
                r.topk_w[t * K + rank] = v;  // the logit, turned into a weight below
            }
        }
        sync();
    }
    {
        // softmax over the selected logits of each token, shifted by the largest
        for (int t = threadIdx.x; t < T; t += 32 * kRouteWarps) {
            float *w = r.topk_w + t * K;
            const float m = w[0];
            float sum = 0.0f;
            for (int k = 0; k < K; ++k) {
                w[k] = expf(w[k] - m);
                sum += w[k];
            }
            for (int k = 0; k < K; ++k) {
                float x = w[k] / sum;
                if (pes)
                    x = x * __ldg(pes + r.topk_idx[t * K + k]);
                w[k] = x;
            }
        }
    }
    sync();
    // ---- grouping: per-warp counts, scans, stable scatter
    const int n = T * K;
    int *wc = r.scratch;                 // [8][E]
    int *base = wc + kRouteWarps * E;    // [8][E]
    int *tix = base + kRouteWarps * E;   // [E]
    for (int i = threadIdx.x; i < kRouteWarps * E; i += 32 * kRouteWarps)
        wc[i] = 0;
    sync();
    const int chunk = (n + kRouteWarps - 1) / kRouteWarps;
    const int lo = min(n, warp * chunk), hi = min(n, lo + chunk);
    for (int s0 = lo; s0 < hi; s0 += 32) {
        const int s = s0 + lane;
        const int e = (s < hi) ? r.topk_idx[s] : -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(m) - 1)
            wc[warp * E + e] += __popc(m);
        __syncwarp();
    }
    sync();
    for (int e = threadIdx.x; e < E; e += 32 * kRouteWarps) {
        int run = 0;
        for (int w = 0; w < kRouteWarps; ++w) {
            base[w * E + e] = run;
            run += wc[w * E + e];
        }
        r.cnt[e] = run;
    }
    sync();
    if (warp == 0) {
        const int per = (E + 31) / 32, e_lo = lane * per, e_hi = min(E, e_lo + per);
        int sc = 0, st = 0;
        for (int e = e_lo; e < e_hi; ++e) {
            sc += r.cnt[e];
            st += (r.cnt[e] + kTileTokens - 1) / kTileTokens;
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
            r.off[e] = oc;
            tix[e] = os;
            oc += r.cnt[e];
            os += (r.cnt[e] + kTileTokens - 1) / kTileTokens;
        }
        if (lane == 31) {
            r.off[E] = ic;
            *r.n_tiles = is;
        }
    }
    sync();
    const unsigned lt = (1u << lane) - 1u;
    for (int s0 = lo; s0 < hi; s0 += 32) {
        const int s = s0 + lane;
        const int e = (s < hi) ? r.topk_idx[s] : -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        if (e >= 0)
            r.perm[r.off[e] + base[warp * E + e] + __popc(m & lt)] = s;
        __syncwarp();
        if (e >= 0 && lane == __ffs(m) - 1)
            base[warp * E + e] += __popc(m);
        __syncwarp();
    }
    for (int e = threadIdx.x; e < E; e += 32 * kRouteWarps) {
        int t = tix[e];
        for (int b = 0; b < r.cnt[e]; b += kTileTokens, ++t) {
            r.tiles[3 * t + 0] = e;
            r.tiles[3 * t + 1] = r.off[e] + b;
            r.tiles[3 * t + 2] = r.off[e] + min(b + kTileTokens, r.cnt[e]);
        }
    }
    sync();
}

} // namespace mx

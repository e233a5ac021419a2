// mx_ffn_decode.cu -- routed + shared expert FFN for small token counts
// (decode, T <= 64 per pass).
//
// "Mference System design" page, section "Metal execution": decode consumes the
// packed values, BF16 scales and BF16 biases directly, and the routed kernels
// fuse affine decode, GeGLU and the weighted expert reduction; section
// "Decode" (cb2 row): the routed top-k branch is reduced with the router
// weights, combined with the shared branch, and scaled by the layer scalar.
//
// Two weight-streaming kernels, two CTAs per SM.  In each CTA one producer warp
// moves blocks of packed weight rows from HBM into a ring of shared-memory
// stages with TMA tensor copies (one copy per block of rows, laid out
// group-major by the tensor map, mx_tma.cu) plus small bulk copies of their
// BF16 scales and biases, completing on an mbarrier per stage; eight consumer
// warps run the math out of shared memory and hand each stage back through an
// "empty" mbarrier.  The routing (top-k, weights, grouping of slots by expert)
// comes from the router kernel.
//   gateup_kernel  persistent.  Work item = 8 hidden units of one expert tile
//                  (or of the shared expert): their 8 gate rows and 8 up rows
//                  form the 16 rows of one m16n8k16 A tile, so gelu(g) * u is
//                  lane-local.  h is written as a BF16 hi/lo pair.
//   down_kernel    one CTA per 16 output rows of D; units = the shared down
//                  rows, then each routed tile's down rows; the CTA reduces
//                  them in a fixed order: out = residual + lambda * (shared +
//                  sum_k w_k y_k).  No atomics, so the result is deterministic
//                  ("Correctness and safety invariants": reordered float
//                  kernels stay deterministic within a path).
// Both launch as programmatic dependents: weights that do not depend on the
// previous kernel are requested before waiting for it.
//
// Math per group of 64 columns: A holds 128 + q as exact BF16 integers (one
// mask-and-or per pair of nibbles), so the MMA returns R = 128 X + P with
// P = sum q*x; with X = sum x, acc += s*R + (b - 128 s)*X = s*P + b*X in fp32,
// which is the dequantized dot product sum (s*q + b)*x.  Gate/up reads X from
// the router kernel's per-group sums of x; the down kernel gets X from an MMA
// against an all-ones A, and holds the hi/lo BF16 parts of h as two columns
// of the same MMA.  Legacy warp MMAs suffice: this path is bound by HBM, and
// register accumulators make the per-group affine step exact and cheap.
#include "mx_common.cuh"
#include "mx_internal.h"

#include <mutex>

namespace mx {

namespace {

constexpr int kCW = 8;                    // consumer warps
constexpr int kThreads = (kCW + 1) * 32;  // + one producer warp
constexpr int kConsumers = kCW * 32;
constexpr uint32_t kOnes = 0x3F803F80u;   // BF16x2 (1.0, 1.0)
constexpr int kBarBytes = 256;            // mbarriers at the start of dynamic smem

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                 "%3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
                 "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
                 : "memory");
}

// 128 + (nibbles j and j+4 of w) as a BF16x2 pair of exact integers.
template <int J>
__device__ __forceinline__ uint32_t nib_pair128(uint32_t w)
{
    return ((w >> (4 * J)) & 0x000F000Fu) | 0x43004300u;
}

__device__ __forceinline__ void build_a(uint2 q0, uint2 q8, uint32_t (&A)[4][4])
{
    // k-step s uses word s/2 of the lane's pair, nibble pairs (j, j+4) and (j+1, j+5), j = 2*(s&1)
    A[0][0] = nib_pair128<0>(q0.x); A[0][1] = nib_pair128<0>(q8.x);
    A[0][2] = nib_pair128<1>(q0.x); A[0][3] = nib_pair128<1>(q8.x);
    A[1][0] = nib_pair128<2>(q0.x); A[1][1] = nib_pair128<2>(q8.x);
    A[1][2] = nib_pair128<3>(q0.x); A[1][3] = nib_pair128<3>(q8.x);
    A[2][0] = nib_pair128<0>(q0.y); A[2][1] = nib_pair128<0>(q8.y);
    A[2][2] = nib_pair128<1>(q0.y); A[2][3] = nib_pair128<1>(q8.y);
    A[3][0] = nib_pair128<2>(q0.y); A[3][1] = nib_pair128<2>(q8.y);
    A[3][2] = nib_pair128<3>(q0.y); A[3][3] = nib_pair128<3>(q8.y);
}

__device__ __forceinline__ void mma_r(const uint32_t (&A)[4][4], uint4 v0, uint4 v1, float (&R)[4])
{
    mma_bf16(R, A[0][0], A[0][1], A[0][2], A[0][3], v0.x, v0.y);
    mma_bf16(R, A[1][0], A[1][1], A[1][2], A[1][3], v0.z, v0.w);
    mma_bf16(R, A[2][0], A[2][1], A[2][2], A[2][3], v1.x, v1.y);
    mma_bf16(R, A[3][0], A[3][1], A[3][2], A[3][3], v1.z, v1.w);
}

__device__ __forceinline__ void mma_x(uint4 v0, uint4 v1, float (&X)[4])
{
    mma_bf16(X, kOnes, kOnes, kOnes, kOnes, v0.x, v0.y);
    mma_bf16(X, kOnes, kOnes, kOnes, kOnes, v0.z, v0.w);
    mma_bf16(X, kOnes, kOnes, kOnes, kOnes, v1.x, v1.y);
    mma_bf16(X, kOnes, kOnes, kOnes, kOnes, v1.z, v1.w);
}

__device__ __forceinline__ void affine_acc(float (&acc)[4], const float (&R)[4], const float (&X)[4], float s0,
                                           float s8, float b0, float b8)
{
    const float c0 = fmaf(-128.f, s0, b0), c8 = fmaf(-128.f, s8, b8);
    acc[0] = fmaf(c0, X[0], fmaf(s0, R[0], acc[0]));
    acc[1] = fmaf(c0, X[1], fmaf(s0, R[1], acc[1]));
    acc[2] = fmaf(c8, X[2], fmaf(s8, R[2], acc[2]));
    acc[3] = fmaf(c8, X[3], fmaf(s8, R[3], acc[3]));
}

template <bool SMEM>
__device__ __forceinline__ void load_b(const uint16_t *p, uint4 &v0, uint4 &v1)
{
    if constexpr (SMEM) {
        v0 = *reinterpret_cast<const uint4 *>(p);
        v1 = *reinterpret_cast<const uint4 *>(p + 8);
    } else {
        v0 = ldg_u4(p);
        v1 = ldg_u4(p + 8);
    }
}

// Routing metadata staged in shared memory.
struct Meta {
    int *tiles;     // [3][max_tiles]
    int *perm;      // [T*K]
    float *topk_w;  // [T*K]
    int *n_tiles;   // [1]
};

__device__ __forceinline__ Meta meta_carve(uint8_t *base, int max_tiles, int tk)
{
    Meta m;
    int *p = reinterpret_cast<int *>(base);
    m.tiles = p;
    p += 3 * max_tiles;
    m.perm = p;
    p += tk;
    m.topk_w = reinterpret_cast<float *>(p);
    p += tk;
    m.n_tiles = p;
    return m;
}

// Consumers: copy the router kernel's grouping into shared memory.
__device__ __forceinline__ void meta_load(const FfnArgs &a, const Meta &m, bool weights)
{
    const int nt = __ldcg(a.n_tiles), tk = a.T * a.K;
    for (int i = threadIdx.x; i < 3 * nt; i += kConsumers)
        m.tiles[i] = __ldcg(a.tiles + i);
    for (int i = threadIdx.x; i < tk; i += kConsumers) {
        m.perm[i] = __ldcg(a.perm + i);
        if (weights)
            m.topk_w[i] = __ldcg(a.topk_w + i);
    }
    if (threadIdx.x == 0)
        *m.n_tiles = nt;
}

// ------------------------------------------------------------------ gate/up

struct GuItem {
    int routed, e, j0;  // expert (routed), first of the 8 hidden units
    int p0, ntok, t0;   // routed: slots [p0, p0+ntok); shared: tokens [t0, t0+ntok)
};

__device__ __forceinline__ GuItem gu_item(const FfnArgs &a, const GuLaunch &L, const Meta &m, int item)
{
    GuItem it;
    if (item < L.n_shared) {
        const int tt = item / (a.S / 8), rb = item % (a.S / 8);
        it.routed = 0;
        it.e = 0;
        it.j0 = rb * 8;
        it.t0 = tt * L.tpt;
        it.ntok = min(L.tpt, a.T - it.t0);
        it.p0 = 0;
    } else {
        const int j = item - L.n_shared, ti = j / (a.I / 8), rb = j % (a.I / 8);
        it.routed = 1;
        it.e = expert_record(a.slot, a.n_slots, m.tiles[3 * ti], a.err);
        it.p0 = m.tiles[3 * ti + 1];
        it.ntok = m.tiles[3 * ti + 2] - it.p0;
        it.j0 = rb * 8;
        it.t0 = 0;
    }
    return it;
}

// Slot: gate tile [G][8 rows][32 B], up tile [G][8][32 B], then gate.s, gate.b,
// up.s, up.b of the 8 rows (16*G bytes each).
template <int NT, int NS, bool BS>
__global__ void __launch_bounds__(kThreads, 2)
    gateup_kernel(const FfnArgs a, const GuLaunch L, const __grid_constant__ FfnMaps maps)
{
    constexpr int TPT = 8 * NT;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + L.stages;
    uint64_t *meta_ready = empty + L.stages;
    const Meta m = meta_carve(smem + L.off_meta, L.max_tiles, a.T * a.K);
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + L.off_xs);  // staged x operand
    float *xg = reinterpret_cast<float *>(smem + L.off_xg);        // [T][G] group sums of x
    uint8_t *ring = smem + L.off_ring;
    float *part = reinterpret_cast<float *>(smem + L.off_part);    // [kCW][16][TPT]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.D / kGroup;
    const uint32_t tile_bytes = 256u * G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        mbar_init(meta_ready, 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCW) {
        // producer: shared-expert items need nothing from the router
        bool meta = false;
        int total = L.n_shared;
        for (int k = 0, item = blockIdx.x;; ++k, item += gridDim.x) {
            if (item >= total && !meta) {
                if (!mbar_wait(meta_ready, 0, a.err))
                    break;
                meta = true;
                total = L.n_shared + *m.n_tiles * (a.I / 8);
            }
            if (item >= total)
                break;
            const int slot = k % L.stages;
            if (k >= L.stages && !mbar_wait(&empty[slot], ((k / L.stages) - 1) & 1, a.err))
                break;
            const GuItem it = gu_item(a, L, m, item);
            uint8_t *dst = ring + (size_t)slot * L.slot_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], 2u * tile_bytes + 4u * 16u * G);
                if (it.routed) {
                    tma_load_4d(dst, &maps.gate, 0, it.j0, 0, it.e, &full[slot]);
                    tma_load_4d(dst + tile_bytes, &maps.up, 0, it.j0, 0, it.e, &full[slot]);
                } else {
                    tma_load_4d(dst, &maps.sgate, 0, it.j0, 0, 0, &full[slot]);
                    tma_load_4d(dst + tile_bytes, &maps.sup, 0, it.j0, 0, 0, &full[slot]);
                }
            }
            __syncwarp();
            if (lane >= 1 && lane <= 4) {
                const int j = lane - 1;  // gate.s, gate.b, up.s, up.b
                const uint16_t *src;
                if (it.routed) {
                    const uint8_t *rec = a.blob + (uint64_t)it.e * a.stride;
                    src = reinterpret_cast<const uint16_t *>(rec + (j & 1 ? a.off_b[j >> 1] : a.off_s[j >> 1]));
                } else {
                    src = j & 1 ? a.sb[j >> 1] : a.ss[j >> 1];
                }
                bulk_g2s(dst + 2 * tile_bytes + j * 16 * G, src + (size_t)it.j0 * G, 16u * G, &full[slot]);
            }
        }
        pdl_wait();
        pdl_trigger();
        return;
    }

    // consumers
    pdl_wait();  // routing, x operand and x group sums of the router kernel
    meta_load(a, m, false);
    const size_t TD = (size_t)a.T * a.D;
    if constexpr (BS) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.xp);
        uint4 *dst = reinterpret_cast<uint4 *>(xs);
        for (int i = threadIdx.x; i < (int)(NS * TD / 8); i += kConsumers)
            dst[i] = __ldcg(src + i);
    }
    for (int i = threadIdx.x; i < a.T * G; i += kConsumers)
        xg[i] = __ldcg(a.xg + i);
    named_sync(1, kConsumers);
    if (threadIdx.x == 0)
        mbar_arrive(meta_ready);
    pdl_trigger();  // the down kernel may start: the router has completed
    const int gid = lane >> 2, c = lane & 3;
    const int total = L.n_shared + *m.n_tiles * (a.I / 8);
    const uint16_t *bsrc = BS ? xs : a.xp;
    bool failed = false;  // a bounded wait gave up: skip the math, keep the barriers
    for (int k = 0, item = blockIdx.x; item < total; ++k, item += gridDim.x) {
        const int slot = k % L.stages;
        const GuItem it = gu_item(a, L, m, item);
        int rowoff[NT], ct0[NT], ct1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = 8 * nt + gid, m0 = 8 * nt + 2 * c, m1 = m0 + 1;
            int tok = -1;
            if (n < it.ntok)
                tok = it.routed ? m.perm[it.p0 + n] / a.K : it.t0 + n;
            rowoff[nt] = tok >= 0 ? tok * a.D : -1;
            ct0[nt] = m0 < it.ntok ? (it.routed ? m.perm[it.p0 + m0] / a.K : it.t0 + m0) : 0;
            ct1[nt] = m1 < it.ntok ? (it.routed ? m.perm[it.p0 + m1] / a.K : it.t0 + m1) : 0;
        }
        const int nnt = (it.ntok + 7) >> 3;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        if (!failed)
            failed = !mbar_wait(&full[slot], (k / L.stages) & 1, a.err);
        const uint8_t *st = ring + (size_t)slot * L.slot_bytes;
        const uint8_t *gate = st + gid * 32 + 8 * c;               // + 256 g
        const uint8_t *up = st + tile_bytes + gid * 32 + 8 * c;    // + 256 g
        const uint16_t *sc = reinterpret_cast<const uint16_t *>(st + 2 * tile_bytes);
        const uint16_t *sg = sc + gid * G, *bg = sc + 8 * G + gid * G;
        const uint16_t *su = sc + 16 * G + gid * G, *bu = sc + 24 * G + gid * G;
#pragma unroll 2
        for (int g = warp; g < (failed ? 0 : G); g += kCW) {
            uint32_t A[4][4];
            build_a(*reinterpret_cast<const uint2 *>(gate + 256 * g), *reinterpret_cast<const uint2 *>(up + 256 * g),
                    A);
            const float s0 = bf2f(sg[g]), s8 = bf2f(su[g]), b0 = bf2f(bg[g]), b8 = bf2f(bu[g]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (nt < nnt) {
                    float R[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int sp = 0; sp < NS; ++sp) {
                        uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
                        if (rowoff[nt] >= 0)
                            load_b<BS>(bsrc + sp * TD + rowoff[nt] + kGroup * g + 16 * c, v0, v1);
                        mma_r(A, v0, v1, R);
                    }
                    const float x0 = xg[ct0[nt] * G + g], x1 = xg[ct1[nt] * G + g];
                    const float X[4] = {x0, x1, x0, x1};
                    affine_acc(acc[nt], R, X, s0, s8, b0, b8);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
        float *pw = part + warp * 16 * TPT;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if (nt < nnt) {
                const int col = 8 * nt + 2 * c;
                pw[gid * TPT + col] = acc[nt][0];
                pw[gid * TPT + col + 1] = acc[nt][1];
                pw[(gid + 8) * TPT + col] = acc[nt][2];
                pw[(gid + 8) * TPT + col + 1] = acc[nt][3];
            }
        }
        named_sync(1, kConsumers);
        uint16_t *h0 = it.routed ? a.hr[0] : a.hs[0];
        uint16_t *h1 = it.routed ? a.hr[1] : a.hs[1];
        const int hld = it.routed ? a.I : a.S;
        const int hrow0 = it.routed ? it.p0 : it.t0;
        for (int el = threadIdx.x; el < 8 * it.ntok; el += kConsumers) {
            const int r = el & 7, n = el >> 3;
            float gs = 0.f, us = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w) {
                gs += part[(w * 16 + r) * TPT + n];
                us += part[(w * 16 + 8 + r) * TPT + n];
            }
            const float h = gelu_tanh(gs) * us;
            const uint16_t hi = f2bf(h);
            const size_t o = (size_t)(hrow0 + n) * hld + perm8(it.j0 + r);
            h0[o] = hi;
            h1[o] = f2bf(h - bf2f(hi));
        }
        named_sync(1, kConsumers);
    }
}

// --------------------------------------------------------------------- down

struct DnUnit {
    int shared_unit, e, G, cols;
    int p0, ntok;
    const uint16_t *s, *b;    // scales / biases of the 16 rows
    const uint16_t *h0, *h1;  // hi / lo rows of this unit's first token
};

__device__ __forceinline__ DnUnit dn_unit(const FfnArgs &a, const Meta &m, int u, int row0)
{
    DnUnit d;
    if (u == 0) {
        d.shared_unit = 1;
        d.e = 0;
        d.cols = a.S;
        d.G = a.S / kGroup;
        d.s = a.ss[2] + (size_t)row0 * d.G;
        d.b = a.sb[2] + (size_t)row0 * d.G;
        d.h0 = a.hs[0];
        d.h1 = a.hs[1];
        d.p0 = 0;
        d.ntok = a.T;
    } else {
        const int ti = u - 1;
        d.shared_unit = 0;
        d.e = expert_record(a.slot, a.n_slots, m.tiles[3 * ti], a.err);
        d.p0 = m.tiles[3 * ti + 1];
        d.ntok = m.tiles[3 * ti + 2] - d.p0;
        d.cols = a.I;
        d.G = a.I / kGroup;
        const uint8_t *rec = a.blob + (uint64_t)d.e * a.stride;
        d.s = reinterpret_cast<const uint16_t *>(rec + a.off_s[2]) + (size_t)row0 * d.G;
        d.b = reinterpret_cast<const uint16_t *>(rec + a.off_b[2]) + (size_t)row0 * d.G;
        d.h0 = a.hr[0] + (size_t)d.p0 * a.I;
        d.h1 = a.hr[1] + (size_t)d.p0 * a.I;
    }
    return d;
}

// Slot: down tile [G][16 rows][32 B], then the 16 rows' scales and biases (32*G bytes each).
template <int NT>  // NT n-tiles of 8 columns; column n = (token n/2, hi/lo part n%2)
__global__ void __launch_bounds__(kThreads, 2)
    down_kernel(const FfnArgs a, const DnLaunch L, const __grid_constant__ FfnMaps maps)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + L.stages;
    uint64_t *meta_ready = empty + L.stages;
    const Meta m = meta_carve(smem + L.off_meta, L.max_tiles, a.T * a.K);
    uint8_t *ring = smem + L.off_ring;
    float *accs = reinterpret_cast<float *>(smem + L.off_acc);  // [kCW][T][16]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * 16;
    const int T = a.T;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        mbar_init(meta_ready, 1);
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < kCW * T * 16; i += kThreads)
        accs[i] = 0.f;
    __syncthreads();

    if (warp == kCW) {
        // The router has completed before the gate/up kernel let this grid
        // launch, so the grouping is valid before this grid's own wait.
        if (!mbar_wait(meta_ready, 0, a.err)) {
            pdl_wait();
            pdl_trigger();
            return;
        }
        const int n_units = 1 + *m.n_tiles;
        for (int u = 0; u < n_units; ++u) {
            const int slot = u % L.stages;
            if (u >= L.stages && !mbar_wait(&empty[slot], ((u / L.stages) - 1) & 1, a.err))
                break;
            const DnUnit d = dn_unit(a, m, u, row0);
            uint8_t *dst = ring + (size_t)slot * L.slot_bytes;
            const uint32_t tile = 512u * d.G;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], tile + 64u * d.G);
                if (d.shared_unit)
                    tma_load_4d(dst, &maps.sdown, 0, row0, 0, 0, &full[slot]);
                else
                    tma_load_4d(dst, &maps.down, 0, row0, 0, d.e, &full[slot]);
            }
            __syncwarp();
            if (lane == 1 || lane == 2)
                bulk_g2s(dst + tile + (lane - 1) * 32 * d.G, lane == 1 ? d.s : d.b, 32u * d.G, &full[slot]);
        }
        pdl_wait();
        pdl_trigger();
        return;
    }

    // consumers
    meta_load(a, m, true);
    named_sync(1, kConsumers);
    if (threadIdx.x == 0)
        mbar_arrive(meta_ready);
    pdl_wait();     // hidden vectors of the gate/up kernel
    pdl_trigger();  // the next kernel may start its prologue
    const int gid = lane >> 2, c = lane & 3;
    const int n_units = 1 + *m.n_tiles;
    float *aw = accs + warp * T * 16;
    bool failed = false;
    for (int u = 0; u < n_units; ++u) {
        const int slot = u % L.stages;
        const DnUnit d = dn_unit(a, m, u, row0);
        // B column n = 8*nt + gid: token n>>1, part n&1
        int rowoff[NT];
        const uint16_t *bp[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = 8 * nt + gid, tok = n >> 1, pt = n & 1;
            rowoff[nt] = tok < d.ntok ? tok * d.cols : -1;
            bp[nt] = pt ? d.h1 : d.h0;
        }
        // the lane's C columns: token 4*nt + c, parts 0 and 1
        int tcol[NT];
        float wcol[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int mm = 4 * nt + c;
            tcol[nt] = -1;
            wcol[nt] = 0.f;
            if (mm < d.ntok) {
                if (d.shared_unit) {
                    tcol[nt] = mm;
                    wcol[nt] = 1.f;
                } else {
                    const int slot_id = m.perm[d.p0 + mm];
                    tcol[nt] = slot_id / a.K;
                    wcol[nt] = m.topk_w[slot_id];
                }
            }
        }
        const int nnt = (2 * d.ntok + 7) >> 3;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        if (!failed)
            failed = !mbar_wait(&full[slot], (u / L.stages) & 1, a.err);
        const uint8_t *st = ring + (size_t)slot * L.slot_bytes;
        const uint8_t *lo = st + gid * 32 + 8 * c, *hi = lo + 256;  // rows gid / gid+8, + 512 g
        const uint16_t *ss = reinterpret_cast<const uint16_t *>(st + 512 * d.G);
        const uint16_t *sb = ss + 16 * d.G;
        const uint16_t *s_lo = ss + gid * d.G, *s_hi = ss + (gid + 8) * d.G;
        const uint16_t *b_lo = sb + gid * d.G, *b_hi = sb + (gid + 8) * d.G;
#pragma unroll 2
        for (int g = warp; g < (failed ? 0 : d.G); g += kCW) {
            uint32_t A[4][4];
            build_a(*reinterpret_cast<const uint2 *>(lo + 512 * g), *reinterpret_cast<const uint2 *>(hi + 512 * g), A);
            const float s0 = bf2f(s_lo[g]), s8 = bf2f(s_hi[g]), b0 = bf2f(b_lo[g]), b8 = bf2f(b_hi[g]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (nt < nnt) {
                    float R[4] = {0.f, 0.f, 0.f, 0.f}, X[4] = {0.f, 0.f, 0.f, 0.f};
                    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
                    if (rowoff[nt] >= 0)
                        load_b<false>(bp[nt] + rowoff[nt] + kGroup * g + 16 * c, v0, v1);
                    mma_r(A, v0, v1, R);
                    mma_x(v0, v1, X);
                    affine_acc(acc[nt], R, X, s0, s8, b0, b8);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int t = tcol[nt];
            if (t >= 0) {
                aw[t * 16 + gid] += wcol[nt] * (acc[nt][0] + acc[nt][1]);
                aw[t * 16 + gid + 8] += wcol[nt] * (acc[nt][2] + acc[nt][3]);
            }
        }
        __syncwarp();
    }
    named_sync(1, kConsumers);
    for (int el = threadIdx.x; el < T * 16; el += kConsumers) {
        const int t = el >> 4, r = el & 15;
        float v = accs[t * 16 + r];
#pragma unroll
        for (int w = 1; w < kCW; ++w)
            v += accs[(w * T + t) * 16 + r];
        float o = a.lam * v;
        const size_t idx = (size_t)t * a.D + row0 + r;
        if (a.act_dtype == 1) {
            if (a.residual)
                o = bf2f(reinterpret_cast<const uint16_t *>(a.residual)[idx]) + o;
            reinterpret_cast<uint16_t *>(a.out)[idx] = f2bf(o);
        } else {
            if (a.residual)
                o = reinterpret_cast<const float *>(a.residual)[idx] + o;
            reinterpret_cast<float *>(a.out)[idx] = o;
        }
    }
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Args &...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

size_t align128(size_t n) { return (n + 127) & ~size_t(127); }

constexpr size_t kSmemLimit = 227 * 1024;  // dynamic shared memory per CTA
constexpr size_t kTwoPerSm = 112 * 1024;   // at most this to fit two CTAs on one SM

int fit_stages(size_t fixed, size_t slot, int lo, int hi, size_t budget)
{
    int n = budget > fixed ? (int)((budget - fixed) / slot) : 0;
    return n < lo ? lo : (n > hi ? hi : n);
}

size_t meta_bytes(const FfnArgs &a, int max_tiles) { return align128(4 * (3 * (size_t)max_tiles + 2 * a.T * a.K + 1)); }

template <int NTD>
cudaError_t launch_down(const FfnArgs &a, const DnLaunch &dl, const FfnMaps &maps, size_t smem, cudaStream_t s)
{
    cudaError_t e = smem_optin(reinterpret_cast<const void *>(down_kernel<NTD>), smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(down_kernel<NTD>, dim3(a.D / 16), dim3(kThreads), smem, s, a, dl, maps);
}

// Gate/up + down for one pass.  NT: 8-token n-tiles of the gate/up kernel.
template <int NT, int NS, bool BS>
cudaError_t launch_nt(const FfnArgs &a, const FfnMaps &maps, int max_tiles, int num_sms, cudaStream_t s)
{
    constexpr int TPT = 8 * NT;
    const int G = a.D / kGroup;
    const int meta_tiles = a.E + (a.T * a.K) / kTileTokens + 1;

    GuLaunch gl{};
    gl.tpt = TPT;
    gl.max_tiles = meta_tiles;
    gl.slot_bytes = (int)align128(2 * 256 * (size_t)G + 64 * (size_t)G);
    gl.n_shared = ((a.T + TPT - 1) / TPT) * (a.S / 8);
    gl.off_meta = kBarBytes;
    gl.off_xs = (int)(gl.off_meta + meta_bytes(a, meta_tiles));
    gl.off_xg = (int)(gl.off_xs + (BS ? align128((size_t)NS * a.T * a.D * 2) : 0));
    gl.off_ring = (int)(gl.off_xg + align128((size_t)a.T * G * 4));
    const size_t part_bytes = (size_t)kCW * 16 * TPT * sizeof(float);
    const bool two = gl.off_ring + 3 * (size_t)gl.slot_bytes + part_bytes <= kTwoPerSm;
    gl.stages = two ? fit_stages(gl.off_ring + part_bytes, gl.slot_bytes, 3, 4, kTwoPerSm)
                    : fit_stages(gl.off_ring + part_bytes, gl.slot_bytes, 2, 4, kSmemLimit);
    gl.off_part = gl.off_ring + gl.stages * gl.slot_bytes;
    const size_t smem_gu = gl.off_part + part_bytes;
    const int items = gl.n_shared + max_tiles * (a.I / 8);
    const int per_sm = two ? 2 : 1;
    int grid = per_sm * num_sms < items ? per_sm * num_sms : items;
    if (grid < 1)
        grid = 1;
    auto kg = gateup_kernel<NT, NS, BS>;
    cudaError_t e = smem_optin(reinterpret_cast<const void *>(kg), smem_gu);
    if (e != cudaSuccess)
        return e;
    prof_begin(kStageGateUp, s);
    e = launch_pdl(kg, dim3(grid), dim3(kThreads), smem_gu, s, a, gl, maps);
    prof_end(kStageGateUp, s);
    if (e != cudaSuccess)
        return e;

    DnLaunch dl{};
    dl.max_tiles = meta_tiles;
    const size_t slot_sh = 576 * (size_t)(a.S / kGroup);
    const size_t slot_rt = 576 * (size_t)(a.I / kGroup);
    dl.slot_bytes = (int)align128(slot_sh > slot_rt ? slot_sh : slot_rt);
    dl.off_meta = kBarBytes;
    dl.off_ring = (int)(dl.off_meta + meta_bytes(a, meta_tiles));
    const size_t acc_bytes = (size_t)kCW * a.T * 16 * sizeof(float);
    dl.stages = fit_stages(dl.off_ring + acc_bytes, dl.slot_bytes, 2, 6, kTwoPerSm);
    if (dl.off_ring + acc_bytes + (size_t)dl.stages * dl.slot_bytes > kTwoPerSm)
        dl.stages = fit_stages(dl.off_ring + acc_bytes, dl.slot_bytes, 2, 6, kSmemLimit);
    dl.off_acc = dl.off_ring + dl.stages * dl.slot_bytes;
    const size_t smem_dn = dl.off_acc + acc_bytes;
    const int ntd = (2 * a.T + 7) / 8;  // down n-tiles: 2 parts per token
    prof_begin(kStageDown, s);
    if (ntd <= 1)
        e = launch_down<1>(a, dl, maps, smem_dn, s);
    else if (ntd <= 2)
        e = launch_down<2>(a, dl, maps, smem_dn, s);
    else if (ntd <= 4)
        e = launch_down<4>(a, dl, maps, smem_dn, s);
    else if (ntd <= 8)
        e = launch_down<8>(a, dl, maps, smem_dn, s);
    else
        e = launch_down<16>(a, dl, maps, smem_dn, s);
    prof_end(kStageDown, s);
    return e;
}

template <int NT, int NS>
cudaError_t launch_bs(const FfnArgs &a, const FfnMaps &maps, int max_tiles, int num_sms, cudaStream_t s)
{
    // stage the x operand in shared memory when it is small
    if ((size_t)NS * a.T * a.D * 2 <= 24 * 1024)
        return launch_nt<NT, NS, true>(a, maps, max_tiles, num_sms, s);
    return launch_nt<NT, NS, false>(a, maps, max_tiles, num_sms, s);
}

template <int NT>
cudaError_t launch_ns(const FfnArgs &a, const FfnMaps &maps, int max_tiles, int num_sms, cudaStream_t s)
{
    if (a.nsplit == 1)
        return launch_bs<NT, 1>(a, maps, max_tiles, num_sms, s);
    return launch_bs<NT, 3>(a, maps, max_tiles, num_sms, s);
}

} // namespace

cudaError_t launch_ffn_decode(const FfnArgs &a, int max_tiles, int num_sms, cudaStream_t s)
{
    FfnMaps maps;
    cudaError_t e = get_ffn_maps(a, &maps);
    if (e != cudaSuccess)
        return e;
    const int nt = (a.T + 7) / 8;  // T <= kDecodeChunk
    if (nt <= 1)
        return launch_ns<1>(a, maps, max_tiles, num_sms, s);
    if (nt <= 2)
        return launch_ns<2>(a, maps, max_tiles, num_sms, s);
    if (nt <= 4)
        return launch_ns<4>(a, maps, max_tiles, num_sms, s);
    return launch_ns<8>(a, maps, max_tiles, num_sms, s);
}

} // namespace mx

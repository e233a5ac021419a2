// mx_ffn_decode.cu -- routed + shared expert FFN for small token counts
// (decode, T <= 64 per pass).
//
// "Mference System design" page, section "Metal execution": decode consumes the
// packed values, BF16 scales and BF16 biases directly, and the routed kernels
// fuse affine decode, GeGLU and the weighted expert reduction; section
// "Decode" (cb2 row): the routed top-k branch is reduced with the router
// weights, combined with the shared branch, and scaled by the layer scalar.
//
// Two launches per pass:
//   gateup_kernel  items = (expert tile, 16 rows of I) for every routed tile,
//                  plus (token tile, 16 rows of S) for the shared expert.  Each
//                  item computes g = W_gate x and u = W_up x for its tokens and
//                  writes h = gelu(g) * u as a BF16 hi/lo pair (fp32 carried).
//   down_kernel    one CTA per 16 output rows of D; it applies the shared down
//                  projection and every routed tile's down projection to those
//                  rows and reduces them in a fixed order:
//                  out = residual + lambda * (shared + sum_k w_k y_k).
// No atomics: the reduction order depends only on the routing, so the result
// is deterministic ("Mference System design", "Correctness and safety
// invariants": reordered float kernels stay deterministic within a path).
//
// Inner loop (warp_qgemm): the warp owns 16 weight rows.  Per group of 64
// columns it loads the rows' packed words with 8-byte streaming loads (a quad
// of lanes covers one 32-byte sector of a row), turns the nibbles into exact
// BF16 integers, and runs m16n8k16 MMAs against the B rows (x or h) for the
// quantized sum P and against an all-ones A for the group sum X; then
//     acc += s * P + b * X
// in fp32.  Legacy warp MMAs suffice here: the decode path is bound by HBM,
// not by the tensor pipe, and register accumulators make the per-group affine
// step exact and cheap.
#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kOnes = 0x3F803F80u;  // BF16x2 (1.0, 1.0)

// Accumulate, for the warp's 16 rows (row0 = lane's gid row, row8 = gid+8),
// groups g = g_begin, g_begin + g_step, ... < g_end.
//   w0, w8     packed words of rows gid / gid+8 (row starts)
//   s0..b8     BF16 scale / bias rows (row starts)
//   bbase[NS]  B split bases; rowoff[nt] = element offset of the B row for
//              token column 8*nt + gid (or -1: zero column)
template <int NT, int NS, int UNR>
__device__ __forceinline__ void warp_qgemm(const uint32_t *__restrict__ w0, const uint32_t *__restrict__ w8,
                                           const uint16_t *__restrict__ s0, const uint16_t *__restrict__ s8,
                                           const uint16_t *__restrict__ b0, const uint16_t *__restrict__ b8,
                                           int g_begin, int g_end, int g_step,
                                           const uint16_t *const (&bbase)[NS], const int (&rowoff)[NT], int nnt,
                                           float (&acc)[NT][4])
{
    const int c = threadIdx.x & 3;
    for (int gb = g_begin; gb < g_end; gb += UNR * g_step) {
        uint2 q0[UNR], q8[UNR];
        float sc0[UNR], sc8[UNR], bi0[UNR], bi8[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int g = gb + u * g_step;
            if (g < g_end) {
                q0[u] = ld_stream_u2(w0 + 8 * g + 2 * c);
                q8[u] = ld_stream_u2(w8 + 8 * g + 2 * c);
                sc0[u] = bf2f(__ldg(s0 + g));
                sc8[u] = bf2f(__ldg(s8 + g));
                bi0[u] = bf2f(__ldg(b0 + g));
                bi8[u] = bf2f(__ldg(b8 + g));
            }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int g = gb + u * g_step;
            if (g >= g_end)
                break;
            // A fragments of the 4 k-steps of this group: k-step s uses word s/2
            // of the lane's pair, nibble pairs (j, j+4) and (j+1, j+5), j = 2*(s&1).
            uint32_t A[4][4];
            A[0][0] = nib_pair<0>(q0[u].x); A[0][1] = nib_pair<0>(q8[u].x);
            A[0][2] = nib_pair<1>(q0[u].x); A[0][3] = nib_pair<1>(q8[u].x);
            A[1][0] = nib_pair<2>(q0[u].x); A[1][1] = nib_pair<2>(q8[u].x);
            A[1][2] = nib_pair<3>(q0[u].x); A[1][3] = nib_pair<3>(q8[u].x);
            A[2][0] = nib_pair<0>(q0[u].y); A[2][1] = nib_pair<0>(q8[u].y);
            A[2][2] = nib_pair<1>(q0[u].y); A[2][3] = nib_pair<1>(q8[u].y);
            A[3][0] = nib_pair<2>(q0[u].y); A[3][1] = nib_pair<2>(q8[u].y);
            A[3][2] = nib_pair<3>(q0[u].y); A[3][3] = nib_pair<3>(q8[u].y);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (nt < nnt) {
                    float P[4] = {0.f, 0.f, 0.f, 0.f};
                    float X[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int sp = 0; sp < NS; ++sp) {
                        uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
                        if (rowoff[nt] >= 0) {
                            const uint16_t *p = bbase[sp] + rowoff[nt] + kGroup * g + 16 * c;
                            v0 = ldg_u4(p);
                            v1 = ldg_u4(p + 8);
                        }
                        mma_bf16(P, A[0][0], A[0][1], A[0][2], A[0][3], v0.x, v0.y);
                        mma_bf16(P, A[1][0], A[1][1], A[1][2], A[1][3], v0.z, v0.w);
                        mma_bf16(P, A[2][0], A[2][1], A[2][2], A[2][3], v1.x, v1.y);
                        mma_bf16(P, A[3][0], A[3][1], A[3][2], A[3][3], v1.z, v1.w);
                        mma_bf16(X, kOnes, kOnes, kOnes, kOnes, v0.x, v0.y);
                        mma_bf16(X, kOnes, kOnes, kOnes, kOnes, v0.z, v0.w);
                        mma_bf16(X, kOnes, kOnes, kOnes, kOnes, v1.x, v1.y);
                        mma_bf16(X, kOnes, kOnes, kOnes, kOnes, v1.z, v1.w);
                    }
                    acc[nt][0] = fmaf(bi0[u], X[0], fmaf(sc0[u], P[0], acc[nt][0]));
                    acc[nt][1] = fmaf(bi0[u], X[1], fmaf(sc0[u], P[1], acc[nt][1]));
                    acc[nt][2] = fmaf(bi8[u], X[2], fmaf(sc8[u], P[2], acc[nt][2]));
                    acc[nt][3] = fmaf(bi8[u], X[3], fmaf(sc8[u], P[3], acc[nt][3]));
                }
            }
        }
    }
}

template <int NT, int NS>
__global__ void __launch_bounds__(kThreads) gateup_kernel(const FfnArgs a)
{
    constexpr int TPT = 8 * NT;               // tokens per tile
    extern __shared__ __align__(16) float part[];  // [kWarps][2][16][TPT]
    __shared__ int tok_s[TPT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, c = lane & 3;
    const int G = a.D / kGroup, RB = a.I / 16, RBS = a.S / 16;
    const int ntiles = *a.n_tiles;
    const int n_sh_tt = (a.T + TPT - 1) / TPT;
    const int routed = ntiles * RB, total = routed + n_sh_tt * RBS;
    const size_t TD = (size_t)a.T * a.D;
    const int wpr = a.D / 8;  // packed words per row

    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const uint32_t *Wm[2];
        const uint16_t *Sm[2], *Bm[2];
        int row0, ntok, hrow0, hld;
        uint16_t *hdst0, *hdst1;
        if (item < routed) {
            const int ti = item / RB, rb = item % RB;
            const int e = a.tiles[3 * ti], p0 = a.tiles[3 * ti + 1], p1 = a.tiles[3 * ti + 2];
            const uint8_t *rec = a.blob + (uint64_t)e * a.stride;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                Wm[m] = reinterpret_cast<const uint32_t *>(rec + a.off_w[m]);
                Sm[m] = reinterpret_cast<const uint16_t *>(rec + a.off_s[m]);
                Bm[m] = reinterpret_cast<const uint16_t *>(rec + a.off_b[m]);
            }
            row0 = rb * 16;
            ntok = p1 - p0;
            if (threadIdx.x < ntok)
                tok_s[threadIdx.x] = a.perm[p0 + threadIdx.x] / a.K;
            hrow0 = p0;
            hld = a.I;
            hdst0 = a.hr[0];
            hdst1 = a.hr[1];
        } else {
            const int j = item - routed, tt = j / RBS, rb = j % RBS;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                Wm[m] = a.sw[m];
                Sm[m] = a.ss[m];
                Bm[m] = a.sb[m];
            }
            row0 = rb * 16;
            const int t0 = tt * TPT;
            ntok = min(TPT, a.T - t0);
            if (threadIdx.x < ntok)
                tok_s[threadIdx.x] = t0 + threadIdx.x;
            hrow0 = t0;
            hld = a.S;
            hdst0 = a.hs[0];
            hdst1 = a.hs[1];
        }
        __syncthreads();
        int rowoff[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = 8 * nt + gid;
            rowoff[nt] = (n < ntok) ? tok_s[n] * a.D : -1;
        }
        const uint16_t *bbase[NS];
#pragma unroll
        for (int sp = 0; sp < NS; ++sp)
            bbase[sp] = a.xp + sp * TD;
        const int nnt = (ntok + 7) >> 3;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            const size_t r0 = (size_t)(row0 + gid);
            warp_qgemm<NT, NS, 4>(Wm[m] + r0 * wpr, Wm[m] + (r0 + 8) * wpr, Sm[m] + r0 * G, Sm[m] + (r0 + 8) * G,
                                  Bm[m] + r0 * G, Bm[m] + (r0 + 8) * G, warp, G, kWarps, bbase, rowoff, nnt, acc);
            float *pw = part + (warp * 2 + m) * 16 * TPT;
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
        }
        __syncthreads();
        for (int el = threadIdx.x; el < 16 * ntok; el += kThreads) {
            const int r = el & 15, n = el >> 4;
            float g = 0.f, u = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                g += part[((w * 2 + 0) * 16 + r) * TPT + n];
                u += part[((w * 2 + 1) * 16 + r) * TPT + n];
            }
            const float h = gelu_tanh(g) * u;
            const uint16_t hi = f2bf(h);
            const uint16_t lo = f2bf(h - bf2f(hi));
            const size_t o = (size_t)(hrow0 + n) * hld + perm8(row0 + r);
            hdst0[o] = hi;
            hdst1[o] = lo;
        }
        __syncthreads();
    }
}

template <int NT>
__global__ void __launch_bounds__(kThreads) down_kernel(const FfnArgs a)
{
    extern __shared__ __align__(16) float accs[];  // [kWarps][T][16]
    __shared__ int wtok[kWarps][kTileTokens];
    __shared__ float wwt[kWarps][kTileTokens];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, c = lane & 3;
    const int row0 = blockIdx.x * 16;
    const int T = a.T, GI = a.I / kGroup, GS = a.S / kGroup;
    float *aw = accs + warp * T * 16;

    // shared expert: this warp's groups of S, all T tokens
    {
        int rowoff[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = 8 * nt + gid;
            rowoff[nt] = (n < T) ? n * a.S : -1;
        }
        const uint16_t *bbase[2] = {a.hs[0], a.hs[1]};
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        const size_t r0 = (size_t)(row0 + gid);
        const int wpr = a.S / 8;
        warp_qgemm<NT, 2, 4>(a.sw[2] + r0 * wpr, a.sw[2] + (r0 + 8) * wpr, a.ss[2] + r0 * GS,
                             a.ss[2] + (r0 + 8) * GS, a.sb[2] + r0 * GS, a.sb[2] + (r0 + 8) * GS, warp, GS, kWarps,
                             bbase, rowoff, (T + 7) >> 3, acc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = 8 * nt + 2 * c;
            if (n < T) {
                aw[n * 16 + gid] = acc[nt][0];
                aw[n * 16 + gid + 8] = acc[nt][2];
            }
            if (n + 1 < T) {
                aw[(n + 1) * 16 + gid] = acc[nt][1];
                aw[(n + 1) * 16 + gid + 8] = acc[nt][3];
            }
        }
    }
    __syncwarp();

    // routed tiles owned by this warp
    const int ntiles = *a.n_tiles;
    const int wpr = a.I / 8;
    for (int ti = warp; ti < ntiles; ti += kWarps) {
        const int e = a.tiles[3 * ti], p0 = a.tiles[3 * ti + 1], p1 = a.tiles[3 * ti + 2];
        const int ntok = p1 - p0;
        for (int n = lane; n < ntok; n += 32) {
            const int slot = a.perm[p0 + n];
            wtok[warp][n] = slot / a.K;
            wwt[warp][n] = a.topk_w[slot];
        }
        __syncwarp();
        int rowoff[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = 8 * nt + gid;
            rowoff[nt] = (n < ntok) ? (p0 + n) * a.I : -1;
        }
        const uint16_t *bbase[2] = {a.hr[0], a.hr[1]};
        const uint8_t *rec = a.blob + (uint64_t)e * a.stride;
        const uint32_t *W = reinterpret_cast<const uint32_t *>(rec + a.off_w[2]);
        const uint16_t *S = reinterpret_cast<const uint16_t *>(rec + a.off_s[2]);
        const uint16_t *B = reinterpret_cast<const uint16_t *>(rec + a.off_b[2]);
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        const size_t r0 = (size_t)(row0 + gid);
        warp_qgemm<NT, 2, 4>(W + r0 * wpr, W + (r0 + 8) * wpr, S + r0 * GI, S + (r0 + 8) * GI, B + r0 * GI,
                             B + (r0 + 8) * GI, 0, GI, 1, bbase, rowoff, (ntok + 7) >> 3, acc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int n = 8 * nt + 2 * c + (i & 1);
                const int r = gid + 8 * (i >> 1);
                if (n < ntok) {
                    const int t = wtok[warp][n];
                    aw[t * 16 + r] += wwt[warp][n] * acc[nt][i];
                }
            }
        }
        __syncwarp();
    }
    __syncthreads();

    for (int el = threadIdx.x; el < T * 16; el += kThreads) {
        const int t = el >> 4, r = el & 15;
        float v = accs[(0 * T + t) * 16 + r];
#pragma unroll
        for (int w = 1; w < kWarps; ++w)
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

template <int NT, int NS>
cudaError_t launch_nt(const FfnArgs &a, int max_tiles, int num_sms, cudaStream_t s)
{
    const int TPT = 8 * NT;
    const int items = max_tiles * (a.I / 16) + ((a.T + TPT - 1) / TPT) * (a.S / 16);
    int grid = num_sms * 8;
    if (grid > items)
        grid = items;
    if (grid < 1)
        grid = 1;
    const size_t smem_gu = (size_t)kWarps * 2 * 16 * TPT * sizeof(float);
    prof_begin(kStageGateUp, s);
    gateup_kernel<NT, NS><<<grid, kThreads, smem_gu, s>>>(a);
    cudaError_t e = cudaGetLastError();
    prof_end(kStageGateUp, s);
    if (e != cudaSuccess)
        return e;
    const size_t smem_dn = (size_t)kWarps * a.T * 16 * sizeof(float);
    prof_begin(kStageDown, s);
    down_kernel<NT><<<a.D / 16, kThreads, smem_dn, s>>>(a);
    e = cudaGetLastError();
    prof_end(kStageDown, s);
    return e;
}

template <int NT>
cudaError_t launch_ns(const FfnArgs &a, int max_tiles, int num_sms, cudaStream_t s)
{
    if (a.nsplit == 1)
        return launch_nt<NT, 1>(a, max_tiles, num_sms, s);
    return launch_nt<NT, 3>(a, max_tiles, num_sms, s);
}

} // namespace

cudaError_t launch_ffn_decode(const FfnArgs &a, int max_tiles, int num_sms, cudaStream_t s)
{
    const int nt = (a.T + 7) / 8;  // T <= kDecodeChunk
    if (nt <= 1)
        return launch_ns<1>(a, max_tiles, num_sms, s);
    if (nt <= 2)
        return launch_ns<2>(a, max_tiles, num_sms, s);
    if (nt <= 4)
        return launch_ns<4>(a, max_tiles, num_sms, s);
    return launch_ns<8>(a, max_tiles, num_sms, s);
}

} // namespace mx

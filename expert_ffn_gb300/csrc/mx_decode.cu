// mx_decode.cu -- single-launch decode path: the whole block, or a stack of
// blocks, for T <= 4 tokens in one persistent cooperative kernel.
//
// What it computes is the block of the "Mference System design" page
// (section "Decode": router GEMV, top-8, softmax; the routed gated experts,
// the unweighted shared expert and the layer scalar; section "Metal
// execution": affine decode fused into the expert math, GeGLU and the weighted
// expert reduction fused), for every layer of the call.
//
// Why one launch.  At T = 1 a layer streams ~37 MB of packed weights, about
// 5.5 us of HBM time on this GPU, while the dependency chain of a layer (x ->
// router -> top-k -> routed gate/up -> routed down -> next x) crosses the whole
// grid three times.  Separate launches pay a ramp at every edge and leave HBM
// idle meanwhile.  Here every SM runs one CTA for the whole call; CTAs hand
// results to each other through global counters (bounded waits), and each CTA's
// producer warp keeps loading weights whose addresses are already known -- the
// shared expert's, also those of the next layer -- so the memory system stays
// busy across the edges.  Every CTA keeps the residual stream x in its own
// shared memory and rebuilds x_{l+1} from the summed down projections, so
// layers hand over without another exchange.
//
// CTA: 8 consumer warps + 1 producer warp.  Work comes in units of 64 hidden
// rows of one expert: rows [64u, 64u + 64) of the shared expert (S/64 units)
// or of an active routed expert (I/64 units each); unit i runs on CTA i mod
// the grid, shared units first (they start before the routing is known).
// The producer streams a unit's 12 items into one ring of shared memory with
// TMA tensor copies (group-major, see mx_tma.cu) and bulk copies of the rows'
// BF16 scales and biases:
//   8 gate/up items: 8 gate + 8 up rows x D (the 16 rows of one MMA tile, so
//     gelu(g) * u is lane-local), one per consumer warp;
//   4 down items: D/4 rows x the unit's 64 columns, row tiles over all warps.
// A unit keeps its 64 hidden values on chip and adds its slice of the down
// projection, for all D outputs, into y in 64-bit fixed point, whose integer
// addition does not depend on the order, so the result is deterministic; every
// CTA then forms x_{l+1} = residual + lambda * y.  Each CTA also computes one
// router row per E / grid of the layer (round-robin), in the fixed order
// below; the logits and y are the only grid-wide exchanges of a layer.
//
//
// Math: legacy warp MMA m16n8k32 with FP8 (e4m3) operands and fp32
// accumulation.  A raw nibble byte n (0..15) is exactly the e4m3 number
// n * 2^-9, so A is built from the packed words with one mask (low nibbles) or
// a shift and a mask (high nibbles) per 4 weights -- the high/low split reorders
// K, and B follows the same order.  B carries the activation (x, or the hidden
// vector for the down projections) scaled by a per-vector power of two and
// split into e4m3 planes whose sum reproduces it (x: 2 planes when it is BF16,
// exact for every element within 2^10 of the vector's largest; 4 planes for
// fp32 x and for the fp32 hidden vectors, about 16 significant bits); the
// planes sit in the columns of the MMA, and each lane adds its plane columns.
// The per-group affine terms are applied in fp32: y += s_g * P_g + b_g * X_g
// with P_g = sum q x from the MMA and X_g = sum x.  The e4m3 MMA accumulates in
// fp32 (checked against exact sums on this GPU).
//
// The router is not on the MMA: its logits are computed in the fixed fp32
// order of the header so the top-k choice matches the oracle bit for bit.
#include "mx_common.cuh"
#include "mx_internal.h"

#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>
#include <type_traits>

namespace mx {

namespace {

constexpr int kCW = 8;                 // consumer warps
constexpr int kCT = kCW * 32;          // consumer threads
constexpr int kPT = kCT + 32;          // + the producer warp
constexpr uint32_t kLo = 0x0F0F0F0Fu;  // low nibble of every byte

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ uint2 lds64(const uint8_t *p) { return *reinterpret_cast<const uint2 *>(p); }

// D += A(16x32 e4m3, row) * B(32x8 e4m3, col), fp32 accumulate.
__device__ __forceinline__ void mma_fp8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> two e4m3 bytes (round to nearest even, saturating): lo in bits 0-7.
__device__ __forceinline__ uint32_t to_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3 bytes (bits 0-15 of v) -> floats, exactly.
__device__ __forceinline__ float2 from_e4m3x2(uint32_t v)
{
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)v));
    return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

// Power-of-two scale 2^k putting the largest magnitude m in [128, 256), and
// the factor 2^(9-k) that turns an MMA sum of (n 2^-9)(x 2^k) back into sum n x.
__device__ __forceinline__ void plane_scale(float m, float &sc, float &back)
{
    const int E = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
    int k = 7 - E;
    k = k > 126 ? 126 : (k < -117 ? -117 : k);
    sc = __uint_as_float((uint32_t)(127 + k) << 23);
    back = __uint_as_float((uint32_t)(127 + 9 - k) << 23);
}

// Power-of-two scale 2^k putting the largest magnitude m in [2^(B-2),
// 2^(B-1)) for a B-bit fixed-point copy, and 2^-k; k is clamped to
// [-126, 126] so that both are normal floats (a vector below 2^(B-128) keeps
// fewer bits).
template <int B>
__device__ __forceinline__ void fixb_scale(float m, float &sc, float &inv)
{
    const int E = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
    int k = B - 2 - E;
    k = k > 126 ? 126 : (k < -126 ? -126 : k);
    sc = __uint_as_float((uint32_t)(127 + k) << 23);
    inv = __uint_as_float((uint32_t)(127 - k) << 23);
}

// Split 8 scaled values into NP e4m3 planes; plane p -> (even elements, odd
// elements) as the b0/b1 register pair of one MMA k-step.
template <int NP>
__device__ __forceinline__ void make_planes(float (&r)[8], uint2 (&out)[NP])
{
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        const uint32_t e0 = to_e4m3x2(r[0], r[2]), e1 = to_e4m3x2(r[4], r[6]);
        const uint32_t o0 = to_e4m3x2(r[1], r[3]), o1 = to_e4m3x2(r[5], r[7]);
        out[p] = make_uint2(e0 | (e1 << 16), o0 | (o1 << 16));
        if (p + 1 < NP) {
            const float2 a = from_e4m3x2(e0), b = from_e4m3x2(e1), c = from_e4m3x2(o0), d = from_e4m3x2(o1);
            r[0] -= a.x; r[2] -= a.y; r[4] -= b.x; r[6] -= b.y;
            r[1] -= c.x; r[3] -= c.y; r[5] -= d.x; r[7] -= d.y;
        }
    }
}

__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                 "%3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
                 "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
                 : "memory");
}

// Optional phase trace (built with -DMX_PD_TRACE): consumer thread 0 of every
// CTA records %globaltimer at the phase edges of one layer.
#ifdef MX_PD_TRACE
constexpr int kTraceLayer = 10, kTraceCtas = 160, kTracePts = 32;
__device__ unsigned long long g_pd_trace[kTraceCtas][kTracePts];
#define PD_STAMP(l, i)                                                                            \
    do {                                                                                          \
        if (threadIdx.x == 0 && (l) == kTraceLayer && blockIdx.x < kTraceCtas)                    \
            g_pd_trace[blockIdx.x][i] = global_ns();                                              \
    } while (0)
// the same from whichever thread reaches it (the caller picks one)
#define PD_STAMP_ANY(l, i)                                                                        \
    do {                                                                                          \
        if ((l) == kTraceLayer && blockIdx.x < kTraceCtas)                                        \
            g_pd_trace[blockIdx.x][i] = global_ns();                                              \
    } while (0)
#else
#define PD_STAMP(l, i) \
    do {               \
    } while (0)
#define PD_STAMP_ANY(l, i) \
    do {                   \
    } while (0)
#endif

// ------------------------------------------------------------ shared memory

struct Rt {  // routing of the current layer (computed by the consumer warps)
    int *n_act;       // [1]
    int *act_e;       // [amax] active experts, ascending
    int *act_n;       // [amax] slots of each
    int *act_slot;    // [amax][4] slot ids s = t*K + k, ascending
    int *slot_e;      // [T*K]
    float *slot_w;    // [T*K] (first the selected logits, then the weights)
    int *emap;        // [E] expert -> active index (then act_r, [amax]: the blob
                      // record of each active expert; act_r(rt, E) gives it)
    uint32_t *emask;  // [16]
};

// The record array follows emap: no pointer of its own, so that the hot loops
// keep the registers they had.
__device__ __forceinline__ int *act_r(const Rt &rt, int E) { return rt.emap + E; }

struct Smem {
    uint64_t *full, *empty, *route_bar;
    uint8_t *ring;         // NR slots: gate/up items (8 + 8 rows x D) and down items (D/4 rows x 64 columns)
    uint8_t *xraw;         // layer input x_l (act dtype) [T][D]
    uint8_t *xq;           // x_l after the optional rmsnorm (act dtype) [T][D]
    float *xg;             // [T][GD] group sums of xq, canonical order
    uint8_t *xpl;          // planes of xq (layout A, NB plane pairs)
    float *uh;             // [64][4] hidden values of the current unit
    uint8_t *upl;          // [4][256] their e4m3 planes (2 pairs)
    float *ux, *ufo;       // [4] their sums and plane back factors
    uint16_t *dss;         // [2][2][D/4] down-item scales and biases (BF16 bits), two buffers
    float *lg;             // [T][E] logits of the layer
    float *pr;             // scratch
    float *fx;             // [T] x plane back factors 2^(9-k)
    float *rn, *xsc;       // [T] rmsnorm factors, x plane scales
    int *vmax;             // [T] plane maxima (float bits)
    float *yfx;            // [2] fixed-point factor of the layer's y and its inverse, then
                           // yfx + 4: [T] shared-branch gates, yfx + 8: [T] post-norm factors
    int *flag;             // [4]
    uint8_t *zero;         // 16 zero bytes
    Rt rt;
};

__device__ __forceinline__ Smem carve(uint8_t *sm, const PdParams &p)
{
    const PdSmem &o = p.sm;
    Smem s;
    s.full = reinterpret_cast<uint64_t *>(sm);
    s.empty = s.full + o.NR;
    s.route_bar = s.empty + o.NR;
    s.ring = sm + o.ring;
    s.xraw = sm + o.xraw;
    s.xq = sm + o.xq;
    s.xg = reinterpret_cast<float *>(sm + o.xg);
    s.xpl = sm + o.xpl;
    s.uh = reinterpret_cast<float *>(sm + o.uh);
    s.upl = sm + o.upl;
    s.dss = reinterpret_cast<uint16_t *>(sm + o.dss);
    s.lg = reinterpret_cast<float *>(sm + o.lg);
    s.pr = reinterpret_cast<float *>(sm + o.pr);
    float *m = reinterpret_cast<float *>(sm + o.misc);
    const int TK = p.T * p.K;
    s.fx = m;
    s.rn = m + 4;
    s.xsc = m + 8;
    s.flag = reinterpret_cast<int *>(m + 12);
    s.ux = m + 16;
    s.ufo = m + 20;
    s.vmax = reinterpret_cast<int *>(m + 24);  // [T]
    s.yfx = m + 28;
    int *r = reinterpret_cast<int *>(sm + o.rt);
    const int amax = TK < p.E ? TK : p.E;
    s.rt.n_act = r;
    s.rt.emask = reinterpret_cast<uint32_t *>(r + 4);
    s.rt.act_e = r + 20;
    s.rt.act_n = s.rt.act_e + amax;
    s.rt.act_slot = s.rt.act_n + amax;
    s.rt.slot_e = s.rt.act_slot + 4 * amax;
    s.rt.slot_w = reinterpret_cast<float *>(s.rt.slot_e + TK);
    s.rt.emap = reinterpret_cast<int *>(s.rt.slot_w + TK);
    s.zero = sm + o.zero;
    return s;
}

// ------------------------------------------------------------- sync helpers

__device__ __forceinline__ int *abort_word(const PdParams &p) { return p.ctr + p.n_layers * p.cstride + 1; }

__device__ __forceinline__ void set_abort(const PdParams &p) { atomicExch(abort_word(p), 1); }

// Spin until *c >= target.  False after p.wait_ns (error word set) or when
// another CTA has given up.
__device__ bool gwait(const int *c, int target, const PdParams &p)
{
    if (ld_acquire(c) >= target)
        return true;
    const unsigned long long t0 = global_ns();
    const int *ab = abort_word(p);
    for (unsigned it = 0;; ++it) {
        __nanosleep(32);
        if (ld_acquire(c) >= target)
            return true;
        if ((it & 63u) == 63u) {
            if (ld_acquire(ab))
                return false;
            if (global_ns() - t0 > p.wait_ns) {
                atomicOr(p.err, kErrTimeout);
                set_abort(p);
                return false;
            }
        }
    }
}

// Producer-side wait: polls with a short sleep, so the waiting warp leaves the
// issue slots of its scheduler to the consumer warps.  Gives up after
// p.wait_ns, or once any CTA has given up (its consumers may then never
// release a slot or publish a routing).
__device__ __forceinline__ bool pwait_sleepy(uint64_t *bar, uint32_t parity, const PdParams &p)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    const int *ab = abort_word(p);
    for (unsigned it = 0; !mbar_try_wait(bar, parity); ++it) {
        __nanosleep(64);
        if ((it & 63u) == 63u && ld_acquire(ab))
            return false;
        if (global_ns() - t0 > p.wait_ns) {
            atomicOr(p.err, kErrTimeout);
            set_abort(p);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool pwait(uint64_t *bar, uint32_t parity, const PdParams &p)
{
    if (mbar_wait(bar, parity, p.err))
        return true;
    set_abort(p);
    return false;
}

__device__ __forceinline__ void csync() { named_sync(1, kCT); }

// Consumer barrier that also ANDs a per-thread verdict, so every consumer
// thread leaves with the same answer (a wait may give up on one thread and not
// on another).
__device__ __forceinline__ bool csync_and(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "barrier.cta.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "r"(kCT)
                 : "memory");
    return r != 0;
}

// All consumer threads: thread 0 waits for *c >= target; returns the verdict to all.
__device__ bool cwait(const int *c, int target, const PdParams &p, const Smem &s)
{
    if (threadIdx.x == 0)
        s.flag[0] = gwait(c, target, p) ? 1 : 0;
    csync();
    const bool ok = s.flag[0] != 0;
    csync();
    return ok;
}

__device__ __forceinline__ void red_add(int *c, int v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(c), "r"(v) : "memory");
}

// The down projections' partial sums are added into y in 64-bit fixed point:
// integer addition is associative, so y does not depend on the order in which
// CTAs arrive.  The unit is 2^-32 / f with a per-layer power of two f that
// follows the square of the block input's magnitude (the hidden vectors are
// products of two projections of x, and y is linear in them): with E =
// floor(log2(max |x|)) over the layer's tokens, f = 2^(4 - 2E), clamped to
// 2^[-100, 100] -- f = 1 for inputs of magnitude 4..8.  Each partial sum must
// satisfy |v f| < 2^23 (at most 2^23 units of 2^32: a few hundred additions
// stay far inside the 64-bit range); a partial outside that range is not
// added and sets kErrRange in the error word.
constexpr float kFix = 4294967296.0f;         // 2^32
constexpr float kUnfix = 2.3283064365386963e-10f;  // 2^-32
constexpr float kFixLimit = 8388608.0f;       // 2^23

// The layer's factor f (and 1/f) from the largest input magnitude m.
__device__ __forceinline__ void fix_factor(float m, float &f, float &inv)
{
    int E = m > 0.f ? (int)((__float_as_uint(m) >> 23) & 0xFF) - 127 : 0;
    int k = 4 - 2 * E;
    k = k > 100 ? 100 : (k < -100 ? -100 : k);
    f = __uint_as_float((uint32_t)(127 + k) << 23);
    inv = __uint_as_float((uint32_t)(127 - k) << 23);
}
// round(v * 2^32) as a 64-bit integer, exact for |v| < 2^23, on the integer
// and fp32 pipes only (no float-to-integer conversion).  A = |v| 2^32 is
// exact (a power-of-two scaling).  Below 2^23, A + 2^23 is a float whose ulp
// is 1, so the addition rounds A to nearest even and the sum's bits minus
// those of 2^23 are round(A) (a carry into the exponent yields 2^23 as well).
// From 2^23 up A is an integer: its significand with the hidden bit, shifted
// left by (biased exponent - 150) <= 31.  Round to nearest even is
// odd-symmetric, so the sign is applied last.
__device__ __forceinline__ long long to_fix(float v)
{
    const float A = fabsf(v) * kFix;
    const uint32_t b = __float_as_uint(A);
    const bool small = A < 8388608.0f;
    const uint32_t rs = __float_as_uint(A + 8388608.0f) - 0x4B000000u;
    const uint32_t mant = (b & 0x7FFFFFu) | 0x800000u, sh = (b >> 23) - 150u;
    const uint32_t lo = small ? rs : __funnelshift_l(0u, mant, sh);
    const uint32_t hi = small ? 0u : __funnelshift_l(mant, 0u, sh);
    const long long m = (long long)(((unsigned long long)hi << 32) | lo);
    return v < 0.f ? -m : m;
}

// The fixed-point sum back as a float: hi + lo 2^-32 (|hi| < 2^24 is exact;
// within 2 ulp of the exact value, and the same bits on every call).
__device__ __forceinline__ float from_fix(long long q)
{
    const int hi = (int)(q >> 32);
    const unsigned lo = (unsigned)(q & 0xffffffffll);
    return (float)hi + __uint2float_rn(lo) * kUnfix;
}

// Adds v f into the fixed-point sum; a value outside the range adds 0 and
// sets `bad` (the caller reports it once, kErrRange), so the hot loop has no
// branch around the add.
__device__ __forceinline__ void red_fix(long long *y, float v, float f, bool &bad)
{
    float a = v * f;
    const bool in = fabsf(a) < kFixLimit;
    bad |= !in;
    a = in ? a : 0.f;
    const long long q = to_fix(a);
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(y), "l"(q) : "memory");
}

// ---------------------------------------------------------------- the math

// Gate/up item on one warp: 8 gate rows -> MMA rows 0-7, 8 up rows -> rows
// 8-15, all G groups of K.  Slot layout: gate tile [G][8][32 B], up tile
// [G][8][32 B], gate.s, gate.b, up.s, up.b ([8][G] BF16).  bp: this lane's B
// column (plane pair) for group 0; bgs/bms/bnbs: strides of group, k-step,
// plane pair.  fo, xgo: the lane's output column (slot c; xgo 16-byte
// aligned).  Four groups in flight, the scale and bias sums kept apart, so the
// loop carries no long dependency chain.  Lane output: gate and up dot products
// of row gid, column slot c.
template <int NB>
__device__ __forceinline__ void gu_item(const uint8_t *st, int G, const uint8_t *bp, int bgs, int bms, int bnbs,
                                        float fo, const float *xgo, float &accg, float &accu)
{
    const int lane = threadIdx.x & 31, gid = lane >> 2, c = lane & 3;
    const uint8_t *gt = st + gid * 32 + c * 8, *ut = gt + 256 * G;
    const uint16_t *sc = reinterpret_cast<const uint16_t *>(st + 512 * G) + gid * G;
    const uint16_t *sg = sc, *bg = sc + 8 * G, *su = sc + 16 * G, *bu = sc + 24 * G;
    float pg[4] = {0.f, 0.f, 0.f, 0.f}, pu[4] = {0.f, 0.f, 0.f, 0.f};
    float qg[4] = {0.f, 0.f, 0.f, 0.f}, qu[4] = {0.f, 0.f, 0.f, 0.f};
    // the MMA part of group g: the row's gate and up dot products (plane
    // columns summed)
    auto dots = [&](int g, float &Rg, float &Ru) {
        const uint2 wg = lds64(gt + 256 * g), wu = lds64(ut + 256 * g);
        Rg = 0.f;
        Ru = 0.f;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const uint2 b0 = lds64(bp + g * bgs + nb * bnbs), b1 = lds64(bp + g * bgs + bms + nb * bnbs);
            mma_fp8(d, wg.x & kLo, wu.x & kLo, (wg.x >> 4) & kLo, (wu.x >> 4) & kLo, b0.x, b0.y);
            mma_fp8(d, wg.y & kLo, wu.y & kLo, (wg.y >> 4) & kLo, (wu.y >> 4) & kLo, b1.x, b1.y);
            Rg += d[0] + d[1];
            Ru += d[2] + d[3];
        }
    };
    int g = 0;
    if ((G & 3) == 0) {
        // four groups at a time; their scales, biases and x sums in vector loads
        for (; g < G; g += 4) {
            const uint2 s4g = lds64(reinterpret_cast<const uint8_t *>(sg + g));
            const uint2 b4g = lds64(reinterpret_cast<const uint8_t *>(bg + g));
            const uint2 s4u = lds64(reinterpret_cast<const uint8_t *>(su + g));
            const uint2 b4u = lds64(reinterpret_cast<const uint8_t *>(bu + g));
            const float4 X4 = *reinterpret_cast<const float4 *>(xgo + g);
            const uint32_t wsg[2] = {s4g.x, s4g.y}, wbg[2] = {b4g.x, b4g.y}, wsu[2] = {s4u.x, s4u.y},
                           wbu[2] = {b4u.x, b4u.y};
            const float X[4] = {X4.x, X4.y, X4.z, X4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float Rg, Ru;
                dots(g + j, Rg, Ru);
                const int h = j >> 1;
                const float fsg = __uint_as_float(j & 1 ? wsg[h] & 0xFFFF0000u : wsg[h] << 16);
                const float fbg = __uint_as_float(j & 1 ? wbg[h] & 0xFFFF0000u : wbg[h] << 16);
                const float fsu = __uint_as_float(j & 1 ? wsu[h] & 0xFFFF0000u : wsu[h] << 16);
                const float fbu = __uint_as_float(j & 1 ? wbu[h] & 0xFFFF0000u : wbu[h] << 16);
                pg[j] = fmaf(fsg, Rg, pg[j]);
                qg[j] = fmaf(fbg, X[j], qg[j]);
                pu[j] = fmaf(fsu, Ru, pu[j]);
                qu[j] = fmaf(fbu, X[j], qu[j]);
            }
        }
    } else {
        for (; g < G; ++g) {
            float Rg, Ru;
            dots(g, Rg, Ru);
            const float X = xgo[g];
            pg[0] = fmaf(bf2f(sg[g]), Rg, pg[0]);
            qg[0] = fmaf(bf2f(bg[g]), X, qg[0]);
            pu[0] = fmaf(bf2f(su[g]), Ru, pu[0]);
            qu[0] = fmaf(bf2f(bu[g]), X, qu[0]);
        }
    }
    accg = fo * ((pg[0] + pg[1]) + (pg[2] + pg[3])) + ((qg[0] + qg[1]) + (qg[2] + qg[3]));
    accu = fo * ((pu[0] + pu[1]) + (pu[2] + pu[3])) + ((qu[0] + qu[1]) + (qu[2] + qu[3]));
}

// 4-way byte dot products: a's bytes unsigned, b's unsigned / signed.
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Gate/up item on one warp for a single token of BF16 activations: integer
// dot products instead of MMAs (an MMA would carry data in 2 of its 8
// columns).  x is a 16-bit fixed-point vector (x 2^k1, max |x| 2^k1 in
// [2^14, 2^15)) split into two byte planes, lo (unsigned) and hi (signed);
// xp: this lane's planes of group 0, [plane][16 B] per group at 128-byte
// pitch, the bytes of its 16 columns in the nibble order of its two packed
// words (even columns of a word, then odd).  Lane (gid, c) takes columns
// 16c .. 16c + 15 of rows gid (gate) and gid (up): per group 16 byte dot
// products, exact in int32 (|sum| < 2^23, so exact in fp32 too); then the
// group's scale term in fp32, the bias term once per row and group (lane c
// takes every fourth group), and the four lanes of a row added by shuffles.  fo = 2^-k1.  The warp
// takes groups [g0, g1) of the item.  Lane output: that part of the gate and
// up dot products of row gid (every lane of the row).
__device__ __forceinline__ void gu_item_t1(const uint8_t *st, int G, int g0, int g1, const uint8_t *xp, float fo,
                                           const float *xg, float &accg, float &accu)
{
    const int lane = threadIdx.x & 31, gid = lane >> 2, c = lane & 3;
    const uint8_t *gt = st + gid * 32 + c * 8, *ut = gt + 256 * G;
    const uint16_t *sc = reinterpret_cast<const uint16_t *>(st + 512 * G) + gid * G;
    const uint16_t *sg = sc, *bg = sc + 8 * G, *su = sc + 16 * G, *bu = sc + 24 * G;
    float pg[2] = {0.f, 0.f}, pu[2] = {0.f, 0.f}, qg = 0.f, qu = 0.f;
    // the bias terms b_g X_g of the row, once per group: lane c takes groups
    // g0 + c, g0 + c + 4, ... (the shuffles below add the four lanes)
    for (int g = g0 + c; g < g1; g += 4) {
        const float X = xg[g];
        qg = fmaf(bf2f(bg[g]), X, qg);
        qu = fmaf(bf2f(bu[g]), X, qu);
    }
#pragma unroll 2
    for (int n = 0; n < g1 - g0; ++n) {
        const int g = g0 + n, h = n & 1;
        const uint2 wg = lds64(gt + 256 * g), wu = lds64(ut + 256 * g);
        const uint4 x0 = *reinterpret_cast<const uint4 *>(xp + 128 * g);
        const uint4 x1 = *reinterpret_cast<const uint4 *>(xp + 128 * g + 16);
        int g0 = 0, g1 = 0, u0 = 0, u1 = 0;
        {
            const uint32_t lo = wg.x & kLo, hi = (wg.x >> 4) & kLo;
            g0 = dp4a_uu(lo, x0.x, g0);
            g0 = dp4a_uu(hi, x0.y, g0);
            g1 = dp4a_us(lo, x1.x, g1);
            g1 = dp4a_us(hi, x1.y, g1);
        }
        {
            const uint32_t lo = wg.y & kLo, hi = (wg.y >> 4) & kLo;
            g0 = dp4a_uu(lo, x0.z, g0);
            g0 = dp4a_uu(hi, x0.w, g0);
            g1 = dp4a_us(lo, x1.z, g1);
            g1 = dp4a_us(hi, x1.w, g1);
        }
        {
            const uint32_t lo = wu.x & kLo, hi = (wu.x >> 4) & kLo;
            u0 = dp4a_uu(lo, x0.x, u0);
            u0 = dp4a_uu(hi, x0.y, u0);
            u1 = dp4a_us(lo, x1.x, u1);
            u1 = dp4a_us(hi, x1.y, u1);
        }
        {
            const uint32_t lo = wu.y & kLo, hi = (wu.y >> 4) & kLo;
            u0 = dp4a_uu(lo, x0.z, u0);
            u0 = dp4a_uu(hi, x0.w, u0);
            u1 = dp4a_us(lo, x1.z, u1);
            u1 = dp4a_us(hi, x1.w, u1);
        }
        pg[h] = fmaf(bf2f(sg[g]), (float)(g1 * 256 + g0), pg[h]);
        pu[h] = fmaf(bf2f(su[g]), (float)(u1 * 256 + u0), pu[h]);
    }
    float ag = fo * (pg[0] + pg[1]) + qg;
    float au = fo * (pu[0] + pu[1]) + qu;
    ag += __shfl_xor_sync(0xffffffffu, ag, 1);
    au += __shfl_xor_sync(0xffffffffu, au, 1);
    ag += __shfl_xor_sync(0xffffffffu, ag, 2);
    au += __shfl_xor_sync(0xffffffffu, au, 2);
    accg = ag;
    accu = au;
}

// Down slice, one token of BF16 activations: the 16 nibbles of one row that a
// lane holds (columns 16c .. 16c + 15, two packed words) against the same
// columns of the unit's hidden vector as 24-bit fixed point in three byte
// planes (h0, h1 unsigned low and middle bytes, h2 signed high bytes, each in
// the nibble order of the two words).  Each plane's sum is exact in int32 and
// the total |sum| < 16 * 15 * 2^23 < 2^31 too; returned as a float (rounded
// once, to 24 bits).
__device__ __forceinline__ float dn_row_t1(uint2 q, const uint4 &h0, const uint4 &h1, const uint4 &h2)
{
    int g0 = 0, g1 = 0, g2 = 0;
    uint32_t lo = q.x & kLo, hi = (q.x >> 4) & kLo;
    g0 = dp4a_uu(lo, h0.x, g0);
    g0 = dp4a_uu(hi, h0.y, g0);
    g1 = dp4a_uu(lo, h1.x, g1);
    g1 = dp4a_uu(hi, h1.y, g1);
    g2 = dp4a_us(lo, h2.x, g2);
    g2 = dp4a_us(hi, h2.y, g2);
    lo = q.y & kLo;
    hi = (q.y >> 4) & kLo;
    g0 = dp4a_uu(lo, h0.z, g0);
    g0 = dp4a_uu(hi, h0.w, g0);
    g1 = dp4a_uu(lo, h1.z, g1);
    g1 = dp4a_uu(hi, h1.w, g1);
    g2 = dp4a_us(lo, h2.z, g2);
    g2 = dp4a_us(hi, h2.w, g2);
    return (float)(g2 * 65536 + g1 * 256 + g0);
}

// The four lanes c of a row group hold partial sums of 4 rows (a0, a8: rows
// gid, gid + 8 of one tile; b0, b8: the same rows of a second tile); two
// shuffle stages leave each lane one complete row sum, the other partials
// having moved to the lanes that keep them: lane c = 0 -> a0, 1 -> b0,
// 2 -> a8, 3 -> b8.  The additions run in the same order on every call.
__device__ __forceinline__ float transpose_sum4(float a0, float a8, float b0, float b8, int c)
{
    const bool sb = c & 1, s8 = c & 2;
    const float k0 = (sb ? b0 : a0) + __shfl_xor_sync(0xffffffffu, sb ? a0 : b0, 1);
    const float k8 = (sb ? b8 : a8) + __shfl_xor_sync(0xffffffffu, sb ? a8 : b8, 1);
    return (s8 ? k8 : k0) + __shfl_xor_sync(0xffffffffu, s8 ? k0 : k8, 2);
}

// One 16-row x 64-column tile of a unit's down slice (one group), one warp;
// t0: this lane's bytes of the tile (tile + gid * 32 + c * 8); sb0 / sb8: the
// BF16 scale (low half) and bias (high half) of rows gid and gid + 8.  hb: the
// B operands of the unit's hidden planes, the same for every tile.
//   ONE: at most 2 hidden vectors, their 4 planes in the 8 columns of one MMA
//        (column 4v + p); hb[0], hb[1]: the two k-steps; the plane columns of
//        vector v sit in lanes c = 2v and 2v + 1 and are added across them.
//   else: 2 plane pairs in 2 MMAs per k-step; hb = {pair 0 k0, pair 0 k1,
//        pair 1 k0, pair 1 k1}; column 2v + pp.
template <bool ONE>
__device__ __forceinline__ void dn_tile(const uint8_t *t0, const uint2 (&hb)[4], uint32_t sb0, uint32_t sb8,
                                        float fo, float X, float &a0, float &a8)
{
    const uint2 q0 = lds64(t0), q8 = lds64(t0 + 256);
    const uint32_t l0 = q0.x & kLo, l8 = q8.x & kLo, h0 = (q0.x >> 4) & kLo, h8 = (q8.x >> 4) & kLo;
    const uint32_t m0 = q0.y & kLo, m8 = q8.y & kLo, k0 = (q0.y >> 4) & kLo, k8 = (q8.y >> 4) & kLo;
    float R0, R8;
    if constexpr (ONE) {
        float d[4] = {0.f, 0.f, 0.f, 0.f}, f[4] = {0.f, 0.f, 0.f, 0.f};
        mma_fp8(d, l0, l8, h0, h8, hb[0].x, hb[0].y);
        mma_fp8(f, m0, m8, k0, k8, hb[1].x, hb[1].y);
        R0 = (d[0] + d[1]) + (f[0] + f[1]);
        R8 = (d[2] + d[3]) + (f[2] + f[3]);
        R0 += __shfl_xor_sync(0xffffffffu, R0, 1);
        R8 += __shfl_xor_sync(0xffffffffu, R8, 1);
    } else {
        float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
        mma_fp8(d, l0, l8, h0, h8, hb[0].x, hb[0].y);
        mma_fp8(e, l0, l8, h0, h8, hb[2].x, hb[2].y);
        mma_fp8(d, m0, m8, k0, k8, hb[1].x, hb[1].y);
        mma_fp8(e, m0, m8, k0, k8, hb[3].x, hb[3].y);
        R0 = (d[0] + d[1]) + (e[0] + e[1]);
        R8 = (d[2] + d[3]) + (e[2] + e[3]);
    }
    a0 = fmaf(bf2f((uint16_t)(sb0 >> 16)), X, bf2f((uint16_t)sb0) * (R0 * fo));
    a8 = fmaf(bf2f((uint16_t)(sb8 >> 16)), X, bf2f((uint16_t)sb8) * (R8 * fo));
}

// ----------------------------------------------------------- plane builders

// e4m3 planes (2 pairs) of nvec fp32 vectors of G*64 values, row stride ld,
// written by other CTAs (read from L2), zero padded to Gp >= G groups.
//   layout A (per_slot false): g*(256*nvec) + m*(128*nvec) + nb*(64*nvec) + (2v+pp)*32 + c*8
//   layout B (per_slot true):  v*(Gp*256) + g*256 + m*128 + nb*64 + pp*32 + c*8
// Also gsum[v][g] (group sums, 0 on padding) and back[v] = 2^(9-k).
__device__ __forceinline__ size_t plane_off(bool per_slot, int nvec, int Gp, int v, int g, int m, int nb, int pp, int c)
{
    return per_slot ? (size_t)v * Gp * 256 + (size_t)g * 256 + m * 128 + nb * 64 + pp * 32 + c * 8
                    : (size_t)g * 256 * nvec + (size_t)m * 128 * nvec + (size_t)nb * 64 * nvec + (2 * v + pp) * 32 + c * 8;
}

__device__ __forceinline__ void store_planes(uint8_t *dst, bool per_slot, int nvec, int Gp, int v, int g, int w,
                                             float sc, float (&x)[8])
{
#pragma unroll
    for (int j = 0; j < 8; ++j)
        x[j] *= sc;
    uint2 pl[4];
    make_planes<4>(x, pl);
    const int m = w & 1, c = w >> 1;
#pragma unroll
    for (int p = 0; p < 4; ++p)
        *reinterpret_cast<uint2 *>(dst + plane_off(per_slot, nvec, Gp, v, g, m, p >> 1, p & 1, c)) = pl[p];
}

// x_l (xraw) -> xq (optionally rmsnorm'd, rounded to the act dtype), its group
// sums in the canonical order (the router's X), and its e4m3 planes (T1: the
// byte planes of gu_item_t1).
template <int NB, bool EXT, bool T1>
__device__ void prologue(const PdParams &p, const PdLayer &L, const Smem &s, int l)
{
    (void)l;
    constexpr int es = NB == 1 ? 2 : 4;
    const int tid = threadIdx.x, lane = tid & 31, T = p.T, D = p.D, GD = D / 64;
    auto ld64 = [&](const uint8_t *base, int t, int g, float (&v)[64]) {
        const uint8_t *r = base + ((size_t)t * D + g * 64) * es;
#pragma unroll
        for (int ch = 0; ch < 4 * es; ++ch) {
            const uint4 w = *reinterpret_cast<const uint4 *>(r + 16 * ch);
            if constexpr (es == 2) {
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[8 * ch + 2 * q] = __uint_as_float(u[q] << 16);
                    v[8 * ch + 2 * q + 1] = __uint_as_float(u[q] & 0xFFFF0000u);
                }
            } else {
                v[4 * ch] = __uint_as_float(w.x);
                v[4 * ch + 1] = __uint_as_float(w.y);
                v[4 * ch + 2] = __uint_as_float(w.z);
                v[4 * ch + 3] = __uint_as_float(w.w);
            }
        }
    };
    if (tid < T)
        s.vmax[tid] = 0;
    if (p.pre_norm) {
        // sum of squares: per group an fma chain, then the groups in order
        for (int i = tid; i < T * GD; i += kCT) {
            const int t = i / GD, g = i - t * GD;
            float v[64];
            ld64(s.xraw, t, g, v);
            float q = 0.f;
#pragma unroll
            for (int k = 0; k < 64; ++k)
                q = fmaf(v[k], v[k], q);
            s.pr[i] = q;
        }
        csync();
        if (tid < T) {
            float ss = 0.f;
            for (int g0 = 0; g0 < GD; g0 += 8) {
                float q[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    q[j] = g0 + j < GD ? s.pr[tid * GD + g0 + j] : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (g0 + j < GD)
                        ss = ss + q[j];
            }
            s.rn[tid] = 1.0f / sqrtf(ss / (float)D + p.eps);
        }
    }
    csync();
    PD_STAMP(l, 24);
    // elementwise: xq = round(x * r), the magnitude maximum per token
    {
        const int n8 = T * D / 8;  // 8-value words
        for (int i = tid; i < n8; i += kCT) {
            const int t = (8 * i) / D;
            float v[8];
            if constexpr (es == 2) {
                const uint4 w = reinterpret_cast<const uint4 *>(s.xraw)[i];
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[2 * q] = __uint_as_float(u[q] << 16);
                    v[2 * q + 1] = __uint_as_float(u[q] & 0xFFFF0000u);
                }
            } else {
                const float4 a = reinterpret_cast<const float4 *>(s.xraw)[2 * i];
                const float4 b = reinterpret_cast<const float4 *>(s.xraw)[2 * i + 1];
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            }
            float mx = 0.f;
            if (p.pre_norm) {
                const float r = s.rn[t];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    v[k] = es == 2 ? bf2f(f2bf(v[k] * r)) : v[k] * r;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mx = fmaxf(mx, fabsf(v[k]));
            if constexpr (es == 2) {
                uint4 w;
                w.x = (__float_as_uint(v[0]) >> 16) | (__float_as_uint(v[1]) & 0xFFFF0000u);
                w.y = (__float_as_uint(v[2]) >> 16) | (__float_as_uint(v[3]) & 0xFFFF0000u);
                w.z = (__float_as_uint(v[4]) >> 16) | (__float_as_uint(v[5]) & 0xFFFF0000u);
                w.w = (__float_as_uint(v[6]) >> 16) | (__float_as_uint(v[7]) & 0xFFFF0000u);
                reinterpret_cast<uint4 *>(s.xq)[i] = w;
            } else {
                reinterpret_cast<float4 *>(s.xq)[2 * i] = make_float4(v[0], v[1], v[2], v[3]);
                reinterpret_cast<float4 *>(s.xq)[2 * i + 1] = make_float4(v[4], v[5], v[6], v[7]);
            }
            // one shared-memory atomic per token present in the warp (lanes of
            // a warp hold two tokens when D is not a multiple of 256 values)
            const unsigned am = __activemask(), m = __match_any_sync(am, t);
            const int wmx = __reduce_max_sync(m, __float_as_int(mx));
            if (wmx > 0 && lane == __ffs(m) - 1)
                atomicMax(&s.vmax[t], wmx);
        }
        (void)lane;
    }
    csync();
    PD_STAMP(l, 25);
    if (tid < T) {
        float sc, bk;
        if constexpr (T1)
            fixb_scale<16>(__int_as_float(s.vmax[tid]), sc, bk);
        else
            plane_scale(__int_as_float(s.vmax[tid]), sc, bk);
        s.xsc[tid] = sc;
        s.fx[tid] = bk;
    }
    if (tid == 0) {
        int m = 0;
        for (int t = 0; t < T; ++t)
            m = max(m, s.vmax[t]);
        fix_factor(__int_as_float(m), s.yfx[0], s.yfx[1]);
    }
    csync();
    PD_STAMP(l, 26);
    // group sums in the canonical order (the router's X), and the planes
    for (int i = tid; i < T * GD; i += kCT) {
        const int t = i / GD, g = i - t * GD;
        float v[64];
        ld64(s.xq, t, g, v);
        float X = 0.f;
#pragma unroll
        for (int k = 0; k < 64; ++k)
            X = X + v[k];
        s.xg[i] = X;
    }
    for (int i = tid; i < T * GD * 8; i += kCT) {
        const int t = i / (GD * 8), rem = i - t * GD * 8, g = rem >> 3, w = rem & 7;
        const uint8_t *src = s.xq + ((size_t)t * D + g * 64 + 8 * w) * es;
        float x[8];
        if constexpr (es == 2) {
            const uint4 q = *reinterpret_cast<const uint4 *>(src);
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                x[2 * j] = __uint_as_float(u[j] << 16);
                x[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
            }
        } else {
            const float4 a = *reinterpret_cast<const float4 *>(src), b = *reinterpret_cast<const float4 *>(src + 16);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        }
        if constexpr (T1) {
            // 16-bit fixed point: x 2^k, max |x| 2^k in [2^14, 2^15) (a BF16
            // value there is an integer of at most 32640)
            const float sc = s.xsc[t];
            uint32_t lo[2] = {0u, 0u}, hi[2] = {0u, 0u};  // [even, odd columns]
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int v = __float2int_rn(x[j] * sc);
                lo[j & 1] |= (uint32_t)(v & 0xFF) << (8 * (j >> 1));
                hi[j & 1] |= (uint32_t)((v >> 8) & 0xFF) << (8 * (j >> 1));
            }
            // lane c = w / 2 holds words 2c, 2c + 1 of the group: word w & 1
            uint8_t *dst = s.xpl + (size_t)g * 128 + (w >> 1) * 32 + (w & 1) * 8;
            *reinterpret_cast<uint2 *>(dst) = make_uint2(lo[0], lo[1]);
            *reinterpret_cast<uint2 *>(dst + 16) = make_uint2(hi[0], hi[1]);
            continue;
        }
        const float sc = s.xsc[t];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            x[j] *= sc;
        uint2 pl[2 * NB];
        make_planes<2 * NB>(x, pl);
        const int m = w & 1, c = w >> 1;
#pragma unroll
        for (int q = 0; q < 2 * NB; ++q) {
            const size_t off = (size_t)g * (2 * NB * 64 * T) + (size_t)m * (NB * 64 * T) + (size_t)(q >> 1) * (64 * T) +
                               (2 * t + (q & 1)) * 32 + c * 8;
            *reinterpret_cast<uint2 *>(s.xpl + off) = pl[q];
        }
    }
    PD_STAMP(l, 27);
    if (EXT && L.shared_gate) {
        // shared-branch gate sigmoid(g . x): per group an fma chain, then the
        // groups in order
        for (int i = tid; i < T * GD; i += kCT) {
            const int t = i / GD, g = i - t * GD;
            float v[64];
            ld64(s.xq, t, g, v);
            const uint4 *gp = reinterpret_cast<const uint4 *>(L.shared_gate + g * 64);
            float q = 0.f;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint4 w = __ldg(gp + ch);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    q = fmaf(__uint_as_float(u[j] << 16), v[8 * ch + 2 * j], q);
                    q = fmaf(__uint_as_float(u[j] & 0xFFFF0000u), v[8 * ch + 2 * j + 1], q);
                }
            }
            s.pr[i] = q;
        }
        csync();
        if (tid < T) {
            float z = 0.f;
            for (int g = 0; g < GD; ++g)
                z = z + s.pr[tid * GD + g];
            s.yfx[4 + tid] = 1.0f / (1.0f + expf(-z));
        }
    }
    csync();
}

// Router rows r = blockIdx.x, + gridDim.x, ...: logits in the fixed order of
// the header.  rq/rsv/rbv: the first row's bytes and affine terms, prefetched.
template <int NB, bool EXT>
__device__ void router_rows(const PdParams &p, const PdLayer &L, const Smem &s, uint4 (&rq)[4], float rsv,
                            float rbv)
{
    constexpr int es = NB == 1 ? 2 : 4;
    const int tid = threadIdx.x, T = p.T, D = p.D, GD = D / 64, C = blockIdx.x, NC = gridDim.x;
    float *P = s.pr;            // [GD][T]
    float *sv = s.pr + GD * T;  // [GD]
    float *bv = sv + GD;        // [GD]
    float *xx = bv + GD;        // [GD][T] group sums of the scaled input (with router_scale)
    // With router_scale the router reads (x_i * rs_i) * rcoef in fp32.
    const bool scaled = EXT && L.router_scale != nullptr;
    for (int r = C; r < p.E; r += NC) {
        if (r != C && tid < GD) {
            const uint4 *q = reinterpret_cast<const uint4 *>(L.rw + (size_t)r * (D / 4) + (size_t)tid * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                rq[j] = __ldg(q + j);
            rsv = bf2f(__ldg(L.rs + (size_t)r * GD + tid));
            rbv = bf2f(__ldg(L.rb + (size_t)r * GD + tid));
        }
        if (tid < GD) {
            const int g = tid;
            sv[g] = rsv;
            bv[g] = rbv;
            for (int t = 0; t < T && scaled; ++t) {
                // 8 columns at a time: the scaled values (x_i * rs_i) * rcoef,
                // their sum and the dot product, both in column order
                const uint8_t *xr = s.xq + ((size_t)t * D + g * 64) * es;
                const uint4 *rp = reinterpret_cast<const uint4 *>(L.router_scale + g * 64);
                float X = 0.f, acc = 0.f;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float xv[8];
                    if constexpr (es == 2) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(xr + 16 * ch);
                        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            xv[2 * q] = __uint_as_float(u[q] << 16);
                            xv[2 * q + 1] = __uint_as_float(u[q] & 0xFFFF0000u);
                        }
                    } else {
                        const float4 a = *reinterpret_cast<const float4 *>(xr + 32 * ch);
                        const float4 b = *reinterpret_cast<const float4 *>(xr + 32 * ch + 16);
                        xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
                        xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
                    }
                    const uint4 s4 = __ldg(rp + ch);
                    const uint32_t su[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float sc = __uint_as_float((j & 1) ? (su[j >> 1] & 0xFFFF0000u) : (su[j >> 1] << 16));
                        xv[j] = __fmul_rn(__fmul_rn(xv[j], sc), L.rcoef);
                        X = X + xv[j];
                    }
                    const uint4 r4 = rq[ch >> 1];
                    const uint32_t w0 = (ch & 1) ? r4.z : r4.x, w1 = (ch & 1) ? r4.w : r4.y;
                    acc = fmaf(byte_f<0>(w0), xv[0], acc);
                    acc = fmaf(byte_f<1>(w0), xv[1], acc);
                    acc = fmaf(byte_f<2>(w0), xv[2], acc);
                    acc = fmaf(byte_f<3>(w0), xv[3], acc);
                    acc = fmaf(byte_f<0>(w1), xv[4], acc);
                    acc = fmaf(byte_f<1>(w1), xv[5], acc);
                    acc = fmaf(byte_f<2>(w1), xv[6], acc);
                    acc = fmaf(byte_f<3>(w1), xv[7], acc);
                }
                xx[g * T + t] = X;
                P[g * T + t] = acc;
            }
            for (int t = 0; t < T && !scaled; ++t) {
                float xv[64];
                const uint8_t *xr = s.xq + ((size_t)t * D + g * 64) * es;
#pragma unroll
                for (int ch = 0; ch < 4 * es; ++ch) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(xr + 16 * ch);
                    if constexpr (es == 2) {
                        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            xv[8 * ch + 2 * q] = __uint_as_float(u[q] << 16);
                            xv[8 * ch + 2 * q + 1] = __uint_as_float(u[q] & 0xFFFF0000u);
                        }
                    } else {
                        xv[4 * ch] = __uint_as_float(w.x);
                        xv[4 * ch + 1] = __uint_as_float(w.y);
                        xv[4 * ch + 2] = __uint_as_float(w.z);
                        xv[4 * ch + 3] = __uint_as_float(w.w);
                    }
                }
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t w = j % 4 == 0 ? rq[j / 4].x : j % 4 == 1 ? rq[j / 4].y
                                     : j % 4 == 2 ? rq[j / 4].z : rq[j / 4].w;
                    acc = fmaf(byte_f<0>(w), xv[4 * j], acc);
                    acc = fmaf(byte_f<1>(w), xv[4 * j + 1], acc);
                    acc = fmaf(byte_f<2>(w), xv[4 * j + 2], acc);
                    acc = fmaf(byte_f<3>(w), xv[4 * j + 3], acc);
                }
                P[g * T + t] = acc;
            }
        }
        csync();
        if (tid < T) {
            float acc = 0.f;
            for (int g0 = 0; g0 < GD; g0 += 8) {
                float a[8], b[8], c[8], d[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int g = g0 + j < GD ? g0 + j : GD - 1;
                    a[j] = sv[g];
                    b[j] = P[g * T + tid];
                    c[j] = bv[g];
                    d[j] = scaled ? xx[g * T + tid] : s.xg[tid * GD + g];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (g0 + j < GD) {
                        acc = fmaf(a[j], b[j], acc);
                        acc = fmaf(c[j], d[j], acc);
                    }
                }
            }
            p.logits[(size_t)tid * p.E + r] = acc;
        }
        csync();
    }
}

// Top-k (descending, ties to the lower expert, NaN as -inf), softmax of the
// selected logits times the per-expert scale, and the grouping of slots by
// expert (ascending expert, ascending slot).  All consumer threads.
template <bool EXT>
__device__ void route_tables(const PdParams &p, const PdLayer &L, const Smem &s, int l)
{
    (void)l;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, T = p.T, E = p.E, K = p.K;
    const Rt &rt = s.rt;
    // top-K and softmax, one warp per token: lane l holds the logits of
    // experts l, l + 32, ... as order-preserving keys (NaN as -inf); K rounds
    // of a warp maximum, ties to the lower expert; lane k keeps round k
    if (E <= 128 && warp < T) {
        const int t = warp;
        constexpr int kPer = 4;
        uint32_t key[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int e = lane + 32 * j;
            float v = e < E ? __ldcg(p.logits + (size_t)t * E + e) : -INFINITY;
            if (isnan(v))
                v = -INFINITY;
            const uint32_t u = __float_as_uint(v);
            // monotone in v; taken and absent entries get 0, below every key
            key[j] = e < E ? (u & 0x80000000u ? ~u : u | 0x80000000u) : 0u;
        }
        PD_STAMP(l, 28);
        int mye = 0;
        float myv = 0.f;
        for (int k = 0; k < K; ++k) {
            uint32_t best = 0u;
            int bj = 0;
#pragma unroll
            for (int j = 0; j < kPer; ++j)
                if (key[j] > best) {
                    best = key[j];
                    bj = j;
                }
            const uint32_t mx = __reduce_max_sync(0xffffffffu, best);
            const int win = __reduce_min_sync(0xffffffffu, best == mx ? lane + 32 * bj : INT_MAX);
            if (lane == (win & 31)) {
#pragma unroll
                for (int j = 0; j < kPer; ++j)
                    if (j == (win >> 5))
                        key[j] = 0u;
            }
            if (lane == k) {
                mye = win;
                myv = __uint_as_float(mx & 0x80000000u ? mx & 0x7FFFFFFFu : ~mx);
            }
        }
        // softmax of the selected logits shifted by the largest (round 0),
        // the sum in ascending k, times the per-expert scale
        const float m = __shfl_sync(0xffffffffu, myv, 0);
        const float ex = lane < K ? expf(myv - m) : 0.f;
        float sum = 0.f;
        for (int k = 0; k < K; ++k)
            sum += __shfl_sync(0xffffffffu, ex, k);
        if (lane < K) {
            float x = ex / sum;
            if (L.pes)
                x = x * __ldg(L.pes + mye);
            rt.slot_e[t * K + lane] = mye;
            rt.slot_w[t * K + lane] = x;
            if (blockIdx.x == 0) {
                L.topk_idx[t * K + lane] = mye;
                L.topk_w[t * K + lane] = x;
            }
            if (T == 1) {
                // one token: K distinct experts with one slot each, active in
                // top-k order (any fixed order of the active experts will do:
                // it only assigns units to CTAs)
                rt.act_e[lane] = mye;
                if constexpr (EXT)
                    act_r(rt, E)[lane] = expert_record(L.slot, L.n_slots, mye, p.err);
                rt.act_n[lane] = 1;
                rt.act_slot[4 * lane] = lane;
                rt.emap[mye] = lane;
            }
        }
        if (T == 1 && lane == 0)
            *rt.n_act = K;
        PD_STAMP(l, 29);
    }
    if (E <= 128 && T == 1) {
        csync();
        return;
    }
    if (E > 128) {
        // more than 128 experts: each logit's rank by a scan of its row
        for (int i = tid; i < T * E; i += kCT) {
            const float v = __ldcg(p.logits + i);
            s.lg[i] = isnan(v) ? -INFINITY : v;
        }
        csync();
        for (int i = tid; i < T * E; i += kCT) {
            const int t = i / E, e = i - t * E;
            const float *row = s.lg + t * E;
            const float v = row[e];
            int rank = 0, j = 0;
            if ((E & 3) == 0) {  // rows 16-byte aligned: four logits per load
#pragma unroll 4
                for (; j < E; j += 4) {
                    const float4 u = *reinterpret_cast<const float4 *>(row + j);
                    rank += ((u.x > v) || (u.x == v && j < e)) + ((u.y > v) || (u.y == v && j + 1 < e)) +
                            ((u.z > v) || (u.z == v && j + 2 < e)) + ((u.w > v) || (u.w == v && j + 3 < e));
                }
            }
            for (; j < E; ++j) {
                const float u = row[j];
                rank += (u > v) || (u == v && j < e);
            }
            if (rank < K) {
                rt.slot_e[t * K + rank] = e;
                rt.slot_w[t * K + rank] = v;
            }
        }
        csync();
        // softmax on warp 1 (lane = token) while warp 0 groups the slots
        if (warp == 1 && lane < T) {
            const int t = lane;
            float *w = rt.slot_w + t * K;
            const float m = w[0];
            float sum = 0.f;
            for (int k = 0; k < K; ++k) {
                w[k] = expf(w[k] - m);
                sum += w[k];
            }
            for (int k = 0; k < K; ++k) {
                float x = w[k] / sum;
                if (L.pes)
                    x = x * __ldg(L.pes + rt.slot_e[t * K + k]);
                w[k] = x;
                if (blockIdx.x == 0) {
                    L.topk_idx[t * K + k] = rt.slot_e[t * K + k];
                    L.topk_w[t * K + k] = x;
                }
            }
        }
    }
    csync();
    if (warp == 0) {
        if (lane < 16)
            rt.emask[lane] = 0u;
        __syncwarp();
        const int nw = (E + 31) >> 5;
        for (int i = lane; i < T * K; i += 32) {
            const int e = rt.slot_e[i];
            atomicOr(&rt.emask[e >> 5], 1u << (e & 31));
        }
        __syncwarp();
        const uint32_t bits = lane < nw ? rt.emask[lane] : 0u;
        const int cnt = __popc(bits);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        int j = incl - cnt;
        for (uint32_t b = bits; b; b &= b - 1u, ++j) {
            const int e = 32 * lane + __ffs(b) - 1;
            rt.act_e[j] = e;
            if constexpr (EXT)
                act_r(rt, E)[j] = expert_record(L.slot, L.n_slots, e, p.err);
            rt.act_n[j] = 0;
            rt.emap[e] = j;
        }
        if (lane == 31)
            *rt.n_act = incl;
        __syncwarp();
        for (int t = 0; t < T; ++t) {
            if (lane < K) {
                const int sl = t * K + lane, a = rt.emap[rt.slot_e[sl]];
                rt.act_slot[4 * a + rt.act_n[a]] = sl;
                rt.act_n[a] += 1;
            }
            __syncwarp();
        }
    }
    csync();
}

// ------------------------------------------------------------------ producer

// Units of a layer: shared units u < GS first, then routed units (active
// expert j, block u) as r = j * GI + u; unit id i goes to CTA i mod NC.
__device__ __forceinline__ int first_routed(int C, int NC, int GS) { return ((C - GS) % NC + NC) % NC; }

template <int NB, bool EXT, bool PK>
__device__ void producer(const PdParams &p, const Smem &s)
{
    const int lane = threadIdx.x & 31, C = blockIdx.x, NC = gridDim.x;
    const int D = p.D, GD = D / 64, GI = p.I / 64, GS = p.S / 64, R4 = D / 4, R16 = D / 16;
    const PdSmem &o = p.sm;
    int k = 0;
    bool ok = true;
    // reserve the next ring slot (lane 0 waits; the verdict is the warp's)
    auto take = [&](uint32_t bytes, uint8_t *&dst, uint64_t *&bar) -> bool {
        const int sl = k % o.NR;
        int good = 1;
        if (k >= o.NR && lane == 0)
            good = pwait_sleepy(&s.empty[sl], ((k / o.NR) - 1) & 1, p) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, good, 0))
            return false;
        dst = s.ring + (size_t)sl * o.slot;
        bar = s.full + sl;
        if (lane == 0)
            mbar_arrive_expect_tx(bar, bytes);
        __syncwarp();
        ++k;
        return true;
    };
    // the 12 items of unit (shared or expert e, block u): 8 gate/up items of
    // 8 + 8 rows, then 4 down items of D/4 rows x the block's 64 columns
    auto issue_unit = [&](const PdLayer &L, bool shared, int e, int u) -> bool {
        for (int w = 0; w < 8; ++w) {
            const int rb = 8 * u + w;  // 8-row block of gate/up
            uint8_t *dst;
            uint64_t *bar;
            if (!take(576u * GD, dst, bar))
                return false;
            if (lane == 0) {
                tma_load_4d(dst, shared ? &L.sgate : &L.gate, 0, 8 * rb, 0, e, bar);
                tma_load_4d(dst + 256 * GD, shared ? &L.sup : &L.up, 0, 8 * rb, 0, e, bar);
            } else if (lane <= 4) {
                const int jj = lane - 1;
                const uint16_t *src;
                if (shared) {
                    src = (jj & 1 ? L.sb[jj >> 1] : L.ss[jj >> 1]) + (size_t)8 * rb * GD;
                } else {
                    const uint8_t *rec = L.blob + (uint64_t)e * L.stride;
                    src = reinterpret_cast<const uint16_t *>(rec + (jj & 1 ? L.off_b[jj >> 1] : L.off_s[jj >> 1])) +
                          (size_t)8 * rb * GD;
                }
                bulk_g2s(dst + 512 * GD + jj * 16 * GD, src, 16u * GD, bar);
            }
        }
        // (with the packed down words, each down item also brings its D/4
        // (scale | bias << 16) words, behind its weights)
        for (int q = 0; q < 4; ++q) {
            uint8_t *dst;
            uint64_t *bar;
            if (!take(32u * R4 + (PK ? 4u * R4 : 0u), dst, bar))
                return false;
            if (lane < 4)
                tma_load_4d(dst + lane * 32 * R16, shared ? &L.sdown : &L.down, 0, q * R4 + lane * R16, u, e, bar);
            else if (PK && lane == 4)
                bulk_g2s(dst + 32 * R4, (shared ? L.dsb_s + (size_t)u * D : L.dsb + ((size_t)e * GI + u) * D) + q * R4,
                         4u * R4, bar);
            __syncwarp();
        }
        return true;
    };
    for (int l = 0; l < p.n_layers && ok; ++l) {
        const PdLayer &L = p.L[l];
        for (int u = C; u < GS && ok; u += NC)
            ok = issue_unit(L, true, 0, u);
        if (!ok)
            break;
        // routing of this layer (from the consumers)
        int good = 1;
        if (lane == 0)
            good = pwait_sleepy(s.route_bar, l & 1, p) ? 1 : 0;
        if (!(ok = __shfl_sync(0xffffffffu, good, 0) != 0))
            break;
        const int nr = *s.rt.n_act * GI;
        if (lane == 0 && first_routed(C, NC, GS) < nr)
            PD_STAMP_ANY(l, 23);
        for (int r = first_routed(C, NC, GS); r < nr && ok; r += NC)
            ok = issue_unit(L, false, EXT ? act_r(s.rt, p.E)[r / GI] : s.rt.act_e[r / GI], r % GI);
    }
    // Leave no copy in flight: wait (bounded) for the last item of every slot.
    __syncwarp();
    if (lane == 0)
        for (int j = (k > o.NR ? k - o.NR : 0); j < k; ++j)
            mbar_wait(&s.full[j % o.NR], (j / o.NR) & 1, p.err);
    __syncwarp();
}

// ----------------------------------------------------------------- consumers

// e4m3 planes (2 pairs), the sum X and the back factor of each of the ne
// hidden vectors of a unit (64 values each, uh[row * 4 + v]).  One warp: lane
// = v * 8 + word.
__device__ void unit_planes(const float *uh, int ne, uint8_t *upl, float *ux, float *ufo)
{
    const int lane = threadIdx.x & 31, v = lane >> 3, w = lane & 7;
    float x[8], sm = 0.f, mx = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        x[j] = v < ne ? uh[(8 * w + j) * 4 + v] : 0.f;
        sm += x[j];
        mx = fmaxf(mx, fabsf(x[j]));
    }
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
        sm += __shfl_xor_sync(0xffffffffu, sm, d);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    }
    if (v < ne) {
        float sc, bk;
        plane_scale(mx, sc, bk);
        store_planes(upl, true, ne, 1, v, 0, w, sc, x);
        if (w == 0) {
            ux[v] = sm;
            ufo[v] = bk;
        }
    }
}

// One token: the unit's hidden vector (64 values, uh[4 i]) as 24-bit fixed
// point in the byte planes of dn_row_t1, lane c's 48 bytes at upl + 64 c (low,
// middle, high plane, 16 bytes each); ux = its sum, ufo = 2^-k (h 2^k
// rounded, the largest magnitude in [2^22, 2^23), 2^23 clamped to 2^23 - 1).
// Warp 0.
__device__ void unit_planes_t1(const float *uh, uint8_t *upl, float *ux, float *ufo)
{
    const int lane = threadIdx.x & 31, w = lane & 7;
    float x[8], sm = 0.f, mx = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        x[j] = uh[(8 * w + j) * 4];
        sm += x[j];
        mx = fmaxf(mx, fabsf(x[j]));
    }
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
        sm += __shfl_xor_sync(0xffffffffu, sm, d);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    }
    float sc, inv;
    fixb_scale<24>(mx, sc, inv);
    if (lane < 8) {
        uint32_t b[3][2] = {};  // [plane][even, odd columns]
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int v = min(__float2int_rn(x[j] * sc), 8388607);
#pragma unroll
            for (int pl = 0; pl < 3; ++pl)
                b[pl][j & 1] |= (uint32_t)((v >> (8 * pl)) & 0xFF) << (8 * (j >> 1));
        }
        uint8_t *dst = upl + (w >> 1) * 64 + (w & 1) * 8;
#pragma unroll
        for (int pl = 0; pl < 3; ++pl)
            *reinterpret_cast<uint2 *>(dst + 16 * pl) = make_uint2(b[pl][0], b[pl][1]);
        if (w == 0) {
            ux[0] = sm;
            ufo[0] = inv;
        }
    }
}

template <int NB, bool EXT, bool T1, bool PK>
__device__ void consumers(const PdParams &p, const Smem &s)
{
    constexpr int es = NB == 1 ? 2 : 4;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, c = lane & 3;
    const int C = blockIdx.x, NC = gridDim.x, T = p.T, K = p.K;
    const int D = p.D, I = p.I, S = p.S, GD = D / 64, GI = I / 64, GS = S / 64, R4 = D / 4;
    const PdSmem &o = p.sm;
    int k = 0;  // ring items consumed so far
    bool ok = true;
    const int xgs = 2 * NB * 64 * T, xms = NB * 64 * T, xnbs = 64 * T;  // x planes (layout A)
    for (int l = 0; l < p.n_layers && ok; ++l) {
        const PdLayer &L = p.L[l];
        int *ctr = p.ctr + l * p.cstride;
        long long *y = p.ybuf + (size_t)l * T * D;
        // this CTA's router row: bytes and affine terms do not depend on x
        uint4 rq[4] = {};
        float rsv = 0.f, rbv = 0.f;
        if (C < p.E && tid < GD) {
            const uint4 *q = reinterpret_cast<const uint4 *>(L.rw + (size_t)C * (D / 4) + (size_t)tid * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                rq[j] = __ldg(q + j);
            rsv = bf2f(__ldg(L.rs + (size_t)C * GD + tid));
            rbv = bf2f(__ldg(L.rb + (size_t)C * GD + tid));
        }
        PD_STAMP(l, 0);
        if (l == 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(L.x_in);
            uint4 *dst = reinterpret_cast<uint4 *>(s.xraw);
            for (int i = tid; i < T * D * es / 16; i += kCT)
                dst[i] = __ldg(src + i);
            csync();
        }
        prologue<NB, EXT, T1>(p, L, s, l);
        PD_STAMP(l, 1);
        router_rows<NB, EXT>(p, L, s, rq, rsv, rbv);  // ends with a consumer barrier
        PD_STAMP(l, 2);
        // (hold_cta: a CTA told by the host not to arrive at the first logit
        // exchange, so that every other CTA's bounded wait runs out)
        if (tid == 0 && !(l == 0 && C == p.hold_cta)) {
            __threadfence();
            red_add(ctr + 0, 1);
        }

        // One unit: the 64 hidden rows [64u, 64u + 64) of the shared expert or
        // of active expert j -- their gate/up (warp w: rows 8w..8w+7, all of
        // K), h kept on chip, then that 64-column slice of the down projection
        // for all D outputs, added into y.  No hidden vector leaves the CTA.
        auto unit = [&](bool shared, int j, int u) -> bool {
            const int ne = shared ? T : s.rt.act_n[j];
            // phase trace: the stamps inside a unit cover the CTA's first routed unit
            const bool tr_first = !shared && (j * GI + u) == first_routed(C, NC, GS);
            (void)tr_first;
            bool good = true;
            // the down slice's scales and biases (column u of the [D][G]
            // tables; 16-bit elements at a row pitch TMA cannot take): loaded
            // now, stored once the gate/up work has hidden their latency
            csync();  // every warp is done with the previous unit
            constexpr int kR = kPdMaxD / kCT;
            uint32_t sbv[kR];  // (bias << 16) | scale of rows tid + i * kCT
            if constexpr (!PK) {  // (with PK the down items bring their words)
                const int G = shared ? GS : GI;
                const uint16_t *sp, *bq;
                if (shared) {
                    sp = L.ss[2] + u;
                    bq = L.sb[2] + u;
                } else {
                    const int rj = EXT ? act_r(s.rt, p.E)[j] : s.rt.act_e[j];
                    const uint8_t *rec = L.blob + (uint64_t)rj * L.stride;
                    sp = reinterpret_cast<const uint16_t *>(rec + L.off_s[2]) + u;
                    bq = reinterpret_cast<const uint16_t *>(rec + L.off_b[2]) + u;
                }
#pragma unroll
                for (int i = 0; i < kR; ++i) {
                    const int r = tid + i * kCT;
                    sbv[i] = r < D ? (uint32_t)__ldg(sp + (size_t)r * G) | ((uint32_t)__ldg(bq + (size_t)r * G) << 16)
                                   : 0u;
                }
            }
            if constexpr (T1) {
                // gate/up, one token: the 8 items in halves of their groups;
                // warp w < 4 takes half 0 of item w, then half 1 of item w + 4,
                // warp w >= 4 half 1 of item w - 4, then half 0 of item w, so
                // the last items to land are shared by two warps.  The halves'
                // partial row sums (in x_q's buffer: the router has read it)
                // are added in half order, the same on every call.
                float2 *part = reinterpret_cast<float2 *>(s.xq);  // [item][half][row]
                const int Gh = GD / 2;
                for (int task = 0; task < 2 && good; ++task) {
                    const int it = warp < 4 ? warp + 4 * task : warp - 4 + 4 * task;
                    const int hf = warp < 4 ? task : 1 - task;
                    const int kk = k + it, sl = kk % o.NR;
                    // with fewer slots than items, wait for the release of the
                    // slot's previous item first (see the general case below)
                    const bool w_ok = it < o.NR || pwait(&s.empty[sl], ((kk / o.NR) - 1) & 1, p);
                    if (!__all_sync(0xffffffffu, w_ok && pwait(&s.full[sl], (kk / o.NR) & 1, p))) {
                        good = false;
                        break;
                    }
                    if (tr_first && lane == 0 && ((warp == 0 && task == 0) || (warp == kCW - 1 && task == 1)))
                        PD_STAMP_ANY(l, task == 0 ? 20 : 21);
                    float ag, au;
                    gu_item_t1(s.ring + (size_t)sl * o.slot, GD, hf ? Gh : 0, hf ? GD : Gh, s.xpl + c * 32, s.fx[0],
                               s.xg, ag, au);
                    if (c == 0)
                        part[(it * 2 + hf) * 8 + gid] = make_float2(ag, au);
                    __syncwarp();
                    if (tr_first && lane == 0 && warp == kCW - 1 && task == 1)
                        PD_STAMP_ANY(l, 22);
                    if (lane == 0)
                        mbar_arrive_n(&s.empty[sl], kCW / 2);
                }
                if (!(good = csync_and(good)))
                    return false;
                if (tid < 64) {  // hidden row tid = 8 item + row
                    const float2 a = part[((tid >> 3) * 2) * 8 + (tid & 7)];
                    const float2 b = part[((tid >> 3) * 2 + 1) * 8 + (tid & 7)];
                    float h = gelu_tanh(a.x + b.x) * (a.y + b.y);
                    if (!shared)
                        h *= s.rt.slot_w[s.rt.act_slot[4 * j]];
                    else if (EXT && L.shared_gate)
                        h *= s.yfx[4];
                    s.uh[tid * 4] = h;
                }
            } else {
                // gate/up: warp w owns item k + w
                const int kk = k + warp, sl = kk % o.NR;
                int bt, ot, oslot = 0;
                bool bvalid;
                if (shared) {
                    bvalid = (gid >> 1) < T;
                    bt = gid >> 1;
                    ot = c < T ? c : 0;
                } else {
                    bvalid = (gid >> 1) < ne;
                    bt = bvalid ? s.rt.act_slot[4 * j + (gid >> 1)] / K : 0;
                    oslot = c < ne ? s.rt.act_slot[4 * j + c] : 0;
                    ot = oslot / K;
                }
                const uint8_t *bp = bvalid ? s.xpl + (2 * bt + (gid & 1)) * 32 + c * 8 : s.zero;
                // With fewer slots than gate/up items, item kk reuses the slot of
                // item kk - NR of this unit, which another warp may not have read
                // yet; a parity wait on the slot's full barrier would then look
                // two phases ahead and pass at once.  Wait for that item's
                // release first: then the wait below is exactly one phase ahead.
                bool w_ok = warp < o.NR || pwait(&s.empty[sl], ((kk / o.NR) - 1) & 1, p);
                if (!__all_sync(0xffffffffu, w_ok && pwait(&s.full[sl], (kk / o.NR) & 1, p))) {
                    good = false;
                } else {
                    float ag = 0.f, au = 0.f;
                    gu_item<NB>(s.ring + (size_t)sl * o.slot, GD, bp, bvalid ? xgs : 0, bvalid ? xms : 0,
                                bvalid ? xnbs : 0, s.fx[ot], s.xg + ot * GD, ag, au);
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_n(&s.empty[sl], kCW);
                    if (c < ne) {
                        float h = gelu_tanh(ag) * au;
                        if (!shared)
                            h *= s.rt.slot_w[oslot];
                        else if (EXT && L.shared_gate)
                            h *= s.yfx[4 + ot];
                        s.uh[(8 * warp + gid) * 4 + c] = h;
                    }
                }
            }
            if (!(good = csync_and(good)))
                return false;
            if (tr_first)
                PD_STAMP(l, 6);
            if (warp == 0) {
                if constexpr (T1)
                    unit_planes_t1(s.uh, s.upl, s.ux, s.ufo);
                else
                    unit_planes(s.uh, ne, s.upl, s.ux, s.ufo);
            }
            csync();
            if (tr_first)
                PD_STAMP(l, 7);
            // down: items k + 8 .. k + 11, D/4 rows each; warp w takes row
            // tiles w, w + 8, ... of every item
            const bool bvalid = (gid >> 1) < ne;
            const uint8_t *bp = bvalid ? s.upl + (gid >> 1) * 256 + (gid & 1) * 32 + c * 8 : s.zero;
            // With at most 2 hidden vectors their 4 planes fill the 8 columns of
            // one MMA: half the MMAs and B operands per tile.
            const bool one = ne <= 2;
            uint2 hb[4] = {};
            uint4 h0 = {}, h1 = {}, h2 = {};  // one token: this lane's byte planes of h
            int oc;   // this lane's hidden vector
            bool out; // whether this lane adds its rows into y
            if (T1) {
                h0 = *reinterpret_cast<const uint4 *>(s.upl + c * 64);
                h1 = *reinterpret_cast<const uint4 *>(s.upl + c * 64 + 16);
                h2 = *reinterpret_cast<const uint4 *>(s.upl + c * 64 + 32);
                oc = 0;
                out = true;
            } else if (one) {
                const int v = gid >> 2, pl = gid & 3;
                if (v < ne) {
                    const uint8_t *b1p = s.upl + v * 256 + (pl >> 1) * 64 + (pl & 1) * 32 + c * 8;
                    hb[0] = lds64(b1p);
                    hb[1] = lds64(b1p + 128);
                }
                oc = (c >> 1) < ne ? (c >> 1) : 0;
                out = (c & 1) == 0 && (c >> 1) < ne;
            } else {
                hb[0] = lds64(bp);
                hb[1] = lds64(bp + (bvalid ? 128 : 0));
                hb[2] = lds64(bp + (bvalid ? 64 : 0));
                hb[3] = lds64(bp + (bvalid ? 192 : 0));
                oc = c < ne ? c : 0;
                out = c < ne;
            }
            const int ot = shared ? oc : s.rt.act_slot[4 * j + oc] / K;  // this lane's token
            const float hfo = s.ufo[oc], hX = s.ux[oc], yf = s.yfx[0];
            bool bad = false;  // a partial sum outside the fixed-point range
            long long *yv = y + (size_t)ot * D;
            for (int q = 0; q < 4; ++q) {
                const int kk = k + 8 + q, sl = kk % o.NR;
                // this item's (scale | bias << 16) words: behind its weights in
                // the ring slot (packed table), else staged into buffer q & 1
                // (the barrier also tells that every warp is done with item
                // q - 1, so buffer q & 1, last read for item q - 2, is free)
                const uint32_t *isb;
                if constexpr (PK) {
                    isb = reinterpret_cast<const uint32_t *>(s.ring + (size_t)sl * o.slot + 32 * R4);
                } else {
                    uint32_t *buf = reinterpret_cast<uint32_t *>(s.dss) + (q & 1) * R4;
#pragma unroll
                    for (int i = 0; i < kR; ++i) {
                        const int r = tid + i * kCT - q * R4;
                        if (r >= 0 && r < R4)
                            buf[r] = sbv[i];
                    }
                    csync();
                    isb = buf;
                }
                if (!__all_sync(0xffffffffu, good && pwait(&s.full[sl], (kk / o.NR) & 1, p))) {
                    good = false;
                    continue;
                }
                if (tr_first)
                    PD_STAMP(l, 12 + q);
                const uint8_t *tile = s.ring + (size_t)sl * o.slot + gid * 32 + c * 8;
                const int nrt = R4 / 16;
                for (int rt = warp; rt < nrt; rt += 2 * kCW) {
                    // two row tiles at a time (the second repeats the first past the end)
                    const int rt2 = rt + kCW < nrt ? rt + kCW : rt;
                    const int r0 = 16 * rt + gid, r2 = 16 * rt2 + gid;
                    if constexpr (T1) {
                        // every lane ends with one row of the two tiles (lane c:
                        // tile rt or rt2 by bit 0, row gid or gid + 8 by bit 1)
                        const uint8_t *ta = tile + rt * 512, *tb = tile + rt2 * 512;
                        const float R = transpose_sum4(
                            dn_row_t1(lds64(ta), h0, h1, h2), dn_row_t1(lds64(ta + 256), h0, h1, h2),
                            dn_row_t1(lds64(tb), h0, h1, h2), dn_row_t1(lds64(tb + 256), h0, h1, h2), c);
                        const int r = 16 * ((c & 1) ? rt2 : rt) + gid + 4 * (c & 2);
                        const uint32_t sb = isb[r];
                        const float a = fmaf(bf2f((uint16_t)(sb >> 16)), hX, bf2f((uint16_t)sb) * (R * hfo));
                        if ((c & 1) == 0 || rt2 != rt)
                            red_fix(yv + q * R4 + r, a, yf, bad);
                        continue;
                    }
                    float a0, a8, b0, b8;
                    if (one) {
                        dn_tile<true>(tile + rt * 512, hb, isb[r0], isb[r0 + 8], hfo, hX, a0, a8);
                        dn_tile<true>(tile + rt2 * 512, hb, isb[r2], isb[r2 + 8], hfo, hX, b0, b8);
                    } else {
                        dn_tile<false>(tile + rt * 512, hb, isb[r0], isb[r0 + 8], hfo, hX, a0, a8);
                        dn_tile<false>(tile + rt2 * 512, hb, isb[r2], isb[r2 + 8], hfo, hX, b0, b8);
                    }
                    if (out) {
                        red_fix(yv + q * R4 + r0, a0, yf, bad);
                        red_fix(yv + q * R4 + r0 + 8, a8, yf, bad);
                        if (rt2 != rt) {
                            red_fix(yv + q * R4 + r2, b0, yf, bad);
                            red_fix(yv + q * R4 + r2 + 8, b8, yf, bad);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s.empty[sl]);
                if (tr_first)
                    PD_STAMP(l, 16 + q);
            }
            if (bad)
                atomicOr(p.err, kErrRange);
            k += 12;
            return csync_and(good);
        };

        for (int u = C; u < GS && ok; u += NC)
            ok = unit(true, 0, u);
        PD_STAMP(l, 3);
        // the routing, once every CTA's logits are in
        if (!(ok = csync_and(ok)))
            break;
        PD_STAMP(l, 30);
        if (!(ok = cwait(ctr + 0, NC, p, s)))
            break;
        PD_STAMP(l, 31);
        if (l > 0) {
            // every CTA has rebuilt x_l from y_{l-1} before its logits of layer
            // l arrived: clear this CTA's share of y_{l-1} for the next call
            long long *yp = p.ybuf + (size_t)(l - 1) * T * D;
            const int n = T * D, per = (n + NC - 1) / NC;
            for (int i = C * per + tid; i < min(n, (C + 1) * per); i += kCT)
                yp[i] = 0;
        }
        PD_STAMP(l, 4);
        route_tables<EXT>(p, L, s, l);
        if (tid == 0)
            mbar_arrive(s.route_bar);
        PD_STAMP(l, 5);
        const int nr = *s.rt.n_act * GI;
        for (int r = first_routed(C, NC, GS); r < nr && ok; r += NC)
            ok = unit(false, r / GI, r % GI);
        if (!(ok = csync_and(ok)))
            break;
        PD_STAMP(l, 9);
        if (tid == 0) {
            __threadfence();
            red_add(ctr + 2, 1);
        }

        // ---- y is complete when every CTA has added its part: out = residual + lambda y
        if (!(ok = cwait(ctr + 2, NC, p, s)))
            break;
        PD_STAMP(l, 10);
        // y from L2: twelve loads per thread in flight at a time (all of y at
        // d_model <= 3072, T = 1)
        constexpr int kYB = NB == 1 ? 12 : 6;
        const float yinv = s.yfx[1];
        if (EXT && L.post_norm) {
            // post-FFN norm factor of each token: per group of 64 an fma chain
            // of squares, then the groups in order
            for (int i = tid; i < T * GD; i += kCT) {
                const long long *yp = y + (size_t)i * 64;  // token i / GD, group i % GD
                float q = 0.f;
#pragma unroll 16
                for (int k2 = 0; k2 < 64; ++k2) {
                    const float v = from_fix(__ldcg(yp + k2)) * yinv;
                    q = fmaf(v, v, q);
                }
                s.pr[i] = q;
            }
            csync();
            if (tid < T) {
                float ss = 0.f;
                for (int g = 0; g < GD; ++g)
                    ss = ss + s.pr[tid * GD + g];
                s.yfx[8 + tid] = 1.0f / sqrtf(ss / (float)D + L.post_eps);
            }
            csync();
        }
        // (two instances of the loop, so that the plain one keeps its code)
        auto rebuild = [&](auto pn_tag) {
        constexpr bool PN = decltype(pn_tag)::value;
        for (int i0 = 0; i0 < T * D; i0 += kYB * kCT) {
            long long yq[kYB];
#pragma unroll
            for (int j = 0; j < kYB; ++j) {
                const int i = i0 + tid + j * kCT;
                yq[j] = i < T * D ? __ldcg(y + i) : 0;
            }
#pragma unroll
            for (int j = 0; j < kYB; ++j) {
            const int i = i0 + tid + j * kCT;
            if (i >= T * D)
                break;
            float yv = from_fix(yq[j]) * yinv;
            if constexpr (PN) {
                const int t = i / D;
                yv = __fmul_rn(__fmul_rn(yv, s.yfx[8 + t]), bf2f(__ldg(L.post_norm + (i - t * D))));
            }
            float res = 0.f;
            if (L.res_mode == 1)
                res = es == 2 ? bf2f(reinterpret_cast<const uint16_t *>(s.xraw)[i])
                              : reinterpret_cast<const float *>(s.xraw)[i];
            else if (L.res_mode == 2)
                res = es == 2 ? bf2f(__ldg(reinterpret_cast<const uint16_t *>(L.residual) + i))
                              : __ldg(reinterpret_cast<const float *>(L.residual) + i);
            const float v = res + L.lam * yv;
            if constexpr (es == 2) {
                const uint16_t h = f2bf(v);
                reinterpret_cast<uint16_t *>(s.xraw)[i] = h;
                if (L.x_out && (i % NC) == C)
                    reinterpret_cast<uint16_t *>(L.x_out)[i] = h;
            } else {
                reinterpret_cast<float *>(s.xraw)[i] = v;
                if (L.x_out && (i % NC) == C)
                    reinterpret_cast<float *>(L.x_out)[i] = v;
            }
            }
        }
        };
        if (EXT && L.post_norm)
            rebuild(std::bool_constant<EXT>{});
        else
            rebuild(std::false_type{});
        csync();
        PD_STAMP(l, 11);
    }
    (void)lane;
}

// EXT: the variant with the layer's optional parts (resident-set table,
// router input scale, shared-branch gate, post-FFN norm); plain layers run the
// variant without their code.
// T1: one token of BF16 activations, gate/up on integer dot products.
// PK: every layer has the packed down (scale | bias) words (layout down_sb).
template <int NB, bool EXT, bool T1, bool PK>
__global__ void __launch_bounds__(kPT, 1) pd_kernel(const __grid_constant__ PdParams p)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    const Smem s = carve(sm, p);
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.sm.NR; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], kCW);  // gate/up items: one warp arrives for all; down items: every warp
        }
        mbar_init(s.route_bar, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 4)
        reinterpret_cast<uint32_t *>(s.zero)[threadIdx.x] = 0u;
    // The fixed-point sums y of every layer are zero on entry: the workspace
    // starts zeroed, and every call clears them again once they are read (layer
    // l - 1 after layer l's logit exchange, the last layer at the end), so a
    // shared-expert unit may add into y before any exchange of this call.
    __syncthreads();
    if (threadIdx.x >= kCT)
        producer<NB, EXT, PK>(p, s);
    else
        consumers<NB, EXT, T1, PK>(p, s);
    __syncthreads();
    // The last CTA to finish clears the counters for the next call (unless a
    // wait gave up: then the workspace must be re-initialised).
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        __threadfence();
        int *done = p.ctr + p.n_layers * p.cstride;
        const int old = atomicAdd(done, 1);
        s_last = (old == (int)gridDim.x - 1) && !ld_acquire(abort_word(p));
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        const int n = p.n_layers * p.cstride + 1;  // counters + done
        for (int i = threadIdx.x; i < n; i += kPT)
            p.ctr[i] = 0;
        // every CTA has read the last layer's y: clear it for the next call
        long long *yp = p.ybuf + (size_t)(p.n_layers - 1) * p.T * p.D;
        for (int i = threadIdx.x; i < p.T * p.D; i += kPT)
            yp[i] = 0;
    }
}

// ------------------------------------------------------------------- host

size_t al(size_t n, size_t a) { return (n + a - 1) / a * a; }

} // namespace

// Shared-memory plan; returns false if no ring depth fits.
bool pd_plan(int T, int D, int I, int S, int E, int K, int act, int n_cta, int smem_max, PdSmem *out)
{
    if (T < 1 || T > kPdMaxT || n_cta < 1 || D % 64 || I % 64 || S % 64 || D > kPdMaxD)
        return false;
    const int NB = act == 0 ? 2 : 1;
    const int GD = D / 64, TK = T * K, amax = TK < E ? TK : E;
    const int es = act == 1 ? 2 : 4;
    const size_t scratch = (size_t)4 * std::max((size_t)T * GD, (size_t)GD * (2 * T + 2));
    for (int nr = 8; nr >= 3; --nr) {
        PdSmem o{};
        o.NR = nr;
        o.slot = (int)al((size_t)576 * GD, 128);  // a gate/up item; a down item takes 512 * GD
        size_t off = al((size_t)8 * (2 * o.NR + 1), 128);
        auto take = [&](size_t bytes) {
            const size_t at = off;
            off = al(off + bytes, 128);
            return (int)at;
        };
        o.ring = take((size_t)o.NR * o.slot);
        o.xraw = take((size_t)T * D * es);
        // (one BF16 token: also the 1 KB of gate/up partial sums once the
        // router has read x_q)
        o.xq = take(std::max((size_t)T * D * es, T == 1 && act == 1 ? (size_t)1024 : (size_t)0));
        o.xg = take((size_t)T * GD * 4);
        o.xpl = take((size_t)GD * 128 * NB * T);
        o.uh = take((size_t)64 * 4 * 4);
        o.upl = take((size_t)4 * 256);
        o.dss = take((size_t)2 * 2 * (D / 4) * 2);
        o.lg = take((size_t)T * E * 4);
        o.rt = take((size_t)4 * (20 + 7 * amax + 2 * TK + E));
        o.pr = take(scratch);
        o.misc = take((size_t)4 * 48);
        o.zero = take(16);
        o.total = (int)off;
        if ((long long)off <= smem_max) {
            *out = o;
            return true;
        }
    }
    return false;
}

size_t pd_ctr_ints(int E, int n_layers) { return (size_t)n_layers * (3 + E) + 2; }

#ifdef MX_PD_TRACE
// Copies the phase trace ([kTraceCtas][kTracePts] nanosecond stamps) to host.
extern "C" __attribute__((visibility("default"))) int mx_pd_trace_read(unsigned long long *host)
{
    return (int)cudaMemcpyFromSymbol(host, g_pd_trace, sizeof(g_pd_trace));
}
#endif

namespace {

template <int NB, bool EXT, bool T1, bool PK = false>
cudaError_t launch_nb(const PdParams &p, cudaStream_t st)
{
    auto k = pd_kernel<NB, EXT, T1, PK>;
    cudaError_t e = smem_optin(reinterpret_cast<const void *>(k), (size_t)p.sm.total);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kPT, p.sm.total);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_cta);
    cfg.blockDim = dim3(kPT);
    cfg.dynamicSmemBytes = p.sm.total;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, p);
}

} // namespace

cudaError_t launch_pd(const PdParams &p, cudaStream_t st)
{
    bool ext = false, pk = true;
    for (int l = 0; l < p.n_layers; ++l) {
        const PdLayer &L = p.L[l];
        ext = ext || L.slot || L.router_scale || L.post_norm || L.shared_gate;
        pk = pk && L.dsb;
    }
    if (p.act == 0)
        return ext ? launch_nb<2, true, false>(p, st) : launch_nb<2, false, false>(p, st);
    if (p.T == 1 && pk)
        return ext ? launch_nb<1, true, true, true>(p, st) : launch_nb<1, false, true, true>(p, st);
    if (p.T == 1)
        return ext ? launch_nb<1, true, true>(p, st) : launch_nb<1, false, true>(p, st);
    return ext ? launch_nb<1, true, false>(p, st) : launch_nb<1, false, false>(p, st);
}

} // namespace mx

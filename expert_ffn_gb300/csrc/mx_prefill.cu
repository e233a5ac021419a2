// mx_prefill.cu -- grouped-GEMM path (T > 4 tokens, BF16 activations): grouped
// GEMMs on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// What it computes is the block of the "Mference System design" page: section
// "Prefill" (token/expert pairs grouped into per-expert work, each expert's
// weights streamed once for all its tokens), section "Metal execution" (affine
// decode of the packed weights fused into the expert kernels, GeGLU, the
// weighted expert reduction), section "Why the runtime has this shape" (shared
// expert without a routing weight, layer scalar).
//
// Sequence (one stream):
//   route    router GEMV + top-k + softmax + grouping of slots by expert
//            (mx_route.cu; exact, the canonical logit order)
//   index    inverse permutation; per-expert token-tile offsets
//   gather   x -> FP16 rows (scaled per token by a power of two, operand column
//            order), once in token order (shared expert) and once per slot in
//            expert order (routed experts)
//   gate/up  grouped GEMM, tiles of 128 weight rows x up to kNT tokens:
//            h = gelu(W_gate x) * (W_up x), FP16 [slot][I] and [T][S]
//   down     grouped GEMM: y = W_down h, fp32 [slot][D] and [T][D]
//   combine  out = residual + lambda * (shared + sum_k w_k y_k), k ascending
//
// The GEMM kernel is persistent (one CTA per SM) and warp-specialised
// (16 warps; warp w runs on scheduler w % 4):
//   warp 0      TMA producer of the packed 4-bit weight tiles (a deep ring of
//               stages in shared memory);
//   warp 1      allocates TMEM; the whole warp walks the MMA loop and one
//               elected lane issues tcgen05.mma (A = the FP16 weights in TMEM,
//               B = the activation tile in shared memory, M = 128, N = the
//               tile's tokens rounded up to 16, K = 16, fp32 accumulators in
//               TMEM) and commits to mbarriers;
//   warp 2      TMA producer of the FP16 activation tiles (up to kNT tokens)
//               (SWIZZLE_128B);
//   warps 4-7   epilogue: tcgen05.ld of the accumulators (TMEM lane quadrant
//               = warp % 4), gelu(g) * u for gate/up, fp32 rows for down;
//   warps 8-15  dequantize: w = s*q + b in FP16 (one fused multiply-add on a
//               half2 of exact integers), tcgen05.st into a TMEM weight slot.
// Why FP16 and not BF16: BF16 rounding of the dequantized weights (8-bit
// significand) alone gives ~1.6e-3 relative error per GEMM, above the 1e-3
// rel-L2 bar on BF16 outputs; FP16 (11-bit significand) gives ~2e-4.  BF16
// activations are exact in FP16 after a per-token power-of-two scale.
#include "mx_common.cuh"
#include "mx_internal.h"

#include <cuda_fp16.h>
#include <mutex>

namespace mx {

namespace {

constexpr int kMT = 128;  // weight rows per tile (MMA M)
// Tokens per tile (MMA N, at most).  An expert's tokens at T = 4096, 256
// experts top-8 average 128 with a spread of ~11: 160 keeps nearly every
// expert in one tile, so its weights are dequantized once per row tile
// instead of once more for a tail of a few tokens.
constexpr int kNT = 160;
// Warp roles.  A warp runs on scheduler (warp % 4): each scheduler gets two
// dequantizing warps (8..15), one epilogue warp (4..7, TMEM lane quadrant =
// warp % 4) and one of: the weight producer (0), the MMA warp (1), the
// activation producer (2), nothing (3).
constexpr int kDqWarps = 8;
constexpr int kWarps = 16, kThreads = kWarps * 32;
constexpr uint32_t kDqMask = 0xFF00u;
constexpr int kEpiWarp0 = 4;
constexpr int kBWarp = 2;
static_assert(__builtin_popcount(kDqMask) == kDqWarps, "dequantizing warps");
// A stage covers AT 64-K atoms.  TMEM (512 columns): accumulators in
// columns [0, kACols), the FP16 weight slots (one per stage) above.  Gate/up
// needs 2 kNT columns per accumulator (gate and up side by side), so it keeps
// one accumulator and three one-atom weight slots; down double-buffers its
// kNT-column accumulator and has three two-atom slots.  The activation ring
// (NB stages) and the packed ring (NP stages) live in shared memory; the
// packed ring runs ahead.
constexpr uint32_t kTmemCols = 512, kACols = 2 * kNT;
template <int MODE> struct Cfg;
// TAB: the per-expert unit tables in shared memory (down: short units, the
// lookups recur often); gate/up keeps them out, so that its shared memory
// stays within the 196 KB carve-out and its L1 keeps room for the scale and
// bias loads (gate/up ran 14% slower with 4 KB more shared memory).
template <> struct Cfg<0> { static constexpr int NMAT = 2, NACC = 1, AT = 1, NA = 3, NB = 6, NP = 8; static constexpr bool TAB = false; };
template <> struct Cfg<1> { static constexpr int NMAT = 1, NACC = 2, AT = 2, NA = 3, NB = 3, NP = 8; static constexpr bool TAB = true; };
constexpr int kBTile = kNT * 128;  // bytes of one operand tile (kNT tokens x 64 FP16)

// ------------------------------------------------------------- tcgen05 glue

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the layout TMA writes with SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor: FP16 A and B (K-major), fp32 D, M = 128, N.
__device__ __forceinline__ uint32_t idesc_f16(int n) { return (1u << 4) | ((uint32_t)(n >> 3) << 17) | (8u << 24); }

// D[tmem] (+)= A[tmem] * B[smem]^T
__device__ __forceinline__ void umma_ts(uint32_t dtm, uint32_t atm, uint64_t bd, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(dtm),
                 "r"(atm), "l"(bd), "r"(idesc), "r"(acc)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// One lane of the (converged) warp: true in exactly one lane.
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(ta));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// This warp's 32 TMEM lanes, NW*4 consecutive columns from ta: lane i writes
// r[0..NW*4) of thread i.
template <int NW>
__device__ __forceinline__ void tmem_st(uint32_t ta, const uint32_t (&r)[4 * NW]);

template <>
__device__ __forceinline__ void tmem_st<8>(uint32_t ta, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(ta),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
                 "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
                 "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

template <>
__device__ __forceinline__ void tmem_st<4>(uint32_t ta, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(ta),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                 "%3}], [%4];" ::"r"(smem_u32(dst)),
                 "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                       uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                 "%3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
                 "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
                 : "memory");
}

// ------------------------------------------------------------------- units

struct Unit {
    int shared;  // 1: the shared expert
    int e;       // routed expert
    int r;       // its record in the blob
    int row0;    // first weight row of the tile
    int slot0;   // first token row of the tile (slot position or token)
    int n;       // tokens in the tile
    int kt_n;    // K tiles
};

// Per-expert tables of the launch in shared memory (every role looks units up
// at every unit start), at a fixed offset of the dynamic shared memory:
// token-tile offsets [E+1], then slot offsets, slot counts and blob records [E].
struct UnitTab {
    const int *tt, *off, *cnt, *rec;
    __device__ __forceinline__ explicit UnitTab(const int *base, int E)
        : tt(base), off(base + E + 1), cnt(base + 2 * E + 1), rec(base + 3 * E + 1)
    {
    }
};

// Unit u of the launch: from the shared-memory tables (TAB) or from global memory.
template <bool TAB>
__device__ __forceinline__ Unit unit_of(const PfArgs &a, int u, int nR, const int *tab)
{
    const UnitTab tb(tab, a.E);
    auto ld = [&](const int *smem_p, const int32_t *gmem_p) { return TAB ? *smem_p : __ldg(gmem_p); };
    Unit U;
    if (u < nR * a.FT) {
        const int tile = u / a.FT, f = u - tile * a.FT;
        int lo = 0, hi = a.E;
        while (lo + 1 < hi) {
            const int mid = (lo + hi) >> 1;
            if (ld(tb.tt + mid, a.tt_off + mid) <= tile)
                lo = mid;
            else
                hi = mid;
        }
        const int tt = tile - ld(tb.tt + lo, a.tt_off + lo);
        const int off = ld(tb.off + lo, a.offsets + lo), cnt = ld(tb.cnt + lo, a.counts + lo);
        U.shared = 0;
        U.e = lo;
        U.r = TAB ? tb.rec[lo] : expert_record(a.slot, a.n_slots, lo, a.err);
        U.row0 = kMT * f;
        U.slot0 = off + kNT * tt;
        U.n = min(kNT, off + cnt - U.slot0);
        U.kt_n = a.KT;
    } else {
        const int v = u - nR * a.FT, tt = v / a.FTs, f = v - tt * a.FTs;
        U.shared = 1;
        U.e = 0;
        U.r = 0;
        U.row0 = kMT * f;
        U.slot0 = kNT * tt;
        U.n = min(kNT, a.T - U.slot0);
        U.kt_n = a.KTs;
    }
    return U;
}

// Bounded mbarrier wait of the GEMM: false once this CTA has given up (a
// wait ran past kWaitLimitNs anywhere in the CTA), so one stuck stage costs one
// time limit, not one per remaining stage.
__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t parity, unsigned *err, volatile int *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort)
            return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            *abort = 1;
            return false;
        }
    }
    return true;
}

// The nibbles at bit offsets O and O+16 of v as exact FP16 integers.  A
// nibble in mantissa bits 0-3 under exponent 2^10 reads 1024 + q; one in
// mantissa bits 4-7 under exponent 2^6 reads 64 + q (no shift needed).
template <int O>
__device__ __forceinline__ __half2 nib_h2(uint32_t v)
{
    constexpr uint32_t mask = 0x000F000Fu << (O & 4), magic = (O & 4) ? 0x54005400u : 0x64006400u;
    const uint32_t t = (v & mask) | magic;
    return __hsub2(*reinterpret_cast<const __half2 *>(&t), __float2half2_rn((O & 4) ? 64.0f : 1024.0f));
}

// One packed word (8 weights of a row) -> 8 FP16 weights in operand order
// [0,4,1,5,2,6,3,7] (four half2 words, low half first), w = s*q + b with one
// rounding.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, __half2 b2, uint32_t *out)
{
    const uint32_t w8 = w >> 8;
    const __half2 p0 = __hfma2(nib_h2<0>(w), s2, b2), p1 = __hfma2(nib_h2<4>(w), s2, b2);
    const __half2 p2 = __hfma2(nib_h2<0>(w8), s2, b2), p3 = __hfma2(nib_h2<4>(w8), s2, b2);
    out[0] = *reinterpret_cast<const uint32_t *>(&p0);
    out[1] = *reinterpret_cast<const uint32_t *>(&p1);
    out[2] = *reinterpret_cast<const uint32_t *>(&p2);
    out[3] = *reinterpret_cast<const uint32_t *>(&p3);
}

// Position of column c in the operand order [0,4,1,5,2,6,3,7] of its 8-block.
__device__ __forceinline__ int opos(int c)
{
    const int a = c & 7;
    return (c & ~7) | (a < 4 ? 2 * a : 2 * (a - 4) + 1);
}

// ------------------------------------------------------------ GEMM kernel

// MODE 0: gate/up (two weight matrices, h = gelu(g) * u).  MODE 1: down.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) pf_gemm(const __grid_constant__ PfArgs a)
{
    constexpr int NMAT = Cfg<MODE>::NMAT, NACC = Cfg<MODE>::NACC;
    constexpr int kNA = Cfg<MODE>::NA, kNB = Cfg<MODE>::NB, kNP = Cfg<MODE>::NP, kAt = Cfg<MODE>::AT;
    constexpr uint32_t kPacked = 128 * 32;               // packed bytes of one matrix atom (128 rows x 64 K)
    constexpr uint32_t kPStage = kAt * NMAT * kPacked;   // packed bytes of one stage
    constexpr uint32_t kBStage = kAt * kBTile;           // activation bytes of one stage
    constexpr uint32_t kAccCols = NMAT * kNT;            // TMEM columns of one accumulator buffer
    constexpr uint32_t kSlotCols = kAt * NMAT * 32;      // TMEM columns of one FP16 weight slot
    static_assert(NACC * kAccCols == kACols && kNA * kSlotCols == kTmemCols - kACols, "TMEM split");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *bring = sm;                      // kNB x kBStage
    uint8_t *pring = bring + kNB * kBStage;   // kNP x kPStage
    uint64_t *bars = reinterpret_cast<uint64_t *>(pring + kNP * kPStage);
    uint64_t *p_full = bars, *p_empty = p_full + kNP, *b_full = p_empty + kNP, *b_empty = b_full + kNB;
    uint64_t *a_full = b_empty + kNB, *a_empty = a_full + kNA;
    uint64_t *acc_full = a_empty + kNA, *acc_empty = acc_full + NACC;
    uint64_t *mma_done = acc_empty + NACC;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tslot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int *tab = reinterpret_cast<int *>(bars + 64);  // past the barriers, tslot and abort (512 bytes)
    for (int i = tid; Cfg<MODE>::TAB && i <= a.E; i += kThreads) {
        tab[i] = __ldg(a.tt_off + i);
        if (i < a.E) {
            const int c = __ldg(a.counts + i);
            tab[a.E + 1 + i] = __ldg(a.offsets + i);
            tab[2 * a.E + 1 + i] = c;
            // (only a selected expert must have a record)
            tab[3 * a.E + 1 + i] = c > 0 ? expert_record(a.slot, a.n_slots, i, a.err) : 0;
        }
    }

    if (tid == 0) {
        for (int i = 0; i < kNP; ++i) {
            mbar_init(&p_full[i], 1);
            mbar_init(&p_empty[i], kDqWarps);
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < kNA; ++i) {
            mbar_init(&a_full[i], kDqWarps);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_init(mma_done, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int nR = __ldg(a.tt_off + a.E);
    const int n_units = nR * a.FT + ((a.T + kNT - 1) / kNT) * a.FTs;

    if (warp == 0 || warp == kBWarp) {
        // ---------------------------------------------------------- producers
        // warp 0: packed weight atoms (released by the dequantizing warps);
        // warp kBWarp: activation atoms (released by the MMA).  A stage holds
        // two 64-K atoms (one at the end of an odd K).  The whole warp walks
        // the loop; one elected lane issues the copies.
        const bool wts = warp == 0;
        const int depth = wts ? kNP : kNB;
        uint64_t *full = wts ? p_full : b_full, *empty = wts ? p_empty : b_empty;
        int kp = 0, sp = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Unit U = unit_of<Cfg<MODE>::TAB>(a, u, nR, tab);
            for (int kt0 = 0; kt0 < U.kt_n; kt0 += kAt) {
                const int nat = min(kAt, U.kt_n - kt0);
                if (kp >= depth) {
                    ok = __all_sync(0xffffffffu, bwait(&empty[sp], ph ^ 1u, a.err, abort));
                    if (!ok)
                        break;
                }
                if (elect_one()) {
                    if (wts) {
                        mbar_arrive_expect_tx(&full[sp], nat * NMAT * kPacked);
                        uint8_t *pk = pring + sp * kPStage;
                        for (int at = 0; at < nat; ++at)
                            for (int m = 0; m < NMAT; ++m) {
                                const CUtensorMap *map = U.shared ? (m ? &a.swb : &a.swa) : (m ? &a.wb : &a.wa);
                                tma_4d(pk + (at * NMAT + m) * kPacked, map, 0, U.row0, kt0 + at, U.shared ? 0 : U.r,
                                       &full[sp]);
                            }
                    } else {
                        mbar_arrive_expect_tx(&full[sp], nat * kBTile);
                        for (int at = 0; at < nat; ++at)
                            tma_2d(bring + sp * kBStage + at * kBTile, U.shared ? &a.xs : &a.xr, 64 * (kt0 + at),
                                   U.slot0, &full[sp]);
                    }
                }
                __syncwarp();
                ++kp;
                if (++sp == depth) {
                    sp = 0;
                    ph ^= 1u;
                }
            }
        }
        // leave no copy in flight (the phases complete with the copies)
        if (elect_one()) {
            const unsigned long long t0 = global_ns();
            for (int k = (kp > depth ? kp - depth : 0); k < kp; ++k)
                while (!mbar_try_wait(&full[k % depth], (k / depth) & 1))
                    if (global_ns() - t0 > kWaitLimitNs)
                        break;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA
        // The whole warp walks the loop (its control and the descriptors stay
        // warp-uniform); one elected lane issues the MMAs and commits.  A (the
        // FP16 weights) comes from TMEM, B (the activations) from shared memory.
        int sa = 0, sb = 0, ai = 0;
        uint32_t pha = 0, phb = 0;
        bool ok = true;
        const uint32_t bring_s = smem_u32(bring);
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++ai) {
            const Unit U = unit_of<Cfg<MODE>::TAB>(a, u, nR, tab);
            const int b = NACC == 1 ? 0 : (ai & 1);
            if (ai >= NACC) {
                ok = __all_sync(0xffffffffu, bwait(&acc_empty[b], ((ai / NACC) - 1) & 1, a.err, abort));
                if (!ok)
                    break;
            }
            tc_fence_after();
            const uint32_t idesc = idesc_f16(max(16, (U.n + 15) & ~15));
            const uint32_t d0 = tmem + (uint32_t)b * kAccCols;
            for (int kt0 = 0; kt0 < U.kt_n; kt0 += kAt) {
                const int nat = min(kAt, U.kt_n - kt0);
                ok = __all_sync(0xffffffffu, bwait(&a_full[sa], pha, a.err, abort) &&
                                                 bwait(&b_full[sb], phb, a.err, abort));
                if (!ok)
                    break;
                tc_fence_after();
                if (elect_one()) {
                    // +2 per 16-element K step in the B descriptor (32 bytes), +8 TMEM columns in A
                    const uint64_t bd0 = sw128_desc(bring_s + (uint32_t)(sb * kBStage));
                    const uint32_t at0 = tmem + kACols + (uint32_t)sa * kSlotCols;
                    for (int at = 0; at < nat; ++at) {
                        const uint64_t bd = bd0 + (uint64_t)(at * (kBTile >> 4));
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint32_t acc = (kt0 | at | ks) ? 1u : 0u;
#pragma unroll
                            for (int m = 0; m < NMAT; ++m)
                                umma_ts(d0 + m * kNT, at0 + (at * NMAT + m) * 32 + 8 * ks, bd + 2 * ks, idesc, acc);
                        }
                    }
                    umma_commit(&a_empty[sa]);
                    umma_commit(&b_empty[sb]);
                }
                __syncwarp();
                if (++sa == kNA) {
                    sa = 0;
                    pha ^= 1u;
                }
                if (++sb == kNB) {
                    sb = 0;
                    phb ^= 1u;
                }
            }
            if (ok && elect_one())
                umma_commit(&acc_full[b]);
            __syncwarp();
        }
        // every MMA this warp issued has completed before TMEM is freed
        if (elect_one()) {
            umma_commit(mma_done);
            mbar_wait(mma_done, 0, a.err);
        }
        __syncwarp();
    } else if ((kDqMask >> warp) & 1u) {
        // ------------------------------------------------------ dequantize
        // Thread = (weight row r = its TMEM lane, part).  Gate/up: part =
        // matrix, all eight words of the row's atom; down: part = half of the
        // row's eight words.  The FP16 weights of an atom go to the slot with
        // one tcgen05.st per thread.
        const int q = warp & 3, part = (warp - 8) >> 2, r = 32 * q + lane;
        const int m = MODE == 0 ? part : 0;
        const int w0 = MODE == 0 ? 0 : 4 * part;
        constexpr int nw = MODE == 0 ? 8 : 4;  // packed words of this thread per atom
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16) + kACols + (uint32_t)(m * 32 + 4 * w0);
        int sp = 0, sa = 0, kf = 0;
        uint32_t php = 0, pha = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Unit U = unit_of<Cfg<MODE>::TAB>(a, u, nR, tab);
            const int rows = U.shared ? a.rows_s : a.rows;
            const int row = U.row0 + r;
            const bool valid = row < rows;
            const int G = U.shared ? a.GK_s : a.GK;  // groups per weight row
            const int j = MODE == 0 ? m : 2;         // gate, up, or down
            const uint16_t *sv, *bv;
            if (U.shared) {
                sv = a.ss[j] + (size_t)row * G;
                bv = a.sb[j] + (size_t)row * G;
            } else {
                const uint8_t *rec = a.blob + (uint64_t)U.r * a.stride;
                sv = reinterpret_cast<const uint16_t *>(rec + a.off_s[j]) + (size_t)row * G;
                bv = reinterpret_cast<const uint16_t *>(rec + a.off_b[j]) + (size_t)row * G;
            }
            // scale and bias of the row's groups in blocks of 8 atoms (one
            // 16-byte load each when the row pitch allows), one block ahead
            // in registers (the loads are L2/DRAM latency; a block of stages
            // takes well over that)
            constexpr int kSB = 8, kSt = kSB / kAt;  // atoms, stages per block
            const bool vec = (G % kSB) == 0;
            auto load_blk = [&](int k0, uint4 &s4, uint4 &b4) {
                s4 = b4 = make_uint4(0, 0, 0, 0);
                if (!valid || k0 >= U.kt_n)
                    return;
                if (vec) {
                    s4 = __ldg(reinterpret_cast<const uint4 *>(sv + k0));
                    b4 = __ldg(reinterpret_cast<const uint4 *>(bv + k0));
                } else {
                    uint32_t sw[kSB], bw[kSB];
#pragma unroll
                    for (int i = 0; i < kSB; ++i) {
                        sw[i] = k0 + i < U.kt_n ? __ldg(sv + k0 + i) : 0u;
                        bw[i] = k0 + i < U.kt_n ? __ldg(bv + k0 + i) : 0u;
                    }
                    s4 = make_uint4(sw[0] | sw[1] << 16, sw[2] | sw[3] << 16, sw[4] | sw[5] << 16, sw[6] | sw[7] << 16);
                    b4 = make_uint4(bw[0] | bw[1] << 16, bw[2] | bw[3] << 16, bw[4] | bw[5] << 16, bw[6] | bw[7] << 16);
                }
            };
            auto half_of = [](const uint4 &v, int h) -> uint16_t {
                const uint32_t w = h < 2 ? v.x : h < 4 ? v.y : h < 6 ? v.z : v.w;
                return (uint16_t)((h & 1) ? (w >> 16) : (w & 0xFFFFu));
            };
            uint4 s_c, b_c, s_n, b_n;
            load_blk(0, s_c, b_c);
            load_blk(kSB, s_n, b_n);
            for (int kb = 0; kb < U.kt_n && ok; kb += kSB) {
#pragma unroll
            for (int jj = 0; jj < kSt; ++jj) {
                const int kt0 = kb + jj * kAt;
                if (kt0 >= U.kt_n)
                    break;
                const int nat = min(kAt, U.kt_n - kt0);
                __half2 s2[kAt], b2[kAt];
#pragma unroll
                for (int at = 0; at < kAt; ++at) {
                    s2[at] = __float2half2_rn(bf2f(half_of(s_c, jj * kAt + at)));
                    b2[at] = __float2half2_rn(bf2f(half_of(b_c, jj * kAt + at)));
                }
                ok = bwait(&p_full[sp], php, a.err, abort) && (kf < kNA || bwait(&a_empty[sa], pha ^ 1u, a.err, abort));
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dequantize the stage's atoms into registers, release the packed stage
                uint32_t o[kAt][4 * nw];
#pragma unroll
                for (int at = 0; at < kAt; ++at) {
                    if (at < nat) {
                        const uint4 *src =
                            reinterpret_cast<const uint4 *>(pring + sp * kPStage + (at * NMAT + m) * kPacked + r * 32);
                        if (MODE == 0) {
                            const uint4 q0 = src[0], q1 = src[1];
                            const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                            for (int w = 0; w < nw; ++w)
                                dequant_word(wv[w], s2[at], b2[at], o[at] + 4 * w);
                        } else {
                            const uint4 qq = src[part];
                            const uint32_t wv[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
                            for (int w = 0; w < nw; ++w)
                                dequant_word(wv[w], s2[at], b2[at], o[at] + 4 * w);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_empty[sp]);
                // store the slot and publish it at once (publishing it one
                // stage later, behind the next stage's arithmetic, kept the
                // MMA waiting: 8% of the step at T = 4096)
#pragma unroll
                for (int at = 0; at < kAt; ++at)
                    if (at < nat)
                        tmem_st<nw>(tl + (uint32_t)sa * kSlotCols + (uint32_t)(at * NMAT * 32), o[at]);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&a_full[sa]);
                ++kf;
                if (++sa == kNA) {
                    sa = 0;
                    pha ^= 1u;
                }
                if (++sp == kNP) {
                    sp = 0;
                    php ^= 1u;
                }
            }
            s_c = s_n;
            b_c = b_n;
            load_blk(kb + 2 * kSB, s_n, b_n);
            }
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        int ai = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++ai) {
            const Unit U = unit_of<Cfg<MODE>::TAB>(a, u, nR, tab);
            const int b = NACC == 1 ? 0 : (ai & 1);
            // gate/up: the token scales of the unit's columns (lane j holds
            // columns j, j + 32, ...), fetched while the unit's MMAs run
            float my_sc[kNT / 32];
            if (MODE == 0) {
#pragma unroll
                for (int i = 0; i < kNT / 32; ++i) {
                    const int col = 32 * i + lane;
                    my_sc[i] = 0.f;
                    if (col < U.n) {
                        const int p = U.slot0 + col;
                        my_sc[i] = __ldg(a.xsc + (U.shared ? p : __ldg(a.perm + p) / a.K));
                    }
                }
            }
            if (!__all_sync(0xffffffffu, bwait(&acc_full[b], (ai / NACC) & 1, a.err, abort)))
                break;
            tc_fence_after();
            const int rows = U.shared ? a.rows_s : a.rows;
            const int row = U.row0 + 32 * q + lane;
            const bool valid = row < rows;
            const uint32_t d0 = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)b * kAccCols;
            for (int c0 = 0; c0 < U.n; c0 += 32) {
                uint32_t g[32];
                tmem_ld32(d0 + c0, g);
                if (MODE == 0) {
                    uint32_t v[32];
                    tmem_ld32(d0 + kNT + c0, v);
                    float sc_c = my_sc[0];
#pragma unroll
                    for (int i = 1; i < kNT / 32; ++i)
                        if (c0 == 32 * i)
                            sc_c = my_sc[i];
                    __half *H = static_cast<__half *>(U.shared ? a.Hs : a.H);
                    const int ld = U.shared ? a.S : a.I;
                    __half *hp = H + (size_t)(U.slot0 + c0) * ld + opos(row);
                    // two columns at a time in packed arithmetic; h rounded to
                    // FP16 with saturation at the largest finite value
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float s0 = __shfl_sync(0xffffffffu, sc_c, j), s1 = __shfl_sync(0xffffffffu, sc_c, j + 1);
                        const uint64_t sc2 = pair_f32(s0, s1);
                        const uint64_t gg = mul_f32x2(pair_f32(__uint_as_float(g[j]), __uint_as_float(g[j + 1])), sc2);
                        const uint64_t uu = mul_f32x2(pair_f32(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), sc2);
                        float h0, h1;
                        unpair_f32(mul_f32x2(gelu_fast_x2(gg), uu), h0, h1);
                        uint32_t hh;
                        asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(hh) : "f"(h1), "f"(h0));
                        if (valid && c0 + j < U.n)
                            *reinterpret_cast<uint16_t *>(hp + (size_t)j * ld) = (uint16_t)(hh & 0xFFFFu);
                        if (valid && c0 + j + 1 < U.n)
                            *reinterpret_cast<uint16_t *>(hp + (size_t)(j + 1) * ld) = (uint16_t)(hh >> 16);
                    }
                } else {
                    float *Y = U.shared ? a.Ys : a.Y;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int col = c0 + j;
                        if (col < U.n && valid)
                            Y[(size_t)(U.slot0 + col) * a.D + row] = __uint_as_float(g[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// -------------------------------------------------------------- small kernels

// inv[perm[i]] = i; block 0 also writes the per-expert token-tile offsets.
__global__ void pf_index(const int32_t *perm, int n, const int32_t *counts, int E, int32_t *inv, int32_t *tt_off)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n)
        inv[__ldg(perm + i)] = i;
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        const int lane = threadIdx.x, per = (E + 31) / 32, e0 = lane * per, e1 = min(E, e0 + per);
        int sum = 0;
        for (int e = e0; e < e1; ++e)
            sum += (__ldg(counts + e) + kNT - 1) / kNT;
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        int run = incl - sum;
        for (int e = e0; e < e1; ++e) {
            tt_off[e] = run;
            run += (__ldg(counts + e) + kNT - 1) / kNT;
        }
        if (lane == 31)
            tt_off[E] = incl;
    }
}

// One CTA per token: optional rmsnorm (canonical order, rounded to BF16), the
// token's power-of-two scale, its FP16 row in operand order, and its per-group
// sums in the fixed add order (the router's X: of (x_i * rsc_i) * rcoef when
// the router input is scaled).  With a gate vector, gv[t] = sigmoid(gvec . x)
// (per group an fma chain, groups in order).
__global__ void __launch_bounds__(256) pf_norm(const uint16_t *x, int D, int pre_norm, float eps, __half *X16,
                                               float *xsc, float *XG, const uint16_t *rsc, float rcoef,
                                               const uint16_t *gvec, float *gv)
{
    extern __shared__ float gs[];  // D floats, then 64 + D/64 scratch
    float *xv = gs, *scr = gs + D;
    const int t = blockIdx.x, tid = threadIdx.x, G = D / 64;
    const uint16_t *xr = x + (size_t)t * D;
    for (int i = tid; i < D; i += 256)
        xv[i] = bf2f(__ldg(xr + i));
    __syncthreads();
    if (pre_norm) {
        for (int g = tid; g < G; g += 256) {
            float q = 0.f;
            for (int k = 0; k < 64; ++k)
                q = fmaf(xv[64 * g + k], xv[64 * g + k], q);
            scr[64 + g] = q;
        }
        __syncthreads();
        if (tid == 0) {
            float ss = 0.f;
            for (int g = 0; g < G; ++g)
                ss = ss + scr[64 + g];
            scr[0] = 1.0f / sqrtf(ss / (float)D + eps);
        }
        __syncthreads();
        const float r = scr[0];
        for (int i = tid; i < D; i += 256)
            xv[i] = bf2f(f2bf(xv[i] * r));
        __syncthreads();
    }
    for (int g = tid; g < G; g += 256) {
        float X = 0.f;
        if (rsc) {
            for (int k = 0; k < 64; ++k)
                X = X + __fmul_rn(__fmul_rn(xv[64 * g + k], bf2f(__ldg(rsc + 64 * g + k))), rcoef);
        } else {
            for (int k = 0; k < 64; ++k)
                X = X + xv[64 * g + k];
        }
        XG[(size_t)t * G + g] = X;
        if (gvec) {
            float q = 0.f;
            for (int k = 0; k < 64; ++k)
                q = fmaf(bf2f(__ldg(gvec + 64 * g + k)), xv[64 * g + k], q);
            scr[64 + g] = q;
        }
    }
    if (gvec) {
        __syncthreads();
        if (tid == 0) {
            float z = 0.f;
            for (int g = 0; g < G; ++g)
                z = z + scr[64 + g];
            gv[t] = 1.0f / (1.0f + expf(-z));
        }
    }
    float mx = 0.f;
    for (int i = tid; i < D; i += 256)
        mx = fmaxf(mx, fabsf(xv[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __syncthreads();
    if ((tid & 31) == 0)
        scr[1 + (tid >> 5)] = mx;
    __syncthreads();
    if (tid == 0) {
        float m = 0.f;
        for (int w = 0; w < 8; ++w)
            m = fmaxf(m, scr[1 + w]);
        // 2^k with m * 2^k in [2^14, 2^15)
        const int E2 = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
        int k = m > 0.f ? 14 - E2 : 0;
        k = k > 100 ? 100 : (k < -100 ? -100 : k);
        scr[0] = ldexpf(1.0f, k);
        xsc[t] = ldexpf(1.0f, -k);
    }
    __syncthreads();
    const float sc = scr[0];
    __half *row = X16 + (size_t)t * D;
    for (int i = tid; i < D; i += 256)
        row[opos(i)] = __float2half_rn(xv[i] * sc);
}

// Copies of each token's FP16 row at the positions of its K slots (expert order).
__global__ void __launch_bounds__(256) pf_scatter(const __half *X16, int D, int K, const int32_t *inv, __half *Xr)
{
    const int t = blockIdx.x, tid = threadIdx.x;
    const uint4 *src = reinterpret_cast<const uint4 *>(X16 + (size_t)t * D);
    for (int k = 0; k < K; ++k) {
        uint4 *dst = reinterpret_cast<uint4 *>(Xr + (size_t)__ldg(inv + (size_t)t * K + k) * D);
        for (int i = tid; i < D / 8; i += 256)
            dst[i] = __ldg(src + i);
    }
}

// The combined FFN output of token t at columns d..d+3: the shared branch (times
// its gate gv[t] when there is one), then the K routed outputs, k ascending.
__device__ __forceinline__ float4 combined(const float *Y, const float *Ys, const int32_t *inv,
                                           const float *topk_w, const float *gv, int t, int D, int K, int d)
{
    float4 acc = *reinterpret_cast<const float4 *>(Ys + (size_t)t * D + d);
    if (gv) {
        const float g = __ldg(gv + t);
        acc.x = g * acc.x;
        acc.y = g * acc.y;
        acc.z = g * acc.z;
        acc.w = g * acc.w;
    }
    for (int k = 0; k < K; ++k) {
        const float w = __ldg(topk_w + (size_t)t * K + k);
        const float4 y = *reinterpret_cast<const float4 *>(Y + (size_t)__ldg(inv + (size_t)t * K + k) * D + d);
        acc.x = acc.x + w * y.x;
        acc.y = acc.y + w * y.y;
        acc.z = acc.z + w * y.z;
        acc.w = acc.w + w * y.w;
    }
    return acc;
}

// out[t] at columns d..d+3 = residual[t] + lambda * v, rounded to BF16.
__device__ __forceinline__ void store_out(const uint16_t *residual, uint16_t *out, int t, int D, int d, float lam,
                                          const float (&v)[4])
{
    float r[4] = {0.f, 0.f, 0.f, 0.f};
    if (residual) {
        const uint2 rv = *reinterpret_cast<const uint2 *>(residual + (size_t)t * D + d);
        r[0] = __uint_as_float(rv.x << 16);
        r[1] = __uint_as_float(rv.x & 0xFFFF0000u);
        r[2] = __uint_as_float(rv.y << 16);
        r[3] = __uint_as_float(rv.y & 0xFFFF0000u);
    }
    const float o[4] = {r[0] + lam * v[0], r[1] + lam * v[1], r[2] + lam * v[2], r[3] + lam * v[3]};
    uint2 ov;
    ov.x = (uint32_t)f2bf(o[0]) | ((uint32_t)f2bf(o[1]) << 16);
    ov.y = (uint32_t)f2bf(o[2]) | ((uint32_t)f2bf(o[3]) << 16);
    *reinterpret_cast<uint2 *>(out + (size_t)t * D + d) = ov;
}

// With a post-FFN norm weight: one CTA per token holds the combined output in
// shared memory, takes its RMS factor (per group of 64 an fma chain of squares,
// groups in order) and writes residual + lambda * (y * r) * weight.
__global__ void __launch_bounds__(256) pf_combine_norm(const float *Y, const float *Ys, const int32_t *inv,
                                                       const float *topk_w, const float *gv, int T, int D, int K,
                                                       float lam, const uint16_t *pnw, float peps,
                                                       const uint16_t *residual, uint16_t *out)
{
    extern __shared__ float ys[];  // D floats, then D/64 group sums and the factor
    const int t = blockIdx.x, tid = threadIdx.x, G = D / 64;
    float *q = ys + D;
    for (int d = 4 * tid; d < D; d += 1024)
        *reinterpret_cast<float4 *>(ys + d) = combined(Y, Ys, inv, topk_w, gv, t, D, K, d);
    __syncthreads();
    for (int g = tid; g < G; g += 256) {
        float a = 0.f;
        for (int k = 0; k < 64; ++k)
            a = fmaf(ys[64 * g + k], ys[64 * g + k], a);
        q[g] = a;
    }
    __syncthreads();
    if (tid == 0) {
        float ss = 0.f;
        for (int g = 0; g < G; ++g)
            ss = ss + q[g];
        q[G] = 1.0f / sqrtf(ss / (float)D + peps);
    }
    __syncthreads();
    const float r = q[G];
    for (int d = 4 * tid; d < D; d += 1024) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] = __fmul_rn(__fmul_rn(ys[d + j], r), bf2f(__ldg(pnw + d + j)));
        store_out(residual, out, t, D, d, lam, v);
    }
}

// out[t] = residual[t] + lambda * (shared[t] + sum_k w[t,k] * y[slot(t,k)]), k ascending.
__global__ void __launch_bounds__(256) pf_combine(const float *Y, const float *Ys, const int32_t *inv,
                                                  const float *topk_w, const float *gv, int T, int D, int K,
                                                  float lam, const uint16_t *residual, uint16_t *out)
{
    const int t = blockIdx.y, d = 4 * (blockIdx.x * 256 + threadIdx.x);
    if (t >= T || d >= D)
        return;
    const float4 acc = combined(Y, Ys, inv, topk_w, gv, t, D, K, d);
    const float v[4] = {acc.x, acc.y, acc.z, acc.w};
    store_out(residual, out, t, D, d, lam, v);
}

// ------------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// FP16 rows [rows][cols] as a 2-D tensor, box (64 columns, 128 rows), 128-byte swizzle.
cudaError_t encode_rows(CUtensorMap *m, const void *base, int rows, int cols)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kNT};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Packed 4-bit weights as (8 words, rows, groups, experts), box (8, 128, 1, 1).
cudaError_t encode_packed(CUtensorMap *m, const void *base, int rows, int cols, int experts, uint64_t record_stride)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    const int G = cols / 64;
    const cuuint64_t pitch = (cuuint64_t)cols / 2;
    cuuint64_t dims[4] = {8, (cuuint64_t)rows, (cuuint64_t)G, (cuuint64_t)experts};
    cuuint64_t strides[3] = {pitch, 32, experts > 1 ? (cuuint64_t)record_stride : pitch * rows};
    cuuint32_t box[4] = {8, (cuuint32_t)kMT, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE>
size_t gemm_smem(int E)
{
    using C = Cfg<MODE>;
    return 1024 + (size_t)C::NB * C::AT * kBTile + (size_t)C::NP * C::AT * C::NMAT * 128 * 32 + 512 +
           (C::TAB ? (size_t)(4 * E + 1) * sizeof(int) : 0);
}

template <int MODE>
cudaError_t launch_gemm(const PfArgs &a, int n_cta, cudaStream_t s)
{
    auto k = pf_gemm<MODE>;
    const size_t smem = gemm_smem<MODE>(a.E);
    cudaError_t e = smem_optin(reinterpret_cast<const void *>(k), smem);
    if (e != cudaSuccess)
        return e;
    k<<<n_cta, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

} // namespace

namespace {

struct PfBufs {
    int32_t *inv, *tt_off;
    float *xsc, *XG, *gv;
    __half *X16, *Xr, *H, *Hs;
    float *Y, *Ys;
    float *QF;
    size_t total;
};

PfBufs pf_carve(uint8_t *w, int T, int D, int I, int S, int E, int K)
{
    auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
    const size_t TK = (size_t)T * K;
    PfBufs b;
    uint8_t *p = w;
    auto take = [&](size_t bytes) {
        uint8_t *at = p;
        p += up(bytes);
        return at;
    };
    b.inv = reinterpret_cast<int32_t *>(take(TK * 4));
    b.tt_off = reinterpret_cast<int32_t *>(take((size_t)(E + 1) * 4));
    b.xsc = reinterpret_cast<float *>(take((size_t)T * 4));
    b.XG = reinterpret_cast<float *>(take((size_t)T * (D / 64) * 4));
    b.gv = reinterpret_cast<float *>(take((size_t)T * 4));
    b.X16 = reinterpret_cast<__half *>(take((size_t)T * D * 2));
    b.Xr = reinterpret_cast<__half *>(take(TK * D * 2));
    b.H = reinterpret_cast<__half *>(take(TK * I * 2));
    b.Hs = reinterpret_cast<__half *>(take((size_t)T * S * 2));
    b.Y = reinterpret_cast<float *>(take(TK * D * 4));
    b.Ys = reinterpret_cast<float *>(take((size_t)T * D * 4));
    b.QF = reinterpret_cast<float *>(take(route_f32_bytes(T, D, E, K)));
    b.total = (size_t)(p - w);
    return b;
}

} // namespace

size_t pf_workspace_bytes(int T, int D, int I, int S, int E, int K)
{
    return pf_carve(nullptr, T, D, I, S, E, K).total;
}

cudaError_t launch_prefill_prepare(const PfCall &c, PfPrepared *out, cudaStream_t s)
{
    const PfBufs b = pf_carve(c.ws, c.T, c.D, c.I, c.S, c.E, c.K);
    const size_t gsm = (size_t)(c.D + 64 + c.D / 64) * 4;
    cudaError_t e = smem_optin(reinterpret_cast<const void *>(pf_norm), gsm);
    if (e != cudaSuccess)
        return e;
    pf_norm<<<c.T, 256, gsm, s>>>(static_cast<const uint16_t *>(c.x), c.D, c.pre_norm, c.eps, b.X16, b.xsc, b.XG,
                                  c.ext.router_scale, c.ext.rcoef, c.ext.shared_gate, b.gv);
    out->X16 = b.X16;
    out->xsc = b.xsc;
    out->XG = b.XG;
    out->QF = b.QF;
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PfCall &c, cudaStream_t s)
{
    const int T = c.T, D = c.D, I = c.I, S = c.S, E = c.E, K = c.K, TK = T * K;
    const PfBufs bf = pf_carve(c.ws, T, D, I, S, E, K);
    int32_t *inv = bf.inv, *tt_off = bf.tt_off;
    float *xsc = bf.xsc, *Y = bf.Y, *Ys = bf.Ys;
    __half *X16 = bf.X16, *Xr = bf.Xr, *H = bf.H, *Hs = bf.Hs;

    cudaError_t e;
    pf_index<<<(TK + 255) / 256, 256, 0, s>>>(c.perm, TK, c.counts, E, inv, tt_off);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    pf_scatter<<<T, 256, 0, s>>>(X16, D, K, inv, Xr);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;

    PfArgs a{};
    a.T = T;
    a.D = D;
    a.I = I;
    a.S = S;
    a.E = E;
    a.K = K;
    a.tt_off = tt_off;
    a.counts = c.counts;
    a.offsets = c.offsets;
    a.perm = c.perm;
    a.xsc = xsc;
    a.blob = c.blob;
    a.stride = c.stride;
    a.slot = c.ext.slot;
    a.n_slots = c.ext.slot ? c.ext.n_slots : E;
    for (int j = 0; j < 3; ++j) {
        a.off_s[j] = c.off_s[j];
        a.off_b[j] = c.off_b[j];
        a.ss[j] = c.ss[j];
        a.sb[j] = c.sb[j];
    }
    a.H = H;
    a.Hs = Hs;
    a.Y = Y;
    a.Ys = Ys;
    a.err = c.err;
    // gate/up: rows I (routed) / S (shared), K = D
    a.mode = 0;
    a.FT = (I + kMT - 1) / kMT;
    a.FTs = (S + kMT - 1) / kMT;
    a.KT = D / 64;
    a.KTs = D / 64;
    a.GK = D / 64;
    a.GK_s = D / 64;
    a.rows = I;
    a.rows_s = S;
    if ((e = encode_packed(&a.wa, c.blob + c.off_w[0], I, D, a.n_slots, c.stride)) != cudaSuccess ||
        (e = encode_packed(&a.wb, c.blob + c.off_w[1], I, D, a.n_slots, c.stride)) != cudaSuccess ||
        (e = encode_packed(&a.swa, c.sw[0], S, D, 1, 0)) != cudaSuccess ||
        (e = encode_packed(&a.swb, c.sw[1], S, D, 1, 0)) != cudaSuccess ||
        (e = encode_rows(&a.xr, Xr, TK, D)) != cudaSuccess || (e = encode_rows(&a.xs, X16, T, D)) != cudaSuccess)
        return e;
    prof_begin(kStageGateUp, s);
    e = launch_gemm<0>(a, c.n_cta, s);
    prof_end(kStageGateUp, s);
    if (e != cudaSuccess)
        return e;
    // down: rows D, K = I (routed) / S (shared)
    a.mode = 1;
    a.FT = (D + kMT - 1) / kMT;
    a.FTs = a.FT;
    a.KT = I / 64;
    a.KTs = S / 64;
    a.GK = I / 64;
    a.GK_s = S / 64;
    a.rows = D;
    a.rows_s = D;
    if ((e = encode_packed(&a.wa, c.blob + c.off_w[2], D, I, a.n_slots, c.stride)) != cudaSuccess ||
        (e = encode_packed(&a.swa, c.sw[2], D, S, 1, 0)) != cudaSuccess ||
        (e = encode_rows(&a.xr, H, TK, I)) != cudaSuccess || (e = encode_rows(&a.xs, Hs, T, S)) != cudaSuccess)
        return e;
    prof_begin(kStageDown, s);
    e = launch_gemm<1>(a, c.n_cta, s);
    const float *gv = c.ext.shared_gate ? bf.gv : nullptr;
    if (e == cudaSuccess && c.ext.post_norm) {
        const size_t nsm = ((size_t)D + D / 64 + 1) * 4;
        if ((e = smem_optin(reinterpret_cast<const void *>(pf_combine_norm), nsm)) == cudaSuccess) {
            pf_combine_norm<<<T, 256, nsm, s>>>(Y, Ys, inv, c.topk_w, gv, T, D, K, c.lam, c.ext.post_norm,
                                                c.ext.post_eps, static_cast<const uint16_t *>(c.residual),
                                                static_cast<uint16_t *>(c.out));
            e = cudaGetLastError();
        }
    } else if (e == cudaSuccess) {
        pf_combine<<<dim3((D / 4 + 255) / 256, T), 256, 0, s>>>(Y, Ys, inv, c.topk_w, gv, T, D, K, c.lam,
                                                               static_cast<const uint16_t *>(c.residual),
                                                               static_cast<uint16_t *>(c.out));
        e = cudaGetLastError();
    }
    prof_end(kStageDown, s);
    return e;
}

} // namespace mx

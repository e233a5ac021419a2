// mx_common.cuh -- device helpers shared by the library's kernels.
//
// Operand convention of the warp-level quantized GEMM (decode path):
//   A = the quantized integers q of 16 weight rows, as exact BF16 integers
//       (0..15), built in registers from the packed nibbles;
//   B = activations (or the gated hidden vector) as BF16, optionally split into
//       2-3 BF16 parts whose sum carries fp32 precision;
//   the per-group affine terms are applied outside the MMA in fp32:
//       y_r += s[r,g] * (sum_{c in g} q[r,c] x_c) + b[r,g] * (sum_{c in g} x_c)
//   which is exactly the dequantized dot product sum_c (s q + b) x_c
//   ("Mference System design" page, "Why the runtime has this shape": BF16
//   scale and bias per group of 64; "Metal execution": kernels consume the
//   packed values, BF16 scales and BF16 biases directly).
//
// Column order inside each 8-column block of a B operand row: [0,4,1,5,2,6,3,7].
// With it, the two BF16 pairs a lane feeds one m16n8k16 k-step come out of a
// packed word with one shift-and-mask each, and its B values are one 64-bit
// load.  Producers of B rows (x preparation, the gated hidden vector) write in
// this order; weights stay in the checkpoint's order.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mx {

constexpr int kGroup = 64;

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// Position of column c in the operand order [0,4,1,5,2,6,3,7] of its 8-block.
__device__ __forceinline__ int perm8(int c)
{
    const int a = c & 7;
    return (c & ~7) | (a < 4 ? 2 * a : 2 * (a - 4) + 1);
}

// Streaming load of packed weights: read once, keep out of L1.
__device__ __forceinline__ uint2 ld_stream_u2(const void *p)
{
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ldg_u4(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }

// Nibbles j and j+4 of w as a BF16x2 pair of exact integers (low half = nibble j).
// 0x4300 is BF16 128.0, whose 7 mantissa bits count units; OR-ing a nibble into
// them gives 128+q exactly, and one fma (x*1 - 128) leaves q exactly.
template <int J>
__device__ __forceinline__ uint32_t nib_pair(uint32_t w)
{
    const uint32_t v = ((w >> (4 * J)) & 0x000F000Fu) | 0x43004300u;
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(0x3F803F80u), "r"(0xC300C300u));
    return r;
}

// D += A(16x16, bf16, row) * B(16x8, bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// GELU, tanh form (the reading taken for the pages' "GeGLU").
__device__ __forceinline__ float gelu_tanh(float z)
{
    const float k0 = 0.7978845608028654f;
    const float k1 = 0.044715f;
    const float inner = k0 * (z + k1 * z * z * z);
    return 0.5f * z * (1.0f + tanhf(inner));
}

__device__ __forceinline__ float exp2f_fast(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_fast(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// The same GELU through the identity 0.5 (1 + tanh(u)) = 1 / (1 + e^(-2u)):
// z / (1 + e^(-2u)) with the fast exponential and division intrinsics (a few
// ulp; the limits z -> -inf and +inf give -0 and z).  For the bulk epilogue of
// the grouped GEMMs, where tanhf dominated the cost.
__device__ __forceinline__ float gelu_fast(float z)
{
    const float k0 = 0.7978845608028654f;
    const float k1 = 0.044715f;
    const float inner = k0 * (z + k1 * z * z * z);
    return __fdividef(z, 1.0f + __expf(-2.0f * inner));
}

// Two fp32 values as one 64-bit register pair, and back; packed two-lane
// arithmetic on such pairs (each lane an IEEE operation, round to nearest).
__device__ __forceinline__ uint64_t pair_f32(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpair_f32(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// d = a * b + d
__device__ __forceinline__ void fma_f32x2(uint64_t &d, uint64_t a, uint64_t b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// GELU (tanh form) of two values through z / (1 + e^(-2u)), u = k0 z (1 +
// k1 z^2): packed arithmetic, the fast base-2 exponential and reciprocal
// (the same approximations as gelu_fast).
__device__ __forceinline__ uint64_t gelu_fast_x2(uint64_t z)
{
    const float k0 = 0.7978845608028654f, k1 = 0.044715f;
    const float c = -2.0f * k0 * 1.4426950408889634f;  // e^(-2 k0 w) = 2^(c w)
    const uint64_t z2 = mul_f32x2(z, z);
    uint64_t t = pair_f32(1.0f, 1.0f);
    fma_f32x2(t, z2, pair_f32(k1, k1));        // 1 + k1 z^2
    const uint64_t a = mul_f32x2(mul_f32x2(z, t), pair_f32(c, c));
    float a0, a1;
    unpair_f32(a, a0, a1);
    const uint64_t d = add_f32x2(pair_f32(exp2f_fast(a0), exp2f_fast(a1)), pair_f32(1.0f, 1.0f));
    float d0, d1;
    unpair_f32(d, d0, d1);
    return mul_f32x2(z, pair_f32(rcp_fast(d0), rcp_fast(d1)));
}

// One packed router byte as an exact float: 2^23 + q built in the mantissa, minus 2^23.
template <int J>
__device__ __forceinline__ float byte_f(uint32_t w)
{
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | J)) - 8388608.0f;
}

// ------------------------------------------------------------------ async copies
// Bulk global->shared copies (the untiled TMA path) completing on an mbarrier.
// Every wait is bounded by the global timer; a wait that gives up records an
// error code in the caller's error word and returns false.

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
constexpr unsigned kErrTimeout = 1u;  // a bounded wait gave up
constexpr unsigned kErrRange = 2u;    // a value outside a fixed-point range (left out)
constexpr unsigned kErrAbsent = 4u;   // a selected expert has no record in the blob

// Record of expert e in the blob: through the resident-set table when there
// is one, else e.  An expert with no record sets kErrAbsent in *err and reads
// record 0 (the call's outputs are then not the block's; the error word says so).
__device__ __forceinline__ int expert_record(const int16_t *slot, int n_slots, int e, unsigned *err)
{
    if (!slot)
        return e;
    const int r = __ldg(slot + e);
    if (r >= 0 && r < n_slots)
        return r;
    atomicOr(err, kErrAbsent);
    return 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// n arrivals at once.
__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t n)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of *bar to complete; false (and *err |= timeout) if
// it has not after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *err)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            if (err)
                atomicOr(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// dst (shared) and src (global) 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// 16-byte asynchronous global->shared copies (L2 only), grouped per thread.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// cp.async.wait_group with a run-time count (0..3).
__device__ __forceinline__ void cp_async_wait_n(int n)
{
    switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    default: cp_async_wait<3>(); break;
    }
}

// Programmatic dependent launch: wait for the preceding kernel's memory, and
// allow the next kernel in the stream to begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier over `count` threads (multiple of 32), id 1..15.
__device__ __forceinline__ void named_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Shared-memory row stride (bytes) for a packed row of `row_bytes` (a multiple
// of 32): padded so that 8 consecutive rows read by the 8 lane quads of a warp
// with 8-byte loads fall in distinct banks (stride/4 = 8 mod 32).
__host__ __device__ constexpr int padded_row_bytes(int row_bytes)
{
    return row_bytes + 4 * ((8 - (row_bytes / 4) % 32 + 32) % 32);
}

} // namespace mx

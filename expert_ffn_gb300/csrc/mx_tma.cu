// mx_tma.cu -- TMA tensor maps of the expert weights (host side).
//
// Each packed 4-bit matrix W [rows][cols/8 words] is described to the tensor
// memory accelerator as a 4-D tensor of 32-bit words
//     (8 words of one group, rows, groups, experts)
// with strides (4 B, row pitch, 32 B, record stride).  The stride order is not
// monotonic on purpose: a box of (8, r rows, all groups, 1 expert) lands in
// shared memory group-major, [group][row][8 words], so the 8 rows a warp's
// lane quads read for one group are 256 contiguous bytes -- no bank conflicts
// -- and one copy moves a whole block of rows.  The routed experts of a layer
// share one map per sub-tensor (gate, up, down) through the record stride of
// the fixed-stride blob ("Mference System design", "The .gturbo directory":
// fixed-stride expert records, one offset per sub-tensor); the shared expert
// has its own maps.
#include "mx_internal.h"

#include <cstring>
#include <mutex>

namespace mx {

namespace {

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

// Map of `experts` matrices [rows][cols] (4-bit) at base + e*record_stride,
// box = (8 words, box_rows rows, box_groups groups (0: all), 1 expert).
cudaError_t encode_qmat(CUtensorMap *m, const void *base, int rows, int cols, int experts, uint64_t record_stride,
                        int box_rows, int box_groups = 0)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    const int G = cols / 64;
    const cuuint64_t pitch = (cuuint64_t)cols / 2;
    cuuint64_t dims[4] = {8, (cuuint64_t)rows, (cuuint64_t)G, (cuuint64_t)experts};
    cuuint64_t strides[3] = {pitch, 32, experts > 1 ? (cuuint64_t)record_stride : pitch * rows};
    cuuint32_t box[4] = {8, (cuuint32_t)box_rows, (cuuint32_t)(box_groups > 0 ? box_groups : G), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct Key {
    const void *blob, *sw0, *sw1, *sw2;
    uint64_t stride, off[3];
    int D, I, S, E, records;
    bool operator==(const Key &o) const { return std::memcmp(this, &o, sizeof(Key)) == 0; }
};

constexpr int kCache = 128;
std::mutex g_mu;
Key g_keys[kCache];
FfnMaps g_maps[kCache];
int g_n = 0, g_next = 0;

} // namespace

cudaError_t smem_optin(const void *k, size_t bytes)
{
    if (bytes <= 48 * 1024)
        return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    struct Entry {
        int dev;
        const void *k;
        size_t bytes;
    };
    static std::mutex mu;
    static Entry done[256];
    static int n = 0;
    std::lock_guard<std::mutex> g(mu);
    int i = 0;
    while (i < n && !(done[i].dev == dev && done[i].k == k))
        ++i;
    if (i < n && done[i].bytes >= bytes)
        return cudaSuccess;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes)) != cudaSuccess)
        return e;
    if (i == n && n < 256)
        done[n++] = Entry{dev, k, 0};
    if (i < n)
        done[i].bytes = bytes;
    return cudaSuccess;
}

cudaError_t get_ffn_maps(const FfnArgs &a, FfnMaps *out)
{
    Key k;
    std::memset(&k, 0, sizeof k);
    k.blob = a.blob;
    k.sw0 = a.sw[0];
    k.sw1 = a.sw[1];
    k.sw2 = a.sw[2];
    k.stride = a.stride;
    for (int j = 0; j < 3; ++j)
        k.off[j] = a.off_w[j];
    k.D = a.D;
    k.I = a.I;
    k.S = a.S;
    k.E = a.E;
    k.records = a.slot ? a.n_slots : a.E;
    {
        std::lock_guard<std::mutex> g(g_mu);
        for (int i = 0; i < g_n; ++i)
            if (g_keys[i] == k) {
                *out = g_maps[i];
                return cudaSuccess;
            }
    }
    FfnMaps m;
    cudaError_t e;
    if ((e = encode_qmat(&m.gate, a.blob + a.off_w[0], a.I, a.D, k.records, a.stride, 8)) != cudaSuccess ||
        (e = encode_qmat(&m.up, a.blob + a.off_w[1], a.I, a.D, k.records, a.stride, 8)) != cudaSuccess ||
        (e = encode_qmat(&m.down, a.blob + a.off_w[2], a.D, a.I, k.records, a.stride, 16)) != cudaSuccess ||
        (e = encode_qmat(&m.sgate, a.sw[0], a.S, a.D, 1, 0, 8)) != cudaSuccess ||
        (e = encode_qmat(&m.sup, a.sw[1], a.S, a.D, 1, 0, 8)) != cudaSuccess ||
        (e = encode_qmat(&m.sdown, a.sw[2], a.D, a.S, 1, 0, 16)) != cudaSuccess ||
        (e = encode_qmat(&m.down1, a.blob + a.off_w[2], a.D, a.I, k.records, a.stride, a.D / 16 < 256 ? a.D / 16 : 256, 1)) !=
            cudaSuccess ||
        (e = encode_qmat(&m.sdown1, a.sw[2], a.D, a.S, 1, 0, a.D / 16 < 256 ? a.D / 16 : 256, 1)) != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> g(g_mu);
    g_keys[g_next] = k;
    g_maps[g_next] = m;
    g_next = (g_next + 1) % kCache;
    if (g_n < kCache)
        ++g_n;
    *out = m;
    return cudaSuccess;
}

} // namespace mx

// mx_profile.cu -- stage profiler: CUDA event pairs around each kernel of a
// block call, recorded on the call's stream while profiling is enabled
// (mx_moe_profile_enable / mx_moe_profile_read).
#include "mx_moe.h"
#include "mx_internal.h"

#include <atomic>
#include <mutex>
#include <vector>

namespace mx {

namespace {

struct Pair {
    int stage;
    cudaEvent_t start, stop;
};

std::atomic<int> g_on{0};
std::mutex g_mu;
std::vector<Pair> g_pairs;          // recorded, not yet read
std::vector<cudaEvent_t> g_free;    // reusable events
thread_local cudaEvent_t t_open[MX_PROFILE_STAGES] = {};  // start event of the launch in flight

cudaEvent_t take_event()
{
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess)
        return nullptr;
    return e;
}

} // namespace

void prof_begin(int stage, cudaStream_t s)
{
    if (!g_on.load(std::memory_order_relaxed))
        return;
    cudaEvent_t e = take_event();
    if (e && cudaEventRecord(e, s) == cudaSuccess)
        t_open[stage] = e;
}

void prof_end(int stage, cudaStream_t s)
{
    if (!g_on.load(std::memory_order_relaxed) || !t_open[stage])
        return;
    cudaEvent_t e = take_event();
    if (!e)
        return;
    if (cudaEventRecord(e, s) == cudaSuccess) {
        std::lock_guard<std::mutex> g(g_mu);
        g_pairs.push_back({stage, t_open[stage], e});
    }
    t_open[stage] = nullptr;
}

} // namespace mx

extern "C" {

mx_status mx_moe_profile_enable(int on)
{
    mx::g_on.store(on ? 1 : 0);
    return MX_OK;
}

mx_status mx_moe_profile_read(double *ms, int *launches, int reset)
{
    using namespace mx;
    double acc[MX_PROFILE_STAGES] = {0, 0, 0};
    int cnt[MX_PROFILE_STAGES] = {0, 0, 0};
    std::vector<Pair> pairs;
    {
        std::lock_guard<std::mutex> g(g_mu);
        pairs = g_pairs;
        if (reset)
            g_pairs.clear();
    }
    mx_status st = MX_OK;
    for (const Pair &p : pairs) {
        float t = 0.f;
        if (cudaEventSynchronize(p.stop) != cudaSuccess || cudaEventElapsedTime(&t, p.start, p.stop) != cudaSuccess) {
            st = MX_ERR_CUDA;
            continue;
        }
        acc[p.stage] += t;
        cnt[p.stage] += 1;
    }
    if (reset) {
        std::lock_guard<std::mutex> g(g_mu);
        for (const Pair &p : pairs) {
            g_free.push_back(p.start);
            g_free.push_back(p.stop);
        }
    }
    for (int i = 0; i < MX_PROFILE_STAGES; ++i) {
        if (ms)
            ms[i] = acc[i];
        if (launches)
            launches[i] = cnt[i];
    }
    return st;
}

} // extern "C"

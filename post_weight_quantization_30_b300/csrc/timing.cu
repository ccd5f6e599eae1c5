// Per-kernel-class timing of the library's own launches, for measurement:
// while recording is on (gq_timing_begin), the launchers of the main kernels
// bracket each launch with a pair of CUDA events on the launch's stream; at
// gq_timing_end the pairs are synchronized and their elapsed times summed per
// class, with the launch count and the useful floating-point operations the
// launchers declared.  Off by default; when off a launcher only tests a flag.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace gq {
namespace {

struct Rec {
    cudaEvent_t a, b;
    int kind;
    double flops;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;  // events reused across recordings
size_t g_used = 0;

cudaEvent_t take_event() {
    if (g_used == g_pool.size()) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_pool.push_back(e);
    }
    return g_pool[g_used++];
}

}  // namespace

int timing_begin(int kind, cudaStream_t s) {
    if (!g_on.load(std::memory_order_relaxed)) return -1;
    std::lock_guard<std::mutex> lock(g_mu);
    Rec r{take_event(), take_event(), kind, 0.0};
    if (!r.a || !r.b || cudaEventRecord(r.a, s) != cudaSuccess) return -1;
    g_recs.push_back(r);
    return (int)g_recs.size() - 1;
}

void timing_end(int idx, cudaStream_t s, double flops) {
    if (idx < 0) return;
    std::lock_guard<std::mutex> lock(g_mu);
    if ((size_t)idx >= g_recs.size()) return;
    g_recs[idx].flops = flops;
    cudaEventRecord(g_recs[idx].b, s);
}

}  // namespace gq

using namespace gq;

extern "C" gq_status gq_timing_begin(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_recs.clear();
    g_used = 0;
    g_on.store(true);
    return GQ_OK;
}

extern "C" gq_status gq_timing_end(double *ms, double *flops, unsigned long long *count, int nkinds) {
    g_on.store(false);
    std::lock_guard<std::mutex> lock(g_mu);
    if (nkinds < 0 || (nkinds > 0 && (!ms || !flops || !count))) return GQ_EINVAL;
    for (int k = 0; k < nkinds; ++k) {
        ms[k] = 0.0;
        flops[k] = 0.0;
        count[k] = 0;
    }
    gq_status st = GQ_OK;
    for (const Rec &r : g_recs) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) {
            st = GQ_ECUDA;
            continue;
        }
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
            st = GQ_ECUDA;
            continue;
        }
        if (r.kind < nkinds) {
            ms[r.kind] += t;
            flops[r.kind] += r.flops;
            count[r.kind] += 1;
        }
    }
    g_recs.clear();
    g_used = 0;
    return st;
}

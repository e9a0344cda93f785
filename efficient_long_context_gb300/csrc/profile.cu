// profile.cu -- optional per-kernel CUDA-event timing of the library's launches.
//
// When enabled by orthros_profile_begin(), every launch site wrapped in a
// ProfScope records one CUDA event before and one after its kernel on the
// kernel's own stream. orthros_profile_end() resolves the pairs. Disabled
// (the default), a ProfScope costs one branch.
#include <cstring>
#include <string>
#include <vector>

#include "internal.cuh"

namespace orthros {
namespace {

struct Rec {
    const char *name;
    cudaEvent_t a, b;
};

bool g_on = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

ProfScope::ProfScope(const char *name, cudaStream_t s) : name_(name), stream_(s), a_(nullptr) {
    if (!g_on) return;
    a_ = take_event();
    if (a_) cudaEventRecord(static_cast<cudaEvent_t>(a_), s);
}

ProfScope::~ProfScope() {
    if (!g_on || !a_) return;
    cudaEvent_t b = take_event();
    if (!b) return;
    cudaEventRecord(b, stream_);
    g_recs.push_back({name_, static_cast<cudaEvent_t>(a_), b});
}

}  // namespace orthros

using namespace orthros;

extern "C" {

orthros_status orthros_profile_begin(void) {
    for (auto &r : g_recs) {
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_recs.clear();
    g_on = true;
    return ORTHROS_OK;
}

int orthros_profile_end(orthros_kernel_time *out, int max_entries) {
    g_on = false;
    std::vector<orthros_kernel_time> agg;
    for (auto &r : g_recs) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -1;
        size_t i = 0;
        for (; i < agg.size(); ++i)
            if (std::strncmp(agg[i].name, r.name, sizeof(agg[i].name)) == 0) break;
        if (i == agg.size()) {
            orthros_kernel_time t{};
            std::strncpy(t.name, r.name, sizeof(t.name) - 1);
            agg.push_back(t);
        }
        agg[i].launches += 1;
        agg[i].total_ms += ms;
    }
    for (size_t i = 0; i < agg.size() && (int)i < max_entries; ++i) out[i] = agg[i];
    return (int)agg.size();
}

}  // extern "C"

// Optional per-kernel CUDA-event timing of the library's launches (see gdn_timing_* in
// include/gdn.h).  Off by default; when off, the hooks cost one branch.
#include <string.h>

#include <map>
#include <string>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {
struct Rec {
    const char* name;
    cudaEvent_t a, b;
};
bool g_on = false;
std::vector<Rec> g_recs;
}  // namespace

void timing_begin(const char* name, cudaStream_t st) {
    if (!g_on) return;
    Rec r{name, nullptr, nullptr};
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return;
    cudaEventRecord(r.a, st);
    g_recs.push_back(r);
}

void timing_end(cudaStream_t st) {
    if (!g_on || g_recs.empty()) return;
    cudaEventRecord(g_recs.back().b, st);
}

}  // namespace gdn

extern "C" {

gdn_status gdn_timing_enable(int32_t enable) {
    gdn::g_on = enable != 0;
    return GDN_OK;
}

gdn_status gdn_timing_collect(gdn_kernel_time* out, int32_t max_entries, int32_t* n_entries) {
    std::map<std::string, std::pair<int, float>> agg;
    std::vector<std::string> order;
    gdn_status st = GDN_OK;
    for (auto& r : gdn::g_recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
            st = GDN_ERR_CUDA;
        if (!agg.count(r.name)) order.push_back(r.name);
        auto& e = agg[r.name];
        e.first += 1;
        e.second += ms;
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    gdn::g_recs.clear();
    int n = 0;
    for (auto& name : order) {
        if (out && n < max_entries) {
            memset(out[n].name, 0, sizeof(out[n].name));
            strncpy(out[n].name, name.c_str(), sizeof(out[n].name) - 1);
            out[n].launches = agg[name].first;
            out[n].total_ms = agg[name].second;
        }
        ++n;
    }
    if (n_entries) *n_entries = n;
    return st;
}

}  // extern "C"

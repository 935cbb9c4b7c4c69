// Per-kernel event timing for benchmarks (dust_profile_enable /
// dust_profile_read). Off by default; when on, each launch is bracketed by
// two CUDA events on the launching stream.
#include <atomic>
#include <cstdio>
#include <mutex>
#include <vector>

#include "dust.h"
#include "internal.cuh"

namespace dust {

namespace {

const char* const kStageNames[kStageCount] = {"scan_local", "scan_carry", "scan_fixup", "weight",
                                              "gemm_simt",  "reduce",     "gemm_tc",    "fused",
                                              "noise",      "jitter",     "zero",
                                              "score",      "scatter",    "forward"};
constexpr int kMaxRecords = 65536;

struct Rec {
    int stage;
    cudaEvent_t a, b;
};

std::mutex g_mu;
bool g_on = false;
std::vector<cudaEvent_t> g_pool;
std::vector<Rec> g_recs;

cudaEvent_t event_at(size_t i) {
    while (g_pool.size() <= i) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_pool.push_back(e);
    }
    return g_pool[i];
}

}  // namespace

ProfScope::ProfScope(int stage_, cudaStream_t s_) : stage(stage_), s(s_), slot(-1) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on || static_cast<int>(g_recs.size()) >= kMaxRecords) return;
    const size_t n = g_recs.size();
    cudaEvent_t a = event_at(2 * n), b = event_at(2 * n + 1);
    if (!a || !b) return;
    if (cudaEventRecord(a, s) != cudaSuccess) return;
    g_recs.push_back(Rec{stage, a, b});
    slot = static_cast<int>(n);
}

ProfScope::~ProfScope() {
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (slot < static_cast<int>(g_recs.size())) cudaEventRecord(g_recs[slot].b, s);
}

namespace {
std::atomic<int> g_inject{0};
}  // namespace

bool take_stall_injection() { return g_inject.exchange(0) != 0; }

bool stall_injection_pending() { return g_inject.load() != 0; }

bool profiling_on() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_on;
}

}  // namespace dust

extern "C" {

dust_status dust_debug_inject_timeout(int32_t on) {
    dust::g_inject.store(on ? 1 : 0);
    return DUST_OK;
}

dust_status dust_profile_enable(int32_t on) {
    std::lock_guard<std::mutex> lk(dust::g_mu);
    dust::g_on = on != 0;
    return DUST_OK;
}

int32_t dust_profile_read(dust_profile_entry* out, int32_t max_entries) {
    if (max_entries < 0 || (max_entries > 0 && !out)) return -DUST_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(dust::g_mu);
    double ms[dust::kStageCount] = {};
    int64_t cnt[dust::kStageCount] = {};
    bool fail = false;
    for (const auto& r : dust::g_recs) {
        float t = 0.0f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
            fail = true;
            continue;
        }
        ms[r.stage] += t;
        cnt[r.stage] += 1;
    }
    dust::g_recs.clear();
    if (fail) return -DUST_ERR_CUDA;
    int32_t n = 0;
    for (int st = 0; st < dust::kStageCount && n < max_entries; ++st) {
        if (!cnt[st]) continue;
        dust_profile_entry& e = out[n++];
        std::snprintf(e.name, sizeof(e.name), "%s", dust::kStageNames[st]);
        e.launches = cnt[st];
        e.total_ms = ms[st];
    }
    return n;
}

}  // extern "C"

// Opt-in per-kernel device timing: when enabled, every kernel launch of the
// library is bracketed by two CUDA events recorded on its launch stream.
// Totals per kernel name are accumulated when they are read.  Off by default;
// when off a launch costs one relaxed atomic load more.
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kda_common.cuh"
#include "kda_timing.cuh"

namespace kda {
namespace {

struct Pending {
    const char* name;
    cudaEvent_t start, stop;
};
struct Total {
    std::string name;
    double ms = 0.0;
    long launches = 0;
};

std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Pending> g_pending;
std::vector<Total> g_totals;
std::vector<cudaEvent_t> g_free;

cudaEvent_t take_event() {
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

void drain_locked() {
    for (auto& p : g_pending) {
        float ms = 0.f;
        cudaEventSynchronize(p.stop);
        cudaEventElapsedTime(&ms, p.start, p.stop);
        Total* t = nullptr;
        for (auto& x : g_totals)
            if (x.name == p.name) t = &x;
        if (!t) {
            g_totals.push_back(Total{p.name, 0.0, 0});
            t = &g_totals.back();
        }
        t->ms += ms;
        t->launches += 1;
        g_free.push_back(p.start);
        g_free.push_back(p.stop);
    }
    g_pending.clear();
}

}  // namespace

TimedLaunch::TimedLaunch(const char* name, cudaStream_t s) : name_(name), s_(s) {
    if (!g_enabled.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    start_ = take_event();
    stop_ = take_event();
    if (start_ && stop_) cudaEventRecord(start_, s_);
    active_ = start_ && stop_;
}

TimedLaunch::~TimedLaunch() {
    if (!active_) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEventRecord(stop_, s_);
    g_pending.push_back(Pending{name_, start_, stop_});
}

}  // namespace kda

extern "C" {

void kda_timing_enable(int on) {
    std::lock_guard<std::mutex> lk(kda::g_mu);
    kda::drain_locked();
    kda::g_totals.clear();
    kda::g_enabled.store(on ? 1 : 0);
}

int kda_timing_count(void) {
    std::lock_guard<std::mutex> lk(kda::g_mu);
    kda::drain_locked();
    return (int)kda::g_totals.size();
}

int kda_timing_entry(int i, char* name, int name_len, double* total_ms, long* launches) {
    std::lock_guard<std::mutex> lk(kda::g_mu);
    kda::drain_locked();
    if (i < 0 || i >= (int)kda::g_totals.size()) return -1;
    const auto& t = kda::g_totals[i];
    if (name && name_len > 0) {
        std::strncpy(name, t.name.c_str(), name_len - 1);
        name[name_len - 1] = '\0';
    }
    if (total_ms) *total_ms = t.ms;
    if (launches) *launches = t.launches;
    return 0;
}

}  // extern "C"

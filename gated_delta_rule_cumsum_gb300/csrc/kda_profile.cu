// kda_profile.cu -- optional per-kernel CUDA-event timing (kda_profile_*).
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "kda_internal.cuh"

namespace {

struct Pending {
    std::string name;
    cudaEvent_t start, stop;
};

struct Totals {
    double ms = 0.0;
    int64_t launches = 0;
};

std::mutex g_mu;
bool g_enabled = false;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free;
std::map<std::string, Totals> g_totals;
thread_local const char *g_open_name = nullptr;
thread_local cudaEvent_t g_open_start = nullptr;

cudaEvent_t take_event() {
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

namespace kda {

void prof_begin(const char *name, cudaStream_t st) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_enabled) return;
    cudaEvent_t e = take_event();
    if (!e) return;
    cudaEventRecord(e, st);
    g_open_name = name;
    g_open_start = e;
}

void prof_end(cudaStream_t st) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_enabled || !g_open_start) return;
    cudaEvent_t e = take_event();
    if (!e) return;
    cudaEventRecord(e, st);
    g_pending.push_back(Pending{g_open_name, g_open_start, e});
    g_open_start = nullptr;
}

}  // namespace kda

extern "C" {

kda_status kda_profile_enable(int enable) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_enabled = enable != 0;
    return KDA_OK;
}

void kda_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto &p : g_pending) {
        cudaEventSynchronize(p.stop);
        g_free.push_back(p.start);
        g_free.push_back(p.stop);
    }
    g_pending.clear();
    g_totals.clear();
}

int kda_profile_report(char *names, size_t names_len, double *total_ms, int64_t *launches,
                       int max_entries) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto &p : g_pending) {
        if (cudaEventSynchronize(p.stop) != cudaSuccess) return -1;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess) return -1;
        Totals &t = g_totals[p.name];
        t.ms += ms;
        t.launches += 1;
        g_free.push_back(p.start);
        g_free.push_back(p.stop);
    }
    g_pending.clear();
    int n = 0;
    size_t off = 0;
    for (auto &kv : g_totals) {
        if (n >= max_entries) break;
        const size_t len = kv.first.size() + 1;
        if (names && off + len <= names_len) {
            std::memcpy(names + off, kv.first.c_str(), len);
            off += len;
        }
        if (total_ms) total_ms[n] = kv.second.ms;
        if (launches) launches[n] = kv.second.launches;
        ++n;
    }
    return n;
}

}  // extern "C"

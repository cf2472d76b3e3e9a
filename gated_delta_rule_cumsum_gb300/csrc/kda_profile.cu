// kda_profile.cu -- benchmark helpers: optional per-kernel CUDA-event timing
// (kda_profile_*) and the fp32 FMA peak microbenchmark
// (kda_measure_fp32_fma_peak).
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

// 16 independent FMA chains per thread; a full SM's worth of threads keeps
// every fp32 FMA lane busy.  Each chain converges to 1 (a <- 0.9999999 a + 1e-7),
// so the sum of positive values is stored only when it equals a negative value
// it never takes: the chains stay live without a memory write per thread, and
// the store's target is a device variable of this file.
constexpr int kChains = 16;
__device__ float g_fma_sink;
__global__ void __launch_bounds__(256) fma_peak_kernel(float seed, int iters) {
    float a[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) a[i] = seed + 1e-3f * i + 1e-7f * threadIdx.x;
    const float m = 0.9999999f, c = 1e-7f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) a[i] = fmaf(a[i], m, c);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += a[i];
    if (s == -1.25f) g_fma_sink = s;
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

kda_status kda_measure_fp32_fma_peak(double *tflops, kda_stream_t stream) {
    if (!tflops) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    constexpr int kIters = 1 << 15;
    const int blocks = sms * 8;  // 8 x 256 threads: a full SM each
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return KDA_ERR_CUDA;
    }
    float best = 0.f;
    bool ok = true;
    for (int rep = 0; rep < 4 && ok; ++rep) {  // the first launch warms up
        ok = cudaEventRecord(e0, st) == cudaSuccess;
        fma_peak_kernel<<<blocks, 256, 0, st>>>(1.0f + rep, kIters);
        ok = ok && cudaGetLastError() == cudaSuccess && cudaEventRecord(e1, st) == cudaSuccess &&
             cudaEventSynchronize(e1) == cudaSuccess;
        float ms = 0.f;
        ok = ok && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess;
        if (ok && rep > 0 && ms > 0.f && (best == 0.f || ms < best)) best = ms;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (!ok || best <= 0.f) return KDA_ERR_CUDA;
    const double flops = 2.0 * kChains * (double)kIters * blocks * 256.0;
    *tflops = flops / (best * 1e-3) / 1e12;
    return KDA_OK;
}

}  // extern "C"

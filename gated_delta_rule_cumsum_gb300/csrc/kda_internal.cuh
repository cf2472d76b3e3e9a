// kda_internal.cuh -- device helpers and launcher declarations shared by the
// translation units of the KDA library.  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kda.h"

namespace kda {

// One-time setup per device (kernel attributes such as the dynamic shared-memory
// limit, device properties): run(dev, set) calls set(*dev) for the current device
// the first time any thread asks for it, and only records success.  Devices
// 0..63; others fail with cudaErrorInvalidDevice.
struct DeviceOnce {
    std::atomic<uint64_t> done{0};
    std::mutex mu;
    template <typename F>
    cudaError_t run(int *dev, F &&set) {
        cudaError_t e = cudaGetDevice(dev);
        if (e != cudaSuccess) return e;
        if (*dev < 0 || *dev >= 64) return cudaErrorInvalidDevice;
        const uint64_t bit = 1ull << *dev;
        if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu);
        if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
        e = set(*dev);
        if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
        return e;
    }
};

// Chunk length of the chunked form (kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md,
// preamble: BT = 64).
constexpr int kBT = 64;

// ----------------------------------------------------------------- scalar I/O
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ void report(int32_t *status, int bits) {
    if (status) atomicOr(status, bits);
}

// Largest index i in [0, n) with a[i] <= x (a non-decreasing); 0 if none.
// Stays in bounds for any contents of a.
__device__ __forceinline__ int upper_bound_minus_one(const int32_t *a, int n, int x) {
    int lo = 0, hi = n;  // first index with a[i] > x lies in [lo, hi]
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (a[mid] <= x)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo > 0 ? lo - 1 : 0;
}

// ----------------------------------------------------------- workspace layout
// Control block at the start of the chunk workspace, written every call by the
// offsets pre-pass and read by the later kernels of the same call.
struct ChunkCtrl {
    int32_t valid;         // 1 when the offsets passed validation
    int32_t total_chunks;  // sum over sequences of ceil(len / BT)
    int32_t pad[62];       // 256 bytes
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Upper bound on the number of BT-row chunks of a call (host and device).
__host__ __device__ inline int64_t chunk_slots(const kda_shape &s, bool packed) {
    const int64_t ntc = (s.T + kBT - 1) / kBT;
    return packed ? ntc + s.num_seqs : (int64_t)s.B * ntc;
}

// ------------------------------------------------------------- stage timing
// When enabled (kda_profile_enable), every kernel the library enqueues is
// bracketed by a pair of CUDA events on its stream; kda_profile_report sums
// the elapsed times per kernel name.  No-ops when disabled.
void prof_begin(const char *name, cudaStream_t st);
void prof_end(cudaStream_t st);

// --------------------------------------------------------------- launchers
// Each returns the launch error (cudaSuccess when enqueued).
cudaError_t launch_validate_offsets(const int32_t *cu, int N, int T, int32_t *dev_status,
                                    ChunkCtrl *ctrl, int32_t *chunk_start, cudaStream_t st);

// Input activations (kda_activation): the natural-log gate
// -exp(A_log[hv]) softplus(g + dt_bias[hv, d]) in g's place when A_log is set,
// beta = sigmoid(x) * beta_scale rounded to the input dtype when beta_scale > 0.
struct GateAct {
    const float *A_log = nullptr;
    const float *dt_bias = nullptr;
    float beta_scale = 0.f;
};
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }
// 2^x by the PTX instruction ex2.approx.ftz.f32: one special-function-unit op,
// relative error near 2^-22, results below 2^-126 flushed to zero.
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// -exp(A_log[hv]) for the channel loop of one value head
__device__ __forceinline__ float gate_neg_a(const GateAct &a, int hv) { return -expf(a.A_log[hv]); }
__device__ __forceinline__ float gate_bias(const GateAct &a, int hv, int d, int K) {
    return a.dt_bias ? a.dt_bias[(size_t)hv * K + d] : 0.f;
}
template <typename T>
__device__ __forceinline__ float beta_activate(float x, float s) {
    const float y = s / (1.f + expf(-x));
    return to_f32(from_f32<T>(y));
}

cudaError_t launch_gate_cumsum(const float *g, float *out, const int32_t *cu, const kda_shape &s,
                               const GateAct &act,
                               int chunk, cudaStream_t st);

struct RecurrentArgs {
    const void *q, *k, *v;
    const float *g;
    const void *beta;
    const float *h0;
    const int32_t *cu;
    void *o;
    float *ht;
    int32_t *status;
    int B, T, H, HV, K, V, N;
    float scale, g_scale;
    int l2norm;
    GateAct act;
};
cudaError_t launch_recurrent(const RecurrentArgs &a, kda_dtype dt, cudaStream_t st);

// Gradients of the token recurrence (kda_recurrent_bwd).
struct RecurrentBwdArgs {
    const void *q, *k, *v;
    const float *g;
    const void *beta;
    const float *h0;
    const int32_t *cu;
    const void *dout;          // [B,T,HV,V], q's dtype
    const float *dht;          // [N,HV,K,V] or NULL
    float *dq, *dk, *dv, *dg, *dbeta, *dh0;  // fp32; dq, dk, dg, dbeta accumulate (zeroed first)
    float *ckpt;               // S at the start of every 8 tokens (per-column blocks)
    int32_t *status;
    int B, T, H, HV, K, V, N;
    float scale, g_scale;
    int l2norm;                // q, k normalised per (token, head) inside the op
    GateAct act;               // raw g / beta activated inside the op
    float *dA_log, *ddt_bias;  // [HV], [HV][K]: summed (zeroed first) when act sets them
};
// Workspace of kda_recurrent_bwd: the checkpoints of every 8 tokens.
size_t recurrent_bwd_ckpt_bytes(int B, int T, int N, int HV, int K, int V);
cudaError_t launch_recurrent_bwd(const RecurrentBwdArgs &a, kda_dtype dt, cudaStream_t st);
// Only the options' chain rules (q/k L2 norm when a.l2norm, the input activations
// when a.act sets them) on gradients already summed with respect to the normalised
// rows and the activated gate and beta (the chunked backward's last step).
cudaError_t launch_bwd_chain(const RecurrentBwdArgs &a, kda_dtype dt, cudaStream_t st);

// How a dense tensor-core forward is cut into pipelined parts: chunks
// [cut[i], cut[i + 1]) of every sequence form part i, cut[0] = 0, cut[parts] = nc.
// Two parts at most: at the training shape three and four parts measured slower
// than two (187-210 us against 181 us), each extra part adding a launch's start-up
// and more of the scans' time beside a prep than the model credits.
constexpr int kMaxPipeParts = 2;
struct PipePlan {
    int parts = 0;
    int cut[kMaxPipeParts + 1] = {};
};

struct ChunkArgs {
    const void *q, *k, *v;
    const float *g;
    const void *beta;
    const float *h0;
    const int32_t *cu;
    void *o;
    float *ht;
    int32_t *status;
    int B, T, H, HV, K, V, N;
    float scale, g_scale;
    int l2norm, g_is_cumsum;
    int test_timeout;      // KDA_FLAG_TEST_WAIT_TIMEOUT: the scan's MMA issuer waits on a
                           // barrier nothing signals (2 us limit) before its first round
    // workspace, carved by the host
    ChunkCtrl *ctrl;
    int32_t *chunk_start;  // [N + 1] (packed only)
    void *units;           // per-(chunk, value head) intermediates
    int64_t slots;         // chunk slots (upper bound)
    // split sequences (tensor-core path): see chunk_tc_split
    GateAct act;
    int split;
    void *qc;              // [slots][HV][64][K] bf16: segment 1's Q_c operand tiles
    float *e0, *e1;        // [N][HV][K][V] fp32: the segments' final states from zero / h0
    void *e0b;             // [N][HV] bf16 [K][V] operand tiles of e0
    float *pm;             // [N][HV][K][K] fp32: segment 1's state transition
    // Pipelined launches (tensor-core path, dense input): every sequence's chunks
    // run in parts [pipe.cut[i], pipe.cut[i + 1]).  Part 0 is prepped on every SM;
    // each later part's prep fills the SMs the scans leave free, and each part's
    // scan starts from the state the previous part's scan left in e0 (read, then
    // overwritten, by the same threads).
    PipePlan pipe;         // pipe.parts == 0: not pipelined
    int prep_c0, prep_c1;  // a prep launch's chunks within every sequence (c1 <= c0: all slots)
    int scan_c0, scan_c1;  // a pipelined scan launch's chunks within every sequence
    // The chunked backward's re-run of the forward: the prep also stores W_c and
    // Akk_c in each unit (tc_layout with bwd), the scan stores the state at the
    // start of every chunk (ck_h, a [dk][V] bf16 operand tile per unit) and v'_c
    // (ck_vp, a [64][V] tile per unit); o may then be null (not stored).
    int bwd = 0;
    void *ck_h = nullptr, *ck_vp = nullptr;
};
size_t chunk_simt_unit_bytes(int K, int V);
cudaError_t launch_chunk_simt(const ChunkArgs &a, kda_dtype dt, cudaStream_t st);

// Tensor-core path (bf16 inputs): K in {64, 128}, V a multiple of 32 up to 256.
bool chunk_tc_supported(int K, int V);
// The parts a dense input of B sequences of T rows is pipelined in on a GPU of
// `sms` SMs; parts == 0 when running the prep and then the scan, each over every
// chunk, is expected to be as fast.
PipePlan chunk_tc_pipe_plan(int B, int HV, int K, int V, int T, int sms);
// Whether a launch splits each sequence's scan into two segments run at once.
bool chunk_tc_split(int N, int HV, int K, int V, int T);
size_t chunk_tc_unit_bytes(int K, int V, bool bwd = false);
cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st);

// Chunked backward (kda_chunk_bwd), bf16 with K = V = 128: the forward re-run with
// `c.bwd` and its checkpoints (final states to hend, [N][HV][K][V] fp32), the reverse
// state scan (dhn, dvp: per-unit tiles; dgs: per unit [V/32][K] fp32 sums of
// h_{c+1} dh_{c+1}), then the per-chunk gradients.  dq and dk must be zeroed first
// when value heads share q/k heads (HV > H) or with packed sequences.
// A dense call of enough chunks pipelines the reverse scan with the gradient kernel
// (dhm: [N][HV][K][V] fp32, the state gradient where the two scan parts meet) unless
// `serial`.  Without `rerun` the forward's tiles, checkpoints and final states are
// already in place (kda_chunk_fwd_save) and the forward is not launched.
bool chunk_bwd_tc_supported(int K, int V);
int chunk_bwd_pipe_m(int B, int HV, int V, int T, int sms);
cudaError_t launch_chunk_bwd_tc(const ChunkArgs &c, const void *dout, const float *dht, float *dq,
                                float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                                void *dhn, void *dvp, float *hend, float *dgs, float *dhm,
                                bool serial, bool rerun, cudaStream_t st);

}  // namespace kda

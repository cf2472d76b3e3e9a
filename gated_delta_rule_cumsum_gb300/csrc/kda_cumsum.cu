// kda_cumsum.cu -- the chunk-local gate cumsum and the device-side validation
// of packed-sequence offsets.
//
// Gate cumsum: kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Stage 1 -- cumsum":
// a per-channel inclusive prefix sum that restarts every `chunk` rows, the
// chunks being counted from the first row of each sequence, times a multiplier
// (1/ln 2 there, where gates are natural logs; 1 for base-2 gates).
//
// Offsets: attention-gym PR #317, review comments on the packed path: validate
// 0 <= begin <= end <= tokens and a zero first offset on the device, on every
// call, with an always-enabled check that stays valid under CUDA-graph replay.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kTile = 64;  // rows per CTA of the cumsum

// One CTA per (64-row tile, batch row x value head), flattened onto grid x.  Threads stride over channels.
// Row t's segment starts at s(t) = bos + chunk * floor((t - bos) / chunk); the
// running sum of the first tile row starts at s(t0), which lies at most
// chunk - 1 rows before the tile, and no segment starts in between.
__global__ void __launch_bounds__(128) gate_cumsum_kernel(const float *__restrict__ g,
                                                          float *__restrict__ out,
                                                          const int32_t *__restrict__ cu,
                                                          int B, int T, int HV, int K, int N,
                                                          int chunk, float g_scale, GateAct act) {
    __shared__ int seg_start[kTile];
    __shared__ int row_valid[kTile];
    const int tiles = (T + kTile - 1) / kTile;
    const int t0 = (int)(blockIdx.x % tiles) * kTile;
    const int bh = (int)(blockIdx.x / tiles);
    const int hv = bh % HV;
    const int b = bh / HV;

    if (threadIdx.x < kTile) {
        const int i = threadIdx.x, t = t0 + i;
        int s = t, valid;
        if (cu) {
            int end = cu[N];
            end = end < 0 ? 0 : (end > T ? T : end);
            valid = t < end;
            if (valid) {
                const int n = upper_bound_minus_one(cu, N + 1, t);
                const int bos = cu[n];
                s = bos + chunk * ((t - bos) / chunk);
            }
        } else {
            valid = t < T;
            s = chunk * (t / chunk);
        }
        // Keep every read inside [t - chunk + 1, t] whatever the offsets hold.
        const int lo = t - chunk + 1 > 0 ? t - chunk + 1 : 0;
        s = s < lo ? lo : (s > t ? t : s);
        seg_start[i] = s;
        row_valid[i] = valid;
    }
    __syncthreads();

    const size_t rstride = (size_t)HV * K;
    const float *gb = g + ((size_t)b * T) * rstride + (size_t)hv * K;
    float *ob = out + ((size_t)b * T) * rstride + (size_t)hv * K;
    for (int d = threadIdx.x; d < K; d += blockDim.x) {
        // the gate of row u: g itself, or the activated -exp(A_log) softplus(g + dt_bias)
        const bool activate = act.A_log != nullptr;
        const float neg_a = activate ? gate_neg_a(act, hv) : 0.f;
        const float bias = activate ? gate_bias(act, hv, d, K) : 0.f;
        auto gate = [&](int u) {
            const float x = gb[(size_t)u * rstride + d];
            return activate ? neg_a * softplus_f(x + bias) : x;
        };
        float acc = 0.f;
        for (int u = seg_start[0]; u < t0; ++u) acc += gate(u);
        for (int i = 0; i < kTile; ++i) {
            if (!row_valid[i]) break;  // rows past the end of the valid range
            const int t = t0 + i;
            if (seg_start[i] == t) acc = 0.f;
            acc += gate(t);
            ob[(size_t)t * rstride + d] = g_scale * acc;
        }
    }
}

// Single CTA: validates cu[0..N] and, when asked, writes the chunk table
// chunk_start[n] = sum_{m < n} ceil((cu[m+1] - cu[m]) / BT) and the control word.
__global__ void __launch_bounds__(1024) validate_offsets_kernel(const int32_t *__restrict__ cu,
                                                                int N, int T,
                                                                int32_t *status, ChunkCtrl *ctrl,
                                                                int32_t *chunk_start) {
    __shared__ int32_t part[1024];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (N + nt - 1) / nt;
    const int lo = tid * per;
    const int hi = min(N, lo + per);
    bool ok = true;
    int32_t local = 0;
    for (int n = lo; n < hi; ++n) {
        const int32_t a = cu[n], c = cu[n + 1];
        ok = ok && (a >= 0) && (a <= c) && (c <= T);
        if (a <= c) local += (c - a + kBT - 1) / kBT;
    }
    if (tid == 0) ok = ok && (cu[0] == 0) && (cu[N] <= T) && (cu[N] >= 0);
    const bool all_ok = __syncthreads_and(ok) != 0;

    if (chunk_start) {
        part[tid] = local;
        __syncthreads();
        if (tid == 0) {  // exclusive scan of the per-thread sums (1024 adds)
            int32_t run = 0;
            for (int i = 0; i < nt; ++i) {
                const int32_t x = part[i];
                part[i] = run;
                run += x;
            }
            if (ctrl) {
                ctrl->total_chunks = all_ok ? run : 0;
                ctrl->valid = all_ok ? 1 : 0;
            }
        }
        __syncthreads();
        int32_t run = part[tid];
        for (int n = lo; n < hi; ++n) {
            chunk_start[n] = run;
            const int32_t a = cu[n], c = cu[n + 1];
            if (a <= c) run += (c - a + kBT - 1) / kBT;
        }
        if (hi == N && lo <= N) chunk_start[N] = run;
        if (N == 0 && tid == 0) chunk_start[0] = 0;
    } else if (ctrl && tid == 0) {
        ctrl->valid = all_ok ? 1 : 0;
        ctrl->total_chunks = 0;
    }
    if (!all_ok && tid == 0) report(status, KDA_DEVICE_BAD_CU_SEQLENS);
}

}  // namespace

cudaError_t launch_validate_offsets(const int32_t *cu, int N, int T, int32_t *dev_status,
                                    ChunkCtrl *ctrl, int32_t *chunk_start, cudaStream_t st) {
    int threads = 32;
    while (threads < 1024 && threads < N) threads *= 2;
    prof_begin("validate_offsets", st);
    validate_offsets_kernel<<<1, threads, 0, st>>>(cu, N, T, dev_status, ctrl, chunk_start);
    prof_end(st);
    return cudaGetLastError();
}

cudaError_t launch_gate_cumsum(const float *g, float *out, const int32_t *cu, const kda_shape &s,
                               const GateAct &act, int chunk, cudaStream_t st) {
    const int tiles = (s.T + kTile - 1) / kTile;
    const int rows = cu ? s.HV : s.B * s.HV;
    if (tiles == 0 || rows == 0) return cudaSuccess;
    const int64_t blocks = (int64_t)tiles * rows;  // flattened onto grid x
    prof_begin("gate_cumsum", st);
    gate_cumsum_kernel<<<(unsigned)blocks, 128, 0, st>>>(g, out, cu, s.B, s.T, s.HV, s.K,
                                                         s.num_seqs, chunk, s.g_scale, act);
    prof_end(st);
    return cudaGetLastError();
}

}  // namespace kda

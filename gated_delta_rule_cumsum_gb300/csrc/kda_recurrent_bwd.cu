// kda_recurrent_bwd.cu -- gradients of the KDA token recurrence.
//
// The backward's contract is that of kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md,
// "Backward" (given do and dht: dq, dk, dv, dbeta, dg with respect to the
// per-token decay, dh0; dq and dk summed over the value heads that share a q/k
// head), computed here for the token recurrence of attention-gym PR #317 (PR
// description), which the chunked form reaches exactly:
//     S' = Diag(e) S_{t-1},  e = 2^(g_scale g_t)      a = S'^T k
//     delta = beta (v - a)                              S_t = S' + k delta^T
//     o_t = scale S_t^T q
// Reverse mode through one token, with dS the gradient of S_t from the tokens
// after it plus dht:
//     dS += scale q do^T            dq = scale S_t do
//     ddelta = dS^T k               dk = dS delta + S' da,   da = -beta ddelta
//     dv = beta ddelta              dbeta = ddelta . (v - a)
//     dS' = dS + k da^T             de = rowsum(dS' o S_{t-1}),  dg = de e ln2 g_scale
//     dS  = Diag(e) dS'             (the gradient of S_{t-1})
//
// Layout: one CTA of 8 warps per (sequence, value head, 32 value columns); warp w
// owns columns 4w .. 4w + 3 of the block for all K <= 128 state rows, lane l the
// rows l + 32 r.  Value columns evolve independently in the recurrence, so the
// warps never exchange state: only dq, dk, de and dbeta sum over columns (shared
// memory atomics within the CTA, then one fp32 global atomic add per (token,
// row) per CTA).  The states S_{t-1} are recomputed: a first pass stores S at
// the start of every 16-token group; the backward then takes each group's two
// 8-token halves in reverse, recomputing from the group's checkpoint and keeping
// the half's eight states in shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kBG = 16;      // tokens per checkpoint
constexpr int kBR = 8;       // tokens per backward half-group
constexpr int kBWarps = 8;
constexpr int kBCols = 4;    // value columns per warp
constexpr int kBBlock = kBWarps * kBCols;
constexpr int kBRows = 4;    // state rows per lane (K <= 128)
constexpr float kLn2 = 0.69314718055994531f;

struct Lane {
    int d[kBRows];      // state rows
    bool rok[kBRows];
    int col[kBCols];    // value columns
    bool cok[kBCols];
};

__device__ __forceinline__ Lane lane_map(const RecurrentBwdArgs &p, int vb, int warp, int lane) {
    Lane L;
#pragma unroll
    for (int r = 0; r < kBRows; ++r) {
        L.d[r] = lane + 32 * r;
        L.rok[r] = L.d[r] < p.K;
    }
#pragma unroll
    for (int c = 0; c < kBCols; ++c) {
        L.col[c] = vb * kBBlock + warp * kBCols + c;
        L.cok[c] = L.col[c] < p.V;
    }
    return L;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// The slot range of sequence n; false (and the status bit) for invalid offsets.
__device__ __forceinline__ bool seq_range(const RecurrentBwdArgs &p, int n, int &b, int &bos,
                                          int &eos) {
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        b = 0;
        const bool ok = bos >= 0 && bos <= eos && eos <= p.T && (n != 0 || bos == 0);
        if (!ok && threadIdx.x == 0) report(p.status, KDA_DEVICE_BAD_CU_SEQLENS);
        return ok;
    }
    b = n;
    bos = 0;
    eos = p.T;
    return true;
}

// Checkpoint slot of group `grp` of sequence n (dense: n * groups per row + grp;
// packed: bos / 16 + n + grp, which never overlaps the next sequence's slots).
__device__ __forceinline__ int64_t ckpt_slot(const RecurrentBwdArgs &p, int n, int bos, int grp) {
    if (!p.cu) return (int64_t)n * ((p.T + kBG - 1) / kBG) + grp;
    return (int64_t)(bos / kBG) + n + grp;
}

// One token's inputs as this lane needs them.
struct Tok {
    float e[kBRows], k[kBRows], q[kBRows];
    float v[kBCols], dout[kBCols];
    float beta;
};

template <typename T>
__device__ __forceinline__ Tok load_tok(const RecurrentBwdArgs &p, const Lane &L, int b, int t,
                                        int h, int hv, bool need_q) {
    Tok x;
    const size_t row = (size_t)b * p.T + t;
    const T *k = static_cast<const T *>(p.k);
    const T *q = static_cast<const T *>(p.q);
    const T *v = static_cast<const T *>(p.v);
    const T *dout = static_cast<const T *>(p.dout);
#pragma unroll
    for (int r = 0; r < kBRows; ++r) {
        x.e[r] = 0.f;
        x.k[r] = 0.f;
        x.q[r] = 0.f;
        if (L.rok[r]) {
            x.k[r] = to_f32(k[(row * p.H + h) * p.K + L.d[r]]);
            if (need_q) x.q[r] = to_f32(q[(row * p.H + h) * p.K + L.d[r]]);
            x.e[r] = exp2f(p.g_scale * p.g[(row * p.HV + hv) * p.K + L.d[r]]);
        }
    }
#pragma unroll
    for (int c = 0; c < kBCols; ++c) {
        x.v[c] = L.cok[c] ? to_f32(v[(row * p.HV + hv) * p.V + L.col[c]]) : 0.f;
        x.dout[c] = (need_q && L.cok[c]) ? to_f32(dout[(row * p.HV + hv) * p.V + L.col[c]]) : 0.f;
    }
    x.beta = to_f32(static_cast<const T *>(p.beta)[row * p.HV + hv]);
    return x;
}

// S <- Diag(e) S + k (beta (v - (Diag(e) S)^T k))^T for this warp's columns.
__device__ __forceinline__ void step(float (&S)[kBRows][kBCols], const Tok &x) {
    float a[kBCols];
#pragma unroll
    for (int c = 0; c < kBCols; ++c) {
        float part = 0.f;
#pragma unroll
        for (int r = 0; r < kBRows; ++r) part = fmaf(x.e[r] * S[r][c], x.k[r], part);
        a[c] = warp_sum(part);
    }
#pragma unroll
    for (int c = 0; c < kBCols; ++c) {
        const float delta = x.beta * (x.v[c] - a[c]);
#pragma unroll
        for (int r = 0; r < kBRows; ++r) S[r][c] = fmaf(x.e[r], S[r][c], x.k[r] * delta);
    }
}

__device__ __forceinline__ void load_state(const float *src, const RecurrentBwdArgs &p, const Lane &L,
                                           float (&S)[kBRows][kBCols]) {
#pragma unroll
    for (int r = 0; r < kBRows; ++r)
#pragma unroll
        for (int c = 0; c < kBCols; ++c)
            S[r][c] = (src && L.rok[r] && L.cok[c]) ? src[(size_t)L.d[r] * p.V + L.col[c]] : 0.f;
}

__device__ __forceinline__ void store_state(float *dst, const RecurrentBwdArgs &p, const Lane &L,
                                            const float (&S)[kBRows][kBCols]) {
#pragma unroll
    for (int r = 0; r < kBRows; ++r)
#pragma unroll
        for (int c = 0; c < kBCols; ++c)
            if (L.rok[r] && L.cok[c]) dst[(size_t)L.d[r] * p.V + L.col[c]] = S[r][c];
}

// Pass 1: the recurrence, storing S at the start of every 16-token group.
template <typename T>
__global__ void __launch_bounds__(kBWarps * 32) recurrent_ckpt_kernel(RecurrentBwdArgs p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvb = (p.V + kBBlock - 1) / kBBlock;
    const int64_t bid = blockIdx.x;
    const int vb = (int)(bid % nvb);
    const int hv = (int)((bid / nvb) % p.HV);
    const int n = (int)(bid / ((int64_t)nvb * p.HV));
    const int h = hv / (p.HV / p.H);
    int b, bos, eos;
    if (!seq_range(p, n, b, bos, eos)) return;
    const Lane L = lane_map(p, vb, warp, lane);
    const size_t hvo = (size_t)hv * p.K * p.V;
    float S[kBRows][kBCols];
    load_state(p.h0 ? p.h0 + (size_t)n * p.HV * p.K * p.V + hvo : nullptr, p, L, S);
    for (int t = bos; t < eos; ++t) {
        const int u = t - bos;
        if (u % kBG == 0)
            store_state(p.ckpt + ckpt_slot(p, n, bos, u / kBG) * p.HV * p.K * p.V + hvo, p, L, S);
        const Tok x = load_tok<T>(p, L, b, t, h, hv, false);
        step(S, x);
    }
}

// Pass 2: the reverse sweep.
template <typename T>
__global__ void __launch_bounds__(kBWarps * 32, 1) recurrent_bwd_kernel(RecurrentBwdArgs p) {
    extern __shared__ __align__(16) float sm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // per warp: the half-group's states S_{t-1}, [kBR][kBRows][32 lanes] float4 (4 columns)
    float4 *st = reinterpret_cast<float4 *>(sm) + (size_t)warp * kBR * kBRows * 32;
    float *acc_q = sm + kBWarps * kBR * kBRows * 32 * 4;  // [kBR][128]
    float *acc_k = acc_q + kBR * 128;
    float *acc_e = acc_k + kBR * 128;
    float *acc_b = acc_e + kBR * 128;                    // [kBR]

    const int nvb = (p.V + kBBlock - 1) / kBBlock;
    const int64_t bid = blockIdx.x;
    const int vb = (int)(bid % nvb);
    const int hv = (int)((bid / nvb) % p.HV);
    const int n = (int)(bid / ((int64_t)nvb * p.HV));
    const int h = hv / (p.HV / p.H);
    int b, bos, eos;
    if (!seq_range(p, n, b, bos, eos)) return;  // uniform over the CTA
    const Lane L = lane_map(p, vb, warp, lane);
    const size_t hvo = (size_t)hv * p.K * p.V;
    const size_t nso = (size_t)n * p.HV * p.K * p.V;

    for (int i = threadIdx.x; i < 3 * kBR * 128 + kBR; i += blockDim.x) acc_q[i] = 0.f;
    float dS[kBRows][kBCols];
    load_state(p.dht ? p.dht + nso + hvo : nullptr, p, L, dS);
    __syncthreads();

    const int len = eos - bos;
    for (int grp = (len + kBG - 1) / kBG - 1; grp >= 0; --grp) {
        const int g0 = bos + grp * kBG;
        const int g1 = min(g0 + kBG, eos);
        const float *ck = p.ckpt + ckpt_slot(p, n, bos, grp) * p.HV * p.K * p.V + hvo;
        for (int half = (g1 - g0 - 1) / kBR; half >= 0; --half) {
            const int s0 = g0 + half * kBR;
            const int s1 = min(s0 + kBR, g1);
            // recompute S_{t-1} for t in [s0, s1) from the group's checkpoint
            float S[kBRows][kBCols];
            load_state(ck, p, L, S);
            for (int t = g0; t < s1; ++t) {
                if (t >= s0) {
#pragma unroll
                    for (int r = 0; r < kBRows; ++r)
                        st[((t - s0) * kBRows + r) * 32 + lane] =
                            make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
                }
                const Tok x = load_tok<T>(p, L, b, t, h, hv, false);
                step(S, x);
            }
            for (int t = s1 - 1; t >= s0; --t) {
                const int u = t - s0;
                const Tok x = load_tok<T>(p, L, b, t, h, hv, true);
                float Sp[kBRows][kBCols];
#pragma unroll
                for (int r = 0; r < kBRows; ++r) {
                    const float4 f = st[(u * kBRows + r) * 32 + lane];
                    Sp[r][0] = f.x; Sp[r][1] = f.y; Sp[r][2] = f.z; Sp[r][3] = f.w;
                }
                float a[kBCols], delta[kBCols];
#pragma unroll
                for (int c = 0; c < kBCols; ++c) {
                    float part = 0.f;
#pragma unroll
                    for (int r = 0; r < kBRows; ++r) part = fmaf(x.e[r] * Sp[r][c], x.k[r], part);
                    a[c] = warp_sum(part);
                    delta[c] = x.beta * (x.v[c] - a[c]);
                }
                // o's gradient into dS, and dq = scale S_t do
                float dqp[kBRows];
#pragma unroll
                for (int r = 0; r < kBRows; ++r) {
                    float s = 0.f;
#pragma unroll
                    for (int c = 0; c < kBCols; ++c) {
                        const float St = fmaf(x.e[r], Sp[r][c], x.k[r] * delta[c]);
                        s = fmaf(St, x.dout[c], s);
                        dS[r][c] = fmaf(p.scale * x.q[r], x.dout[c], dS[r][c]);
                    }
                    dqp[r] = p.scale * s;
                }
                float ddel[kBCols], da[kBCols];
                float dbp = 0.f;
#pragma unroll
                for (int c = 0; c < kBCols; ++c) {
                    float part = 0.f;
#pragma unroll
                    for (int r = 0; r < kBRows; ++r) part = fmaf(dS[r][c], x.k[r], part);
                    ddel[c] = warp_sum(part);
                    da[c] = -x.beta * ddel[c];
                    dbp = fmaf(ddel[c], x.v[c] - a[c], dbp);
                }
                if (lane == 0) {
                    const size_t vrow = ((size_t)b * p.T + t) * p.HV + hv;
#pragma unroll
                    for (int c = 0; c < kBCols; ++c)
                        if (L.cok[c]) p.dv[vrow * p.V + L.col[c]] = x.beta * ddel[c];
                    atomicAdd(&acc_b[u], dbp);
                }
#pragma unroll
                for (int r = 0; r < kBRows; ++r) {
                    float kp = 0.f, ep = 0.f;
#pragma unroll
                    for (int c = 0; c < kBCols; ++c) {
                        kp = fmaf(dS[r][c], delta[c], kp);
                        kp = fmaf(x.e[r] * Sp[r][c], da[c], kp);
                        const float dSp = fmaf(x.k[r], da[c], dS[r][c]);
                        ep = fmaf(dSp, Sp[r][c], ep);
                        dS[r][c] = x.e[r] * dSp;
                    }
                    if (L.rok[r]) {
                        atomicAdd(&acc_q[u * 128 + L.d[r]], dqp[r]);
                        atomicAdd(&acc_k[u * 128 + L.d[r]], kp);
                        atomicAdd(&acc_e[u * 128 + L.d[r]], ep);
                    }
                }
            }
            __syncthreads();  // the half-group's sums are complete
            for (int i = threadIdx.x; i < (s1 - s0) * 128; i += blockDim.x) {
                const int u = i >> 7, d = i & 127;
                if (d < p.K) {
                    const size_t row = (size_t)b * p.T + s0 + u;
                    atomicAdd(&p.dq[(row * p.H + h) * p.K + d], acc_q[i]);
                    atomicAdd(&p.dk[(row * p.H + h) * p.K + d], acc_k[i]);
                    const size_t gi = (row * p.HV + hv) * p.K + d;
                    const float e = exp2f(p.g_scale * p.g[gi]);
                    atomicAdd(&p.dg[gi], acc_e[i] * e * kLn2 * p.g_scale);
                }
                acc_q[i] = acc_k[i] = acc_e[i] = 0.f;
            }
            if ((int)threadIdx.x < s1 - s0) {
                atomicAdd(&p.dbeta[((size_t)b * p.T + s0 + threadIdx.x) * p.HV + hv],
                          acc_b[threadIdx.x]);
                acc_b[threadIdx.x] = 0.f;
            }
            __syncthreads();
        }
    }
    if (p.dh0) store_state(p.dh0 + nso + hvo, p, L, dS);
}

template <typename T>
cudaError_t launch_bwd_typed(const RecurrentBwdArgs &a, cudaStream_t st) {
    const int64_t blocks = (int64_t)a.N * a.HV * ((a.V + kBBlock - 1) / kBBlock);
    if (blocks == 0) return cudaSuccess;
    const int smem = (kBWarps * kBR * kBRows * 32 * 4 + 3 * kBR * 128 + kBR) * (int)sizeof(float);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(recurrent_bwd_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    prof_begin("recurrent_ckpt", st);
    recurrent_ckpt_kernel<T><<<(unsigned)blocks, kBWarps * 32, 0, st>>>(a);
    prof_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prof_begin("recurrent_bwd", st);
    recurrent_bwd_kernel<T><<<(unsigned)blocks, kBWarps * 32, smem, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

}  // namespace

int64_t recurrent_bwd_ckpt_slots(int B, int T, int N) {
    const int64_t dense = (int64_t)B * ((T + kBG - 1) / kBG);
    const int64_t packed = (int64_t)T / kBG + N + 1;
    return dense > packed ? dense : packed;
}

cudaError_t launch_recurrent_bwd(const RecurrentBwdArgs &a, kda_dtype dt, cudaStream_t st) {
    if (dt == KDA_DTYPE_BF16) return launch_bwd_typed<__nv_bfloat16>(a, st);
    return launch_bwd_typed<float>(a, st);
}

}  // namespace kda

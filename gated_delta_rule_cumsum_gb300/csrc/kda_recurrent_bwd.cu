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
// Layout: one CTA of 16 warps per (sequence, value head, 16 value columns); warp
// w owns column w of the block for all K <= 128 state rows, lane l the rows
// l + 32 r.  Value columns evolve independently in the recurrence, so the warps
// never exchange state: only dq, dk, de and dbeta sum over columns.  Tokens go in
// groups of 16: the CTA stages a group's k, 2^g, q, v, do and beta in shared
// memory, the next group's values travelling in registers while the current one
// is computed.  The states S_{t-1} are recomputed: a first pass stores S at the
// start of every 8-token half of a group; the backward then takes the halves in
// reverse, recomputing each from its own checkpoint and keeping its eight states
// in shared memory.  The reverse loop keeps only what is per column
// (dS, delta, da, dv); the sums over columns follow from the stored S_{t-1} and
// dS after the half:
//     dq = scale (e . sum_c S'_c do_c + k sum_c delta_c do_c)     (S_t = e S' + k delta^T)
//     dk = sum_c dS_c delta_c + e . sum_c S'_c da_c
//     de = sum_c dS_c . S'_c + k . sum_c da_c S'_c
// one thread per (token, row), then one fp32 global atomic add per (token, row)
// per CTA.  With the q/k L2-norm flag the staged
// rows are normalised per token and a last kernel applies the norm's chain rule
// to the summed dq and dk.  With the input activations (raw gate and beta) the
// staging activates them exactly as the forward does, and a last kernel turns the
// summed gradients of the gate and beta the recurrence used into those of the raw
// inputs, A_log and dt_bias.
#include "kda_internal.cuh"

#include <algorithm>

namespace kda {
namespace {

constexpr int kBG = 16;       // tokens per staged group
constexpr int kBR = 8;        // tokens per backward half-group and per checkpoint
constexpr int kBWarps = 16;   // one value column per warp
constexpr int kBThreads = kBWarps * 32;
constexpr int kBRows = 4;     // state rows per lane (K <= 128)
constexpr int kBK = 128;
constexpr int kBPlane = kBWarps * kBR * kBK;  // one value per (warp, token, row)
constexpr float kLn2 = 0.69314718055994531f;

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

// Checkpoint slot of half-group `hg` (tokens 8 hg ..) of sequence n (dense:
// n * halves per row + hg; packed: bos / 8 + n + hg, which never overlaps the
// next sequence's slots).
__device__ __forceinline__ int64_t ckpt_slot(const RecurrentBwdArgs &p, int n, int bos, int hg) {
    if (!p.cu) return (int64_t)n * ((p.T + kBR - 1) / kBR) + hg;
    return (int64_t)(bos / kBR) + n + hg;
}

// A checkpoint slot holds, per value head, the CTA blocks' 16 columns one after
// another, each column as the ceil(K / 32) x 32 rows its warp holds (lane l of
// row block r at r * 32 + l): every warp's stores and loads are whole lines.
__device__ __forceinline__ float *ckpt_col(const RecurrentBwdArgs &p, int64_t slot, int hv, int col) {
    const int nvb = (p.V + kBWarps - 1) / kBWarps, nr = (p.K + 31) / 32;
    return p.ckpt + (((size_t)slot * p.HV + hv) * nvb * kBWarps + col) * (size_t)nr * 32;
}
__device__ __forceinline__ void ckpt_store(float *dst, int K, int lane, const float (&S)[kBRows]) {
#pragma unroll
    for (int r = 0; r < kBRows; ++r)
        if (32 * r < K) dst[r * 32 + lane] = S[r];
}
__device__ __forceinline__ void ckpt_load(const float *src, int K, int lane, float (&S)[kBRows]) {
#pragma unroll
    for (int r = 0; r < kBRows; ++r) S[r] = 32 * r < K ? src[r * 32 + lane] : 0.f;
}

// A group's token inputs in shared memory: rows [kBG][128] of k, 2^g and (for
// the backward) q; columns [kBG][kBWarps] of v and do; beta [kBG].
struct Stage {
    float *k, *e, *q, *v, *dout, *beta;
};
constexpr int kStageFloats = 3 * kBG * kBK + 2 * kBG * kBWarps + kBG;

__device__ __forceinline__ Stage stage_at(float *base) {
    Stage s;
    s.k = base;
    s.e = s.k + kBG * kBK;
    s.q = s.e + kBG * kBK;
    s.v = s.q + kBG * kBK;
    s.dout = s.v + kBG * kBWarps;
    s.beta = s.dout + kBG * kBWarps;
    return s;
}

// The group's values this thread carries: (token, row) pairs tid + 512 i of the
// 16 x 128 rows, (token, column) pair tid of the 16 x 16 columns, beta tid < 16.
// They stay in the input dtype until carry_store: a conversion right after the
// load would wait for it there, and the loads would no longer overlap the
// current group's work.
template <typename T>
struct Carry {
    T k[4], q[4];
    float g[4];
    T v, dout, beta;
};

template <typename T, bool Q>
__device__ __forceinline__ void carry_load(const RecurrentBwdArgs &p, Carry<T> &c, int b, int t0,
                                           int t1, int h, int hv, int col0) {
    const T *k = static_cast<const T *>(p.k);
    const T *q = static_cast<const T *>(p.q);
    const T *v = static_cast<const T *>(p.v);
    const T *dout = static_cast<const T *>(p.dout);
    const T zero = from_f32<T>(0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + kBThreads * i, u = idx >> 7, d = idx & 127;
        c.k[i] = c.q[i] = zero;
        c.g[i] = 0.f;
        if (t0 + u < t1 && d < p.K) {
            const size_t row = (size_t)b * p.T + t0 + u;
            c.k[i] = k[(row * p.H + h) * p.K + d];
            c.g[i] = p.g[(row * p.HV + hv) * p.K + d];
            if (Q) c.q[i] = q[(row * p.H + h) * p.K + d];
        }
    }
    const int u = threadIdx.x / kBWarps, cc = threadIdx.x % kBWarps;  // 512 threads: 32 x 16
    c.v = c.dout = zero;
    if (u < kBG && t0 + u < t1 && col0 + cc < p.V) {
        const size_t vr = (((size_t)b * p.T + t0 + u) * p.HV + hv) * p.V + col0 + cc;
        c.v = v[vr];
        if (Q) c.dout = dout[vr];
    }
    c.beta = zero;
    if ((int)threadIdx.x < kBG && t0 + (int)threadIdx.x < t1)
        c.beta = static_cast<const T *>(p.beta)[((size_t)b * p.T + t0 + threadIdx.x) * p.HV + hv];
}

template <typename T, bool Q>
__device__ __forceinline__ void carry_store(const RecurrentBwdArgs &p, const Carry<T> &c,
                                            const Stage &s, int hv) {
    const float na = p.act.A_log ? gate_neg_a(p.act, hv) : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + kBThreads * i, d = idx & 127;
        float g = c.g[i];  // entries past K or the group: g = 0, unused
        if (p.act.A_log && d < p.K) g = na * softplus_f(g + gate_bias(p.act, hv, d, p.K));
        s.k[idx] = to_f32(c.k[i]);
        s.e[idx] = exp2f(p.g_scale * g);
        if (Q) s.q[idx] = to_f32(c.q[i]);
    }
    const int u = threadIdx.x / kBWarps, cc = threadIdx.x % kBWarps;
    if (u < kBG) {
        s.v[u * kBWarps + cc] = to_f32(c.v);
        if (Q) s.dout[u * kBWarps + cc] = to_f32(c.dout);
    }
    if ((int)threadIdx.x < kBG) {
        const float x = to_f32(c.beta);
        s.beta[threadIdx.x] = p.act.beta_scale > 0.f ? beta_activate<T>(x, p.act.beta_scale) : x;
    }
}

// With the L2-norm flag: the staged k (and q) rows of each token scaled by
// 1 / sqrt(sum x^2 + 1e-6); warp w takes token w (16 warps, 16 tokens).
template <bool Q>
__device__ __forceinline__ void normalise_stage(const Stage &s, int warp, int lane) {
    if (warp >= kBG) return;
    float *rows[2] = {s.k, s.q};
#pragma unroll
    for (int x = 0; x < (Q ? 2 : 1); ++x) {
        float *r = rows[x] + warp * kBK;
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < kBRows; ++i) ss = fmaf(r[lane + 32 * i], r[lane + 32 * i], ss);
        const float rn = 1.f / sqrtf(warp_sum(ss) + 1e-6f);
#pragma unroll
        for (int i = 0; i < kBRows; ++i) r[lane + 32 * i] *= rn;
    }
}

// S <- Diag(e) S + k (beta (v - (Diag(e) S)^T k))^T for this warp's column (token u of the stage);
// a = (Diag(e) S)^T k and delta are returned.
__device__ __forceinline__ void step(float (&S)[kBRows], const Stage &s, int u, int lane, int w,
                                     float &a, float &delta) {
    float e[kBRows], k[kBRows], part = 0.f;
#pragma unroll
    for (int r = 0; r < kBRows; ++r) {
        e[r] = s.e[u * kBK + lane + 32 * r];
        k[r] = s.k[u * kBK + lane + 32 * r];
        part = fmaf(e[r] * S[r], k[r], part);
    }
    a = warp_sum(part);
    delta = s.beta[u] * (s.v[u * kBWarps + w] - a);
#pragma unroll
    for (int r = 0; r < kBRows; ++r) S[r] = fmaf(e[r], S[r], k[r] * delta);
}

__device__ __forceinline__ void load_col(const float *src, const RecurrentBwdArgs &p, int lane,
                                         int col, float (&S)[kBRows]) {
#pragma unroll
    for (int r = 0; r < kBRows; ++r) {
        const int d = lane + 32 * r;
        S[r] = (src && d < p.K && col < p.V) ? src[(size_t)d * p.V + col] : 0.f;
    }
}

__device__ __forceinline__ void store_col(float *dst, const RecurrentBwdArgs &p, int lane, int col,
                                          const float (&S)[kBRows]) {
#pragma unroll
    for (int r = 0; r < kBRows; ++r) {
        const int d = lane + 32 * r;
        if (d < p.K && col < p.V) dst[(size_t)d * p.V + col] = S[r];
    }
}

// Pass 1: the recurrence, storing S at the start of every 8-token half-group.
template <typename T>
__global__ void __launch_bounds__(kBThreads) recurrent_ckpt_kernel(RecurrentBwdArgs p) {
    __shared__ float sm[kStageFloats];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvb = (p.V + kBWarps - 1) / kBWarps;
    const int64_t bid = blockIdx.x;
    const int vb = (int)(bid % nvb);
    const int hv = (int)((bid / nvb) % p.HV);
    const int n = (int)(bid / ((int64_t)nvb * p.HV));
    const int h = hv / (p.HV / p.H);
    int b, bos, eos;
    if (!seq_range(p, n, b, bos, eos)) return;
    const int col0 = vb * kBWarps, col = col0 + warp;
    const size_t hvo = (size_t)hv * p.K * p.V;
    const Stage s = stage_at(sm);
    float S[kBRows];
    load_col(p.h0 ? p.h0 + (size_t)n * p.HV * p.K * p.V + hvo : nullptr, p, lane, col, S);
    const int ng = (eos - bos + kBG - 1) / kBG;
    Carry<T> c;
    if (ng > 0) carry_load<T, false>(p, c, b, bos, eos, h, hv, col0);
    for (int grp = 0; grp < ng; ++grp) {
        const int t0 = bos + grp * kBG, t1 = min(t0 + kBG, eos);
        __syncthreads();  // the previous group is done with the stage
        carry_store<T, false>(p, c, s, hv);
        if (grp + 1 < ng) carry_load<T, false>(p, c, b, t1, min(t1 + kBG, eos), h, hv, col0);
        __syncthreads();
        if (p.l2norm) {
            normalise_stage<false>(s, warp, lane);
            __syncthreads();
        }
        for (int u = 0; u < t1 - t0; ++u) {
            if (u % kBR == 0)
                ckpt_store(ckpt_col(p, ckpt_slot(p, n, bos, 2 * grp + u / kBR), hv, col), p.K, lane, S);
            float a, delta;
            step(S, s, u, lane, warp, a, delta);
        }
    }
}

// Pass 2: the reverse sweep.
template <typename T>
__global__ void __launch_bounds__(kBThreads) recurrent_bwd_kernel(RecurrentBwdArgs p) {
    extern __shared__ __align__(16) float sm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Stage s = stage_at(sm);
    // [warp][kBR][kBRows][32] planes: S_{t-1} and dL/dS_t of each warp's column;
    // element (token j, row d) of warp w at (w kBR + j) 128 + d
    float *sSp = sm + kStageFloats;
    float *sdS = sSp + kBPlane;
    float *sDel = sdS + kBPlane;            // [kBR][kBWarps]: delta
    float *sDa = sDel + kBR * kBWarps;      // da
    float *sDb = sDa + kBR * kBWarps;       // ddelta (v - a): the column's dbeta term
    float *sAv = sDb + kBR * kBWarps;       // a = S'^T k, from the recompute
    float *st = sSp + (size_t)warp * kBR * kBK;
    float *sd = sdS + (size_t)warp * kBR * kBK;

    const int nvb = (p.V + kBWarps - 1) / kBWarps;
    const int64_t bid = blockIdx.x;
    const int vb = (int)(bid % nvb);
    const int hv = (int)((bid / nvb) % p.HV);
    const int n = (int)(bid / ((int64_t)nvb * p.HV));
    const int h = hv / (p.HV / p.H);
    int b, bos, eos;
    if (!seq_range(p, n, b, bos, eos)) return;  // uniform over the CTA
    const int col0 = vb * kBWarps, col = col0 + warp;
    const bool cok = col < p.V;
    const size_t hvo = (size_t)hv * p.K * p.V;
    const size_t nso = (size_t)n * p.HV * p.K * p.V;

    float dS[kBRows];
    load_col(p.dht ? p.dht + nso + hvo : nullptr, p, lane, col, dS);

    const int ng = (eos - bos + kBG - 1) / kBG;
    Carry<T> c;
    // the checkpoint of the next half to run, loaded one half ahead
    float Sn[kBRows];
    if (ng > 0) {
        const int g0 = bos + (ng - 1) * kBG;
        carry_load<T, true>(p, c, b, g0, eos, h, hv, col0);
        ckpt_load(ckpt_col(p, ckpt_slot(p, n, bos, (eos - bos - 1) / kBR), hv, col), p.K, lane, Sn);
    }
    for (int grp = ng - 1; grp >= 0; --grp) {
        const int g0 = bos + grp * kBG, g1 = min(g0 + kBG, eos);
        __syncthreads();  // the previous group is done with the stage
        carry_store<T, true>(p, c, s, hv);
        if (grp > 0) carry_load<T, true>(p, c, b, g0 - kBG, g0, h, hv, col0);
        __syncthreads();
        if (p.l2norm) {
            normalise_stage<true>(s, warp, lane);
            __syncthreads();
        }
        for (int half = (g1 - g0 - 1) / kBR; half >= 0; --half) {
            const int u0 = half * kBR, u1 = min(u0 + kBR, g1 - g0);
            // recompute S_{t-1} for the half's tokens from its checkpoint
            float S[kBRows];
#pragma unroll
            for (int r = 0; r < kBRows; ++r) S[r] = Sn[r];
            const int hg = 2 * grp + half;
            if (hg > 0) ckpt_load(ckpt_col(p, ckpt_slot(p, n, bos, hg - 1), hv, col), p.K, lane, Sn);
            for (int u = u0; u < u1; ++u) {
#pragma unroll
                for (int r = 0; r < kBRows; ++r) st[((u - u0) * kBRows + r) * 32 + lane] = S[r];
                float a, delta;
                step(S, s, u, lane, warp, a, delta);
                if (lane == 0) {  // a column past V has both zero
                    sAv[(u - u0) * kBWarps + warp] = a;
                    sDel[(u - u0) * kBWarps + warp] = delta;
                }
            }
            __syncwarp();
            for (int u = u1 - 1; u >= u0; --u) {
                const int j = u - u0;
                float e[kBRows], k[kBRows], q[kBRows];
#pragma unroll
                for (int r = 0; r < kBRows; ++r) {
                    e[r] = s.e[u * kBK + lane + 32 * r];
                    k[r] = s.k[u * kBK + lane + 32 * r];
                    q[r] = s.q[u * kBK + lane + 32 * r];
                }
                const float beta = s.beta[u];
                const float vv = s.v[u * kBWarps + warp], dd = s.dout[u * kBWarps + warp];
                const float a = sAv[j * kBWarps + warp];
                float dpart = 0.f;
#pragma unroll
                for (int r = 0; r < kBRows; ++r) {
                    dS[r] = fmaf(p.scale * q[r], dd, dS[r]);  // dL/dS_t
                    dpart = fmaf(dS[r], k[r], dpart);
                    sd[(j * kBRows + r) * 32 + lane] = dS[r];
                }
                const float ddel = warp_sum(dpart);
                const float da = -beta * ddel;
                if (lane == 0) {  // a column past V has all of these zero
                    if (cok) p.dv[(((size_t)b * p.T + g0 + u) * p.HV + hv) * p.V + col] = beta * ddel;
                    sDa[j * kBWarps + warp] = da;
                    sDb[j * kBWarps + warp] = ddel * (vv - a);
                }
#pragma unroll
                for (int r = 0; r < kBRows; ++r) dS[r] = e[r] * fmaf(k[r], da, dS[r]);
            }
            __syncthreads();  // the half-group's planes are complete
            // sums over the block's columns: thread (token j, row d)
            const int hl = u1 - u0, d = threadIdx.x & (kBK - 1);
            for (int j = threadIdx.x / kBK; j < hl; j += kBThreads / kBK) {
                const int u = u0 + j;
                float sa = 0.f, sb = 0.f, sc = 0.f, sdd = 0.f, ed = 0.f;
#pragma unroll
                for (int w = 0; w < kBWarps; ++w) {
                    const float sp = sSp[(w * kBR + j) * kBK + d], ds = sdS[(w * kBR + j) * kBK + d];
                    const float dow = s.dout[u * kBWarps + w];
                    const float del = sDel[j * kBWarps + w], daw = sDa[j * kBWarps + w];
                    sa = fmaf(sp, dow, sa);
                    sb = fmaf(sp, daw, sb);
                    sc = fmaf(ds, del, sc);
                    sdd = fmaf(ds, sp, sdd);
                    ed = fmaf(del, dow, ed);
                }
                const size_t row = (size_t)b * p.T + g0 + u;
                if (d < p.K) {
                    const float e = s.e[u * kBK + d], kk = s.k[u * kBK + d];
                    atomicAdd(&p.dq[(row * p.H + h) * p.K + d], p.scale * fmaf(e, sa, kk * ed));
                    atomicAdd(&p.dk[(row * p.H + h) * p.K + d], fmaf(e, sb, sc));
                    atomicAdd(&p.dg[(row * p.HV + hv) * p.K + d],
                              fmaf(kk, sb, sdd) * e * kLn2 * p.g_scale);
                }
                if (d == 0) {
                    float db = 0.f;
#pragma unroll
                    for (int w = 0; w < kBWarps; ++w) db += sDb[j * kBWarps + w];
                    atomicAdd(&p.dbeta[row * p.HV + hv], db);
                }
            }
            __syncthreads();
        }
    }
    if (p.dh0) store_col(p.dh0 + nso + hvo, p, lane, col, dS);
}

// The L2 norm's chain rule, after every contribution to dq and dk has been
// summed: for a raw row x with r = 1 / sqrt(sum x^2 + 1e-6) and x^ = r x, the
// gradient of x is r (dx^ - x^ (x^ . dx^)).  One warp per (row, head) of q or k;
// rows at or past the last offset (packed) hold zeros and are left alone.
template <typename T>
__global__ void __launch_bounds__(256) l2norm_bwd_kernel(RecurrentBwdArgs p, int64_t rows) {
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= 2 * rows) return;
    const bool is_k = w >= rows;
    const int64_t rh = is_k ? w - rows : w;  // (token row) * H + head
    const int64_t tok = rh / p.H;
    if (p.cu && (tok % p.T) >= p.cu[p.N]) return;
    const T *x = static_cast<const T *>(is_k ? p.k : p.q) + rh * p.K;
    float *dx = (is_k ? p.dk : p.dq) + rh * p.K;
    float xv[kBRows], dv[kBRows], ss = 0.f;
#pragma unroll
    for (int i = 0; i < kBRows; ++i) {
        const int d = lane + 32 * i;
        xv[i] = d < p.K ? to_f32(x[d]) : 0.f;
        dv[i] = d < p.K ? dx[d] : 0.f;
        ss = fmaf(xv[i], xv[i], ss);
    }
    const float r = 1.f / sqrtf(warp_sum(ss) + 1e-6f);
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < kBRows; ++i) dot = fmaf(xv[i] * r, dv[i], dot);
    dot = warp_sum(dot);
#pragma unroll
    for (int i = 0; i < kBRows; ++i) {
        const int d = lane + 32 * i;
        if (d < p.K) dx[d] = r * (dv[i] - xv[i] * r * dot);
    }
}

// The input activations' chain rule, after the sweep has summed dg and dbeta with
// respect to the gate and beta the recurrence used.  With x = g + dt_bias and
// g' = -exp(A_log) softplus(x): dg'/dx = -exp(A_log) sigmoid(x) (also dt_bias's
// gradient) and dg'/dA_log = g'.  With beta' = s sigmoid(y): dbeta'/dy =
// s sigmoid(y) (1 - sigmoid(y)); the rounding of beta' to the input dtype passes
// the gradient through.  Thread column c of the HV * K gate columns takes rows
// blockIdx.y, + gridDim.y, ...; the sums over rows go to dt_bias's gradient by
// one atomic per (block, column) and to A_log's through shared memory.  Rows at
// or past the last offset (packed) are left alone.
template <typename T>
__global__ void __launch_bounds__(256) act_bwd_kernel(RecurrentBwdArgs p, int64_t rows) {
    __shared__ float sA[256];  // A_log sums of the value heads this block's columns touch
    const int cols = p.HV * p.K;
    const int c0 = blockIdx.x * 256, c = c0 + threadIdx.x, hv0 = c0 / p.K;
    const int64_t end = p.cu ? min((int64_t)max(p.cu[p.N], 0), rows) : rows;
    sA[threadIdx.x] = 0.f;
    __syncthreads();
    if (p.act.A_log && c < cols) {
        const int hv = c / p.K, d = c - hv * p.K;
        const float na = gate_neg_a(p.act, hv), bias = gate_bias(p.act, hv, d, p.K);
        float sb = 0.f, sa = 0.f;
        for (int64_t r = blockIdx.y; r < end; r += gridDim.y) {
            const size_t i = (size_t)r * cols + c;
            const float x = p.g[i] + bias, dga = p.dg[i];
            const float dx = dga * na / (1.f + expf(-x));
            p.dg[i] = dx;
            sb += dx;
            sa = fmaf(dga, na * softplus_f(x), sa);
        }
        if (p.ddt_bias) atomicAdd(&p.ddt_bias[c], sb);
        atomicAdd(&sA[hv - hv0], sa);
    }
    if (blockIdx.x == 0 && p.act.beta_scale > 0.f) {
        const T *beta = static_cast<const T *>(p.beta);
        for (int hv = threadIdx.x; hv < p.HV; hv += blockDim.x)
            for (int64_t r = blockIdx.y; r < end; r += gridDim.y) {
                const size_t i = (size_t)r * p.HV + hv;
                const float sg = 1.f / (1.f + expf(-to_f32(beta[i])));
                p.dbeta[i] *= p.act.beta_scale * sg * (1.f - sg);
            }
    }
    __syncthreads();
    const int hv = hv0 + threadIdx.x;
    if (p.act.A_log && hv <= (min(cols, c0 + 256) - 1) / p.K) atomicAdd(&p.dA_log[hv], sA[threadIdx.x]);
}

template <typename T>
cudaError_t launch_chain_typed(const RecurrentBwdArgs &a, cudaStream_t st);

template <typename T>
cudaError_t launch_bwd_typed(const RecurrentBwdArgs &a, cudaStream_t st) {
    const int64_t blocks = (int64_t)a.N * a.HV * ((a.V + kBWarps - 1) / kBWarps);
    if (blocks == 0) return cudaSuccess;
    const int smem = (kStageFloats + 2 * kBPlane + 4 * kBR * kBWarps) * (int)sizeof(float);
    static DeviceOnce once;
    int dev = 0;
    {
        const cudaError_t e = once.run(&dev, [smem](int) {
            return cudaFuncSetAttribute(recurrent_bwd_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        });
        if (e != cudaSuccess) return e;
    }
    prof_begin("recurrent_ckpt", st);
    recurrent_ckpt_kernel<T><<<(unsigned)blocks, kBThreads, 0, st>>>(a);
    prof_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prof_begin("recurrent_bwd", st);
    recurrent_bwd_kernel<T><<<(unsigned)blocks, kBThreads, smem, st>>>(a);
    prof_end(st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_chain_typed<T>(a, st);
}

// The options' chain rules on summed gradients (the q/k L2 norm, then the input
// activations), shared with the chunked backward.
template <typename T>
cudaError_t launch_chain_typed(const RecurrentBwdArgs &a, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    const int64_t rows = (int64_t)a.B * a.T;
    if (rows == 0) return cudaSuccess;
    if (a.l2norm) {
        const int64_t nb = (2 * rows * a.H * 32 + 255) / 256;
        prof_begin("l2norm_bwd", st);
        l2norm_bwd_kernel<T><<<(unsigned)nb, 256, 0, st>>>(a, rows * a.H);
        prof_end(st);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.act.A_log || a.act.beta_scale > 0.f) {
        // about four blocks per SM, each block's threads over a share of the rows
        const unsigned gx = (unsigned)((a.HV * a.K + 255) / 256);
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        const int64_t want = (4 * (int64_t)sms + gx - 1) / gx;
        const unsigned gy = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, std::min<int64_t>(rows, 65535)));
        prof_begin("act_bwd", st);
        act_bwd_kernel<T><<<dim3(gx, gy), 256, 0, st>>>(a, rows);
        prof_end(st);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

size_t recurrent_bwd_ckpt_bytes(int B, int T, int N, int HV, int K, int V) {
    const int64_t dense = (int64_t)B * ((T + kBR - 1) / kBR);
    const int64_t packed = (int64_t)T / kBR + N + 1;
    const int64_t slots = dense > packed ? dense : packed;
    const int64_t cols = (int64_t)((V + kBWarps - 1) / kBWarps) * kBWarps;
    return (size_t)(slots * HV * cols * ((K + 31) / 32) * 32 * (int64_t)sizeof(float));
}

cudaError_t launch_recurrent_bwd(const RecurrentBwdArgs &a, kda_dtype dt, cudaStream_t st) {
    if (dt == KDA_DTYPE_BF16) return launch_bwd_typed<__nv_bfloat16>(a, st);
    return launch_bwd_typed<float>(a, st);
}

cudaError_t launch_bwd_chain(const RecurrentBwdArgs &a, kda_dtype dt, cudaStream_t st) {
    if (dt == KDA_DTYPE_BF16) return launch_chain_typed<__nv_bfloat16>(a, st);
    return launch_chain_typed<float>(a, st);
}

}  // namespace kda

// kda_recurrent.cu -- token-by-token KDA forward (decode and inference prefill).
//
// attention-gym PR #317 "Add fused recurrent_kda for decode and inference
// prefill", PR description: a sequential scan over the tokens of each
// (sequence, head, value block) with the [K, BV] fp32 state held in registers,
// fp32 arithmetic whatever the input dtype, queries scaled by 1/sqrt(K),
// device-resident int32 offsets with empty slots passing their state through
// bitwise.  The review comments of that PR add: work flattened onto grid x (so
// N * HV beyond 65535 launches), and offsets validated on the device on every
// call with an always-on check rather than an assertion.
//
// One CTA per (sequence n, value head hv, value block of 128 columns).  Warp w
// holds state rows d in [16w, 16w + 16); lane l holds columns [4l, 4l + 4) of
// the block, so each thread keeps a 16 x 4 fp32 tile of S in registers and the
// state streams through HBM in coalesced 512-byte rows.
//
// Per token the update is evaluated as
//     a     = S^T (2^g * k)          b = S^T (2^g * q)          (one pass over S)
//     delta = beta (v - a / |k|)                                 (|.| = 1 w/o L2 norm)
//     o     = scale (b / |q| + delta (k.q) / (|k||q|))
//     S     = Diag(2^g) S + (k / |k|) delta^T
// which equals S_t = (I - beta k k^T) Diag(2^g) S_{t-1} + beta k v^T followed by
// o_t = scale S_t^T q_t, since (Diag(2^g) S + k delta^T)^T q expands into the two
// terms of o.  Both reductions over d read the OLD state, so a token costs a
// single block-wide exchange (double-buffered shared memory, one barrier).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kRows = 16;      // state rows per warp
constexpr int kCols = 4;       // state columns per lane
constexpr int kBlockV = 128;   // value columns per CTA (32 lanes x 4)
constexpr int kRedStride = 2 * kBlockV + 4;  // per-warp partials: a[128], b[128], |k|^2, |q|^2, k.q

template <typename T, bool VEC>
__global__ void __launch_bounds__(512) recurrent_kernel(RecurrentArgs p) {
    extern __shared__ float red[];  // [2][nwarps][kRedStride]
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvb = (p.V + kBlockV - 1) / kBlockV;

    const int64_t bid = blockIdx.x;
    const int vb = (int)(bid % nvb);
    const int64_t nh = bid / nvb;
    const int hv = (int)(nh % p.HV);
    const int n = (int)(nh / p.HV);
    const int h = hv / (p.HV / p.H);

    int b, bos, eos;
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        b = 0;
        const bool ok = bos >= 0 && bos <= eos && eos <= p.T && (n != 0 || bos == 0);
        if (!ok) {  // skip the whole slot: nothing is read or written
            if (threadIdx.x == 0) report(p.status, KDA_DEVICE_BAD_CU_SEQLENS);
            return;
        }
    } else {
        b = n;
        bos = 0;
        eos = p.T;
    }

    const int d0 = warp * kRows;
    const int c0 = vb * kBlockV + lane * kCols;
    const size_t sbase = ((size_t)n * p.HV + hv) * (size_t)p.K * p.V;
    const bool lane_full = c0 + kCols <= p.V;

    float S[kRows][kCols];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const int d = d0 + r;
        if (p.h0 && d < p.K) {
            const float *src = p.h0 + sbase + (size_t)d * p.V + c0;
            if (VEC && lane_full) {
                const float4 x = *reinterpret_cast<const float4 *>(src);
                S[r][0] = x.x; S[r][1] = x.y; S[r][2] = x.z; S[r][3] = x.w;
            } else {
#pragma unroll
                for (int j = 0; j < kCols; ++j) S[r][j] = (c0 + j < p.V) ? src[j] : 0.f;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kCols; ++j) S[r][j] = 0.f;
        }
    }

    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    const T *beta = static_cast<const T *>(p.beta);
    T *o = static_cast<T *>(p.o);
    const int dl = d0 + lane;  // the row lanes 0..15 fetch
    const bool row_lane = lane < kRows && dl < p.K;

    // Inputs of token t, fetched one token ahead (the activations applied as they
    // arrive: the gate's per-channel constants are loaded once).
    const bool gate_act = p.act.A_log != nullptr;
    const float neg_a = gate_act ? gate_neg_a(p.act, hv) : 0.f;
    const float gbias = gate_act && row_lane ? gate_bias(p.act, hv, dl, p.K) : 0.f;
    float kr = 0.f, qr = 0.f, gr = 0.f, vv[kCols] = {0.f, 0.f, 0.f, 0.f}, bt = 0.f;
    auto fetch = [&](int t) {
        const size_t row = (size_t)b * p.T + t;
        if (row_lane) {
            kr = to_f32(k[(row * p.H + h) * p.K + dl]);
            qr = to_f32(q[(row * p.H + h) * p.K + dl]);
            gr = p.g[(row * p.HV + hv) * p.K + dl];
            if (gate_act) gr = neg_a * softplus_f(gr + gbias);
        }
        const size_t vrow = (row * p.HV + hv) * p.V;
#pragma unroll
        for (int j = 0; j < kCols; ++j) vv[j] = (c0 + j < p.V) ? to_f32(v[vrow + c0 + j]) : 0.f;
        bt = to_f32(beta[row * p.HV + hv]);
        if (p.act.beta_scale > 0.f) bt = beta_activate<T>(bt, p.act.beta_scale);
    };
    if (bos < eos) fetch(bos);

    int buf = 0;
    for (int t = bos; t < eos; ++t) {
        const float k_t = kr, q_t = qr, b_t = bt;
        const float dec = row_lane ? exp2f(p.g_scale * gr) : 1.f;
        float v_t[kCols];
#pragma unroll
        for (int j = 0; j < kCols; ++j) v_t[j] = vv[j];
        if (t + 1 < eos) fetch(t + 1);

        const float kd = k_t * dec, qd = q_t * dec;
        float a[kCols] = {0.f, 0.f, 0.f, 0.f}, bq[kCols] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float kd_r = __shfl_sync(0xffffffffu, kd, r);
            const float qd_r = __shfl_sync(0xffffffffu, qd, r);
#pragma unroll
            for (int j = 0; j < kCols; ++j) {
                a[j] = fmaf(S[r][j], kd_r, a[j]);
                bq[j] = fmaf(S[r][j], qd_r, bq[j]);
            }
        }
        float ks = k_t * k_t, qs = q_t * q_t, kq = k_t * q_t;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {  // lanes >= 16 hold zeros
            ks += __shfl_xor_sync(0xffffffffu, ks, off);
            qs += __shfl_xor_sync(0xffffffffu, qs, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }
        float *rb = red + ((size_t)buf * nwarps + warp) * kRedStride;
#pragma unroll
        for (int j = 0; j < kCols; ++j) {
            rb[lane * kCols + j] = a[j];
            rb[kBlockV + lane * kCols + j] = bq[j];
        }
        if (lane == 0) {
            rb[2 * kBlockV + 0] = ks;
            rb[2 * kBlockV + 1] = qs;
            rb[2 * kBlockV + 2] = kq;
        }
        __syncthreads();

        float A[kCols] = {0.f, 0.f, 0.f, 0.f}, Bq[kCols] = {0.f, 0.f, 0.f, 0.f};
        float nk = 0.f, nq = 0.f, nkq = 0.f;
        const float *rall = red + (size_t)buf * nwarps * kRedStride;
        for (int w = 0; w < nwarps; ++w) {
            const float *rw = rall + (size_t)w * kRedStride;
#pragma unroll
            for (int j = 0; j < kCols; ++j) {
                A[j] += rw[lane * kCols + j];
                Bq[j] += rw[kBlockV + lane * kCols + j];
            }
            nk += rw[2 * kBlockV + 0];
            nq += rw[2 * kBlockV + 1];
            nkq += rw[2 * kBlockV + 2];
        }
        const float rk = p.l2norm ? 1.f / sqrtf(nk + 1e-6f) : 1.f;
        const float rq = p.l2norm ? 1.f / sqrtf(nq + 1e-6f) : 1.f;
        const float kq_hat = nkq * rk * rq;
        float delta[kCols];
#pragma unroll
        for (int j = 0; j < kCols; ++j) delta[j] = b_t * (v_t[j] - rk * A[j]);
        if (warp == 0) {
            const size_t orow = (((size_t)b * p.T + t) * p.HV + hv) * p.V;
#pragma unroll
            for (int j = 0; j < kCols; ++j)
                if (c0 + j < p.V)
                    o[orow + c0 + j] = from_f32<T>(p.scale * (rq * Bq[j] + delta[j] * kq_hat));
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float kn_r = __shfl_sync(0xffffffffu, k_t, r) * rk;
            const float dec_r = __shfl_sync(0xffffffffu, dec, r);
#pragma unroll
            for (int j = 0; j < kCols; ++j) S[r][j] = fmaf(S[r][j], dec_r, kn_r * delta[j]);
        }
        buf ^= 1;
    }

    if (p.ht) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int d = d0 + r;
            if (d >= p.K) continue;
            float *dst = p.ht + sbase + (size_t)d * p.V + c0;
            if (VEC && lane_full) {
                *reinterpret_cast<float4 *>(dst) = make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
            } else {
#pragma unroll
                for (int j = 0; j < kCols; ++j)
                    if (c0 + j < p.V) dst[j] = S[r][j];
            }
        }
    }
}

// ---------------------------------------------------------------- long sequences
// The same recurrence for slots of many tokens, laid out so that no token needs
// a CTA-wide exchange.  One CTA of 8 warps per (sequence, value head, value
// block of 128 columns); warp w owns columns [16w, 16w + 16) of the block for
// ALL state rows (K <= 128): lane l holds rows d = 8r + (l >> 2), r = 0..15, and
// columns 4 (l & 3) .. 4 (l & 3) + 3.  The reductions over d are a sum over the
// thread's 16 rows plus three xor-shuffle levels across the warp's 8 row groups,
// after which every lane holds the full S^T(2^g k) and S^T(2^g q) of its columns.
// Rows d and d + 8 of a column sit in one float2 so that the paired fp32
// instructions (two lanes of arithmetic per instruction, each rounded as fmaf)
// carry the state update and both reductions.
//
// Tokens go in groups of 16.  While a group is computed, the next group's k, q,
// g rows (17 of them: the group plus the token after it) and v rows stream into
// shared memory with cp.async.  A transform pass turns them, per (token u, row
// pair), into two float4 planes: A = {2^g_u, k_u} and B = {2^g_{u+1} k_{u+1},
// 2^g_{u+1} q_{u+1}} (each value for rows d and d + 8), plus the token scalars
// {1/|k|, 1/|q|, (k.q)/(|k||q|), beta}.  The state update of token u and the
// reductions for token u+1 then run as ONE pass over the registers:
//     S[d][j] = 2^g_u[d] S[d][j] + k_u[d] dk_j;   a_j += S[d][j] 2^g_{u+1} k_{u+1}[d]; ...
constexpr int kLG = 16;       // tokens per group
constexpr int kLPairs = 8;    // row pairs per thread (16 rows)
constexpr int kLMaxK = 128;
constexpr int kLThreads = 256;
// A group runs in the scaled form while every row's running exponent stays
// within 2^+-60 (k / D and S / D then stay far from fp32 overflow).
constexpr float kLWide = 60.f;

template <typename T>
struct LongSmem {
    static constexpr int kRawRows = kLG + 1;
    static constexpr int planeA = 0;                                  // float4 [kLG][8][8]
    static constexpr int planeB = planeA + kLG * 64 * 16;             // float4 [kLG][8][8]
    static constexpr int pro = planeB + kLG * 64 * 16;                // float4 [8][8]
    static constexpr int scal = pro + 64 * 16;                        // float4 [kLG]
    static constexpr int dlast = scal + kLG * 16;                     // float [128]
    static constexpr int raw = dlast + kLMaxK * 4;                    // two buffers
    static constexpr int rk = 0;                                      // T [17][128]
    static constexpr int rq = rk + kRawRows * kLMaxK * (int)sizeof(T);
    static constexpr int rg = rq + kRawRows * kLMaxK * (int)sizeof(T);  // float [17][128]
    static constexpr int rv = rg + kRawRows * kLMaxK * 4;             // T [16][128]
    static constexpr int raw_bytes = rv + kLG * 128 * (int)sizeof(T);
    static constexpr int total = raw + 2 * raw_bytes;
    static_assert(rq % 16 == 0 && rg % 16 == 0 && rv % 16 == 0 && raw_bytes % 16 == 0, "align");
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ void load4(const float *p, float (&x)[4]) {
    const float4 f = *reinterpret_cast<const float4 *>(p);
    x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&x)[4]) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    x[0] = lo.x; x[1] = lo.y; x[2] = hi.x; x[3] = hi.y;
}
__device__ __forceinline__ void store4(float *p, const float (&x)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, const float (&x)[4]) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]);
    __nv_bfloat162 hi = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<unsigned *>(&lo);
    u.y = *reinterpret_cast<unsigned *>(&hi);
    *reinterpret_cast<uint2 *>(p) = u;
}

// Queue the raw rows of the group starting at token t0 (nrows k/q/g rows, nv v rows).
template <typename T>
__device__ __forceinline__ void long_issue(const RecurrentArgs &p, unsigned char *buf, int b,
                                           int h, int hv, int c_base, int vcols, int t0,
                                           int nrows, int nv) {
    using S = LongSmem<T>;
    constexpr int kPer = 16 / (int)sizeof(T);  // elements per 16-byte chunk
    const int kc = p.K / kPer, gc = p.K / 4, vc = vcols / kPer;
    const int nk = nrows * kc, ng = nrows * gc, nvv = nv * vc;
    const T *k = static_cast<const T *>(p.k);
    const T *q = static_cast<const T *>(p.q);
    const T *v = static_cast<const T *>(p.v);
    for (int c = threadIdx.x; c < 2 * nk + ng + nvv; c += kLThreads) {
        if (c < 2 * nk) {
            const int which = c >= nk, cc = c - which * nk;
            const int row = cc / kc, col = cc - row * kc;
            const size_t grow = (size_t)b * p.T + t0 + row;
            const T *src = (which ? q : k) + (grow * p.H + h) * p.K + col * kPer;
            cp_async16(buf + (which ? S::rq : S::rk) + (row * kLMaxK + col * kPer) * sizeof(T), src);
        } else if (c < 2 * nk + ng) {
            const int cc = c - 2 * nk, row = cc / gc, col = cc - row * gc;
            const size_t grow = (size_t)b * p.T + t0 + row;
            cp_async16(buf + S::rg + (row * kLMaxK + col * 4) * 4, p.g + (grow * p.HV + hv) * p.K + col * 4);
        } else {
            const int cc = c - 2 * nk - ng, row = cc / vc, col = cc - row * vc;
            const size_t grow = (size_t)b * p.T + t0 + row;
            cp_async16(buf + S::rv + (row * 128 + col * kPer) * sizeof(T),
                       v + (grow * p.HV + hv) * p.V + c_base + col * kPer);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kLThreads, 2) recurrent_long_kernel(RecurrentArgs p) {
    using SM = LongSmem<T>;
    extern __shared__ __align__(16) unsigned char smem[];
    float4 *planeA = reinterpret_cast<float4 *>(smem + SM::planeA);
    float4 *planeB = reinterpret_cast<float4 *>(smem + SM::planeB);
    float4 *pro = reinterpret_cast<float4 *>(smem + SM::pro);
    float *scal = reinterpret_cast<float *>(smem + SM::scal);
    float *sDlast = reinterpret_cast<float *>(smem + SM::dlast);
    __shared__ int sWide;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rgrp = lane >> 2, cgrp = lane & 3;
    const int nvb = (p.V + 127) / 128;
    const int64_t bid = blockIdx.x;
    const int vb = (int)(bid % nvb);
    const int64_t nh = bid / nvb;
    const int hv = (int)(nh % p.HV);
    const int n = (int)(nh / p.HV);
    const int h = hv / (p.HV / p.H);

    int b, bos, eos;
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        b = 0;
        const bool ok = bos >= 0 && bos <= eos && eos <= p.T && (n != 0 || bos == 0);
        if (!ok) {
            if (threadIdx.x == 0) report(p.status, KDA_DEVICE_BAD_CU_SEQLENS);
            return;
        }
    } else {
        b = n;
        bos = 0;
        eos = p.T;
    }

    const int c_base = vb * 128;
    const int vcols = min(128, p.V - c_base);
    const int cl = warp * 16 + cgrp * 4;  // first of this thread's columns within the block
    const bool colok = cl < vcols;        // V % 4 == 0: the four columns are valid together
    const size_t sbase = ((size_t)n * p.HV + hv) * (size_t)p.K * p.V + c_base + cl;

    // S2[i][j] = {S[d][j], S[d + 8][j]} with d = 16 i + rgrp.
    float2 S2[kLPairs][4];
#pragma unroll
    for (int i = 0; i < kLPairs; ++i) {
        float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
        const int d = 16 * i + rgrp;
        if (p.h0 && colok) {
            if (d < p.K) load4(p.h0 + sbase + (size_t)d * p.V, lo);
            if (d + 8 < p.K) load4(p.h0 + sbase + (size_t)(d + 8) * p.V, hi);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) S2[i][j] = make_float2(lo[j], hi[j]);
    }

    const int L = eos - bos;
    const int ngroups = (L + kLG - 1) / kLG;
    const T *beta = static_cast<const T *>(p.beta);
    T *o = static_cast<T *>(p.o);
    const bool gate_act = p.act.A_log != nullptr;
    const float neg_a = gate_act ? gate_neg_a(p.act, hv) : 0.f;
    auto fetch_beta = [&](int t0, int cnt) {
        float x = 0.f;
        if ((int)threadIdx.x < cnt) {
            const size_t row = (size_t)b * p.T + t0 + threadIdx.x;
            x = to_f32(beta[row * p.HV + hv]);
            if (p.act.beta_scale > 0.f) x = beta_activate<T>(x, p.act.beta_scale);
        }
        return x;
    };

    float2 a2[4], b2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) a2[j] = b2[j] = make_float2(0.f, 0.f);
    float bnext = 0.f;
    if (threadIdx.x == 0) sWide = 0;
    if (ngroups > 0) {
        long_issue<T>(p, smem + SM::raw, b, h, hv, c_base, vcols, bos, min(kLG + 1, L), min(kLG, L));
        cp_async_commit();
        bnext = fetch_beta(bos, min(kLG, L));
    }
    for (int gi = 0; gi < ngroups; ++gi) {
        const int t0 = bos + gi * kLG;
        const int ntok = min(kLG, eos - t0);
        const int nrows = min(kLG + 1, eos - t0);
        unsigned char *raw = smem + SM::raw + (gi & 1) * SM::raw_bytes;
        const T *rk = reinterpret_cast<const T *>(raw + SM::rk);
        const T *rq = reinterpret_cast<const T *>(raw + SM::rq);
        float *rg = reinterpret_cast<float *>(raw + SM::rg);
        const T *rv = reinterpret_cast<const T *>(raw + SM::rv);
        cp_async_wait_all();
        __syncthreads();  // this group's rows have landed; the previous group is computed

        if (warp >= 4) {
            // Token scalars: warp 4 + w takes tokens u = w, w + 4, ...; lane l rows l + 32 m.
            for (int u = warp - 4; u < ntok; u += 4) {
                float ks = 0.f, qs = 0.f, kq = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int d = lane + 32 * m;
                    if (d < p.K) {
                        const float kr = to_f32(rk[u * kLMaxK + d]);
                        const float qr = to_f32(rq[u * kLMaxK + d]);
                        ks = fmaf(kr, kr, ks);
                        qs = fmaf(qr, qr, qs);
                        kq = fmaf(kr, qr, kq);
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    ks += __shfl_xor_sync(0xffffffffu, ks, off);
                    qs += __shfl_xor_sync(0xffffffffu, qs, off);
                    kq += __shfl_xor_sync(0xffffffffu, kq, off);
                }
                if (lane == 0) {
                    const float rkn = p.l2norm ? 1.f / sqrtf(ks + 1e-6f) : 1.f;
                    const float rqn = p.l2norm ? 1.f / sqrtf(qs + 1e-6f) : 1.f;
                    scal[u * 4 + 0] = rkn;
                    scal[u * 4 + 1] = rqn;
                    scal[u * 4 + 2] = kq * rkn * rqn;
                }
            }
        } else {
            // Thread d runs down row d: x_u = g_scale g_u (activated when asked, kept
            // in place for the unscaled planes), G_u = x_0 + ... + x_u and D_u = 2^G_u.
            // Plane A gets {k_u / D_u (rows d, d + 8), D_{u+1} k_{u+1} (rows d, d + 8)},
            // plane B {D_{u+1} q_{u+1}}, the prologue D_0 {k_0, q_0}; D of the group's
            // last token is kept for the rescale after it.
            const int d = threadIdx.x;
            const int pi = 8 * (d >> 4) + (d & 7), hf = (d >> 3) & 1;
            float *c4 = reinterpret_cast<float *>(planeA);
            float *c2 = reinterpret_cast<float *>(planeB);
            float *pf = reinterpret_cast<float *>(pro);
            float G = 0.f, gmax = 0.f;
            for (int u = 0; u < nrows; ++u) {
                float kr = 0.f, qr = 0.f;
                if (d < p.K) {
                    float gr = rg[u * kLMaxK + d];
                    if (gate_act) gr = neg_a * softplus_f(gr + gate_bias(p.act, hv, d, p.K));
                    const float x = p.g_scale * gr;
                    rg[u * kLMaxK + d] = x;
                    G += x;
                    kr = to_f32(rk[u * kLMaxK + d]);
                    qr = to_f32(rq[u * kLMaxK + d]);
                }
                gmax = fmaxf(gmax, fabsf(G));
                const float Dp = exp2f(G);
                if (u < kLG) c4[(u * 64 + pi) * 4 + hf] = kr * exp2f(-G);
                if (u >= 1) {
                    c4[((u - 1) * 64 + pi) * 4 + 2 + hf] = kr * Dp;
                    c2[((u - 1) * 64 + pi) * 2 + hf] = qr * Dp;
                }
                if (u == 0) {
                    pf[pi * 4 + hf] = kr * Dp;
                    pf[pi * 4 + 2 + hf] = qr * Dp;
                }
                if (u == ntok - 1) sDlast[d] = Dp;
            }
            if (!(gmax <= kLWide)) sWide = 1;
        }
        __syncthreads();  // scaled planes, token scalars and the range flag ready
        const bool wide = sWide != 0;
        if (wide) {
            // The unscaled planes A = {2^x_u, k_u}, B = {2^x_{u+1} k_{u+1}, 2^x_{u+1} q_{u+1}}
            // (row pairs as above) over the scaled ones: warp w takes tokens w, w + 8, 16.
            for (int u = warp; u <= kLG; u += 8) {
                const bool valid = u < nrows;
#pragma unroll 1
                for (int m = 0; m < 2; ++m) {
                    const int pi = lane + 32 * m;
                    const int d0 = 16 * (pi >> 3) + (pi & 7);
                    float kr[2] = {0.f, 0.f}, qr[2] = {0.f, 0.f}, dec[2] = {0.f, 0.f};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int d = d0 + 8 * e;
                        if (valid && d < p.K) {
                            kr[e] = to_f32(rk[u * kLMaxK + d]);
                            qr[e] = to_f32(rq[u * kLMaxK + d]);
                            dec[e] = exp2f(rg[u * kLMaxK + d]);
                        }
                    }
                    if (u < kLG) planeA[u * 64 + pi] = make_float4(dec[0], dec[1], kr[0], kr[1]);
                    if (u >= 1)
                        planeB[(u - 1) * 64 + pi] =
                            make_float4(kr[0] * dec[0], kr[1] * dec[1], qr[0] * dec[0], qr[1] * dec[1]);
                }
            }
        }
        if ((int)threadIdx.x < kLG) scal[threadIdx.x * 4 + 3] = bnext;
        if (gi + 1 < ngroups) {
            const int t1 = t0 + kLG;
            long_issue<T>(p, smem + SM::raw + ((gi + 1) & 1) * SM::raw_bytes, b, h, hv, c_base, vcols,
                          t1, min(kLG + 1, eos - t1), min(kLG, eos - t1));
            cp_async_commit();
            bnext = fetch_beta(t1, min(kLG, eos - t1));
        }
        __syncthreads();  // planes ready
        if (threadIdx.x == 0) sWide = 0;  // every thread has read it

        if (gi == 0) {
#pragma unroll
            for (int i = 0; i < kLPairs; ++i) {
                const float4 e = pro[8 * i + rgrp];
                const float2 kd2 = make_float2(e.x, e.y), qd2 = make_float2(e.z, e.w);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    a2[j] = __ffma2_rn(S2[i][j], kd2, a2[j]);
                    b2[j] = __ffma2_rn(S2[i][j], qd2, b2[j]);
                }
            }
        }
        for (int u = 0; u < ntok; ++u) {
            float a[4], bq[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                a[j] = a2[j].x + a2[j].y;
                bq[j] = b2[j].x + b2[j].y;
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    a[j] += __shfl_xor_sync(0xffffffffu, a[j], off);
                    bq[j] += __shfl_xor_sync(0xffffffffu, bq[j], off);
                }
            }
            const float4 sc = reinterpret_cast<const float4 *>(scal)[u];
            float vv[4], ov[4];
            float2 dk2[4];
            load4(rv + u * 128 + cl, vv);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float delta = sc.w * (vv[j] - sc.x * a[j]);
                const float dk = sc.x * delta;
                dk2[j] = make_float2(dk, dk);
                ov[j] = p.scale * (sc.y * bq[j] + delta * sc.z);
                a2[j] = b2[j] = make_float2(0.f, 0.f);
            }
            if (rgrp == 0 && colok)
                store4(o + (((size_t)b * p.T + t0 + u) * p.HV + hv) * p.V + c_base + cl, ov);
            if (!wide) {
                // S~ += (k / D) dk^T; the reductions for the next token read S~ against D k', D q'
#pragma unroll
                for (int i = 0; i < kLPairs; ++i) {
                    const float4 e = planeA[u * 64 + 8 * i + rgrp];
                    const float2 f = reinterpret_cast<const float2 *>(planeB)[u * 64 + 8 * i + rgrp];
                    const float2 kt2 = make_float2(e.x, e.y), kd2 = make_float2(e.z, e.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        S2[i][j] = __ffma2_rn(kt2, dk2[j], S2[i][j]);
                        a2[j] = __ffma2_rn(S2[i][j], kd2, a2[j]);
                        b2[j] = __ffma2_rn(S2[i][j], f, b2[j]);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < kLPairs; ++i) {
                    const float4 ea = planeA[u * 64 + 8 * i + rgrp];
                    const float4 eb = planeB[u * 64 + 8 * i + rgrp];
                    const float2 dec2 = make_float2(ea.x, ea.y), k2 = make_float2(ea.z, ea.w);
                    const float2 kd2 = make_float2(eb.x, eb.y), qd2 = make_float2(eb.z, eb.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        S2[i][j] = __ffma2_rn(S2[i][j], dec2, __fmul2_rn(k2, dk2[j]));
                        a2[j] = __ffma2_rn(S2[i][j], kd2, a2[j]);
                        b2[j] = __ffma2_rn(S2[i][j], qd2, b2[j]);
                    }
                }
            }
        }
        if (!wide) {
            // back to the true state: S = D_last S~ per row
#pragma unroll
            for (int i = 0; i < kLPairs; ++i) {
                const float2 dl = make_float2(sDlast[16 * i + rgrp], sDlast[16 * i + rgrp + 8]);
#pragma unroll
                for (int j = 0; j < 4; ++j) S2[i][j] = __fmul2_rn(S2[i][j], dl);
            }
        }
    }

    if (p.ht && colok) {
#pragma unroll
        for (int i = 0; i < kLPairs; ++i) {
            const int d = 16 * i + rgrp;
            float lo[4], hi[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo[j] = S2[i][j].x;
                hi[j] = S2[i][j].y;
            }
            if (d < p.K) store4(p.ht + sbase + (size_t)d * p.V, lo);
            if (d + 8 < p.K) store4(p.ht + sbase + (size_t)(d + 8) * p.V, hi);
        }
    }
}

template <typename T>
bool long_form_fits(const RecurrentArgs &a) {
    auto al = [](const void *x) { return x == nullptr || ((uintptr_t)x % 16) == 0; };
    const int per = 16 / (int)sizeof(T);
    // slots average >= 8 tokens: below that the per-group staging does not pay
    return a.K <= kLMaxK && a.K % per == 0 && a.V % per == 0 && al(a.q) && al(a.k) && al(a.v) &&
           al(a.g) && al(a.o) && al(a.h0) && al(a.ht) && (int64_t)a.B * a.T >= 8LL * a.N;
}

template <typename T>
cudaError_t launch_long(const RecurrentArgs &a, cudaStream_t st) {
    static DeviceOnce once;
    const int smem = LongSmem<T>::total;
    int dev = 0;
    cudaError_t e = once.run(&dev, [&](int) {
        return cudaFuncSetAttribute(recurrent_long_kernel<T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.N * a.HV * ((a.V + 127) / 128);
    prof_begin("recurrent_long", st);
    recurrent_long_kernel<T><<<(unsigned)blocks, kLThreads, smem, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const RecurrentArgs &a, cudaStream_t st) {
    const int nwarps = (a.K + kRows - 1) / kRows;
    const int threads = nwarps * 32;
    const int nvb = (a.V + kBlockV - 1) / kBlockV;
    const int64_t blocks = (int64_t)a.N * a.HV * nvb;
    if (blocks == 0) return cudaSuccess;
    if (long_form_fits<T>(a)) return launch_long<T>(a, st);
    const size_t smem = sizeof(float) * 2 * nwarps * kRedStride;
    const bool vec = (a.V % 4 == 0) && (!a.h0 || ((uintptr_t)a.h0 % 16 == 0)) &&
                     (!a.ht || ((uintptr_t)a.ht % 16 == 0));
    prof_begin("recurrent", st);
    if (vec) {
        recurrent_kernel<T, true><<<(unsigned)blocks, threads, smem, st>>>(a);
    } else {
        recurrent_kernel<T, false><<<(unsigned)blocks, threads, smem, st>>>(a);
    }
    prof_end(st);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentArgs &a, kda_dtype dt, cudaStream_t st) {
    if (dt == KDA_DTYPE_BF16) return launch_typed<__nv_bfloat16>(a, st);
    return launch_typed<float>(a, st);
}

}  // namespace kda

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

template <typename T>
cudaError_t launch_typed(const RecurrentArgs &a, cudaStream_t st) {
    const int nwarps = (a.K + kRows - 1) / kRows;
    const int threads = nwarps * 32;
    const int nvb = (a.V + kBlockV - 1) / kBlockV;
    const int64_t blocks = (int64_t)a.N * a.HV * nvb;
    if (blocks == 0) return cudaSuccess;
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

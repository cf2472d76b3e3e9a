// kda_chunk_simt.cu -- chunked KDA forward in fp32 SIMT arithmetic.
//
// The path for fp32 inputs, whose 1e-4 tolerance rules out bf16/tf32 tensor-core
// operands.  It follows kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Forward":
//
//   prep (parallel over every (chunk, value head)):
//     Stage 1   g2 = chunk-local cumsum of g (fp32), G = g2 at the last valid row
//     Stage 2   Aqk[i,j] = scale sum_d q_i k_j 2^(g2_i - g2_j)   (i >= j)
//               L[i,j]   = beta_i sum_d k_i k_j 2^(g2_i - g2_j)  (i > j)
//               Akk = (I + L)^-1,  w = Akk (beta 2^g2 k),  u = Akk (beta v)
//               kg = k 2^(G - g2),  qg = scale q 2^g2,  decay = 2^G
//   scan (sequential over the chunks of one (sequence, value head, 32 columns)):
//     Stage 3+4 v' = u - w h,  o = qg h + Aqk v',  h = Diag(2^G) h + kg^T v'
//
// Every 2^(g2_i - g2_j) is evaluated directly with i >= j, so the exponent is
// never positive whatever the gate magnitude (ALGORITHM.md, "The numerics law").
// The intermediates go through the caller's workspace, fp32.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kScanBV = 32;

struct UnitLayout {  // float offsets inside one (chunk, value head) unit
    int64_t w, u, kg, qg, aqk, dec, stride;
};

__host__ __device__ inline UnitLayout unit_layout(int K, int V) {
    UnitLayout L;
    int64_t off = 0;
    L.w = off;   off += (int64_t)kBT * K;
    L.u = off;   off += (int64_t)kBT * V;
    L.kg = off;  off += (int64_t)kBT * K;
    L.qg = off;  off += (int64_t)kBT * K;
    L.aqk = off; off += (int64_t)kBT * kBT;
    L.dec = off; off += K;
    L.stride = (int64_t)align_up((size_t)off, 64);  // 256-byte units
    return L;
}

// Maps a chunk slot to its rows.  Returns false for slots past the last chunk
// or when the offsets failed validation.
__device__ __forceinline__ bool locate_chunk(const ChunkArgs &p, int64_t gc, int &b, int &r0,
                                             int &nr) {
    if (p.cu) {
        if (!p.ctrl->valid || gc >= p.ctrl->total_chunks) return false;
        const int n = upper_bound_minus_one(p.chunk_start, p.N + 1, (int)gc);
        const int c = (int)gc - p.chunk_start[n];
        b = 0;
        r0 = p.cu[n] + kBT * c;
        nr = min(kBT, p.cu[n + 1] - r0);
    } else {
        const int ntc = (p.T + kBT - 1) / kBT;
        b = (int)(gc / ntc);
        r0 = (int)(gc % ntc) * kBT;
        nr = min(kBT, p.T - r0);
    }
    return nr > 0;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <typename T, int KK>
__global__ void __launch_bounds__(kThreads) chunk_prep_kernel(ChunkArgs p) {
    extern __shared__ float sm[];
    float *sQ = sm;                    // [64][KK] q, later beta * 2^g2 * k
    float *sK = sQ + kBT * KK;         // [64][KK] k
    float *sG = sK + kBT * KK;         // [64][KK] g2
    float *sL = sG + kBT * KK;         // [64][64] L
    float *sA = sL + kBT * kBT;        // [64][64] Akk
    float *sB = sA + kBT * kBT;        // [64] beta
    float *sNq = sB + kBT;             // [64] q row scale
    float *sNk = sNq + kBT;            // [64] k row scale

    const int64_t gc = blockIdx.x;
    const int hv = blockIdx.y;
    int b, r0, nr;
    if (!locate_chunk(p, gc, b, r0, nr)) return;
    const int h = hv / (p.HV / p.H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const UnitLayout Lo = unit_layout(KK, p.V);
    float *U = static_cast<float *>(p.units) + (gc * p.HV + hv) * Lo.stride;
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    const T *beta = static_cast<const T *>(p.beta);
    const size_t row0 = (size_t)b * p.T + r0;

    for (int idx = tid; idx < kBT * KK; idx += kThreads) {
        const int i = idx / KK, d = idx % KK;
        const bool ok = i < nr;
        const size_t src = ((row0 + i) * p.H + h) * KK + d;
        sQ[idx] = ok ? to_f32(q[src]) : 0.f;
        sK[idx] = ok ? to_f32(k[src]) : 0.f;
    }
    if (tid < kBT) {
        float bv = tid < nr ? to_f32(beta[(row0 + tid) * p.HV + hv]) : 0.f;
        if (p.act.beta_scale > 0.f && tid < nr) bv = beta_activate<T>(bv, p.act.beta_scale);
        sB[tid] = bv;
    }
    const bool gate_act = p.act.A_log != nullptr;
    const float neg_a = gate_act ? gate_neg_a(p.act, hv) : 0.f;
    for (int d = tid; d < KK; d += kThreads) {  // Stage 1: chunk-local cumsum
        const float gbias = gate_act ? gate_bias(p.act, hv, d, KK) : 0.f;
        float acc = 0.f;
        for (int i = 0; i < nr; ++i) {
            float gv = p.g[((row0 + i) * p.HV + hv) * KK + d];
            if (gate_act) gv = neg_a * softplus_f(gv + gbias);
            acc = p.g_is_cumsum ? gv : acc + p.g_scale * gv;
            sG[i * KK + d] = acc;
        }
        for (int i = nr; i < kBT; ++i) sG[i * KK + d] = acc;  // padding rows hold G
    }
    __syncthreads();

    if (p.l2norm) {  // x / sqrt(sum x^2 + 1e-6) per row
        for (int i = warp; i < kBT; i += kThreads / 32) {
            float sq = 0.f, sk = 0.f;
            for (int d = lane; d < KK; d += 32) {
                sq += sQ[i * KK + d] * sQ[i * KK + d];
                sk += sK[i * KK + d] * sK[i * KK + d];
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            if (lane == 0) {
                sNq[i] = 1.f / sqrtf(sq + 1e-6f);
                sNk[i] = 1.f / sqrtf(sk + 1e-6f);
            }
        }
        __syncthreads();
        for (int idx = tid; idx < kBT * KK; idx += kThreads) {
            sQ[idx] *= sNq[idx / KK];
            sK[idx] *= sNk[idx / KK];
        }
        __syncthreads();
    }

    // Stage 2: gated grams.  One warp per row pair, lanes over channels.
    for (int i = warp; i < kBT; i += kThreads / 32) {
        for (int j = 0; j <= i; ++j) {
            float aq = 0.f, ak = 0.f;
            for (int d = lane; d < KK; d += 32) {
                const float e = exp2f(sG[i * KK + d] - sG[j * KK + d]);
                const float kj = sK[j * KK + d] * e;
                aq = fmaf(sQ[i * KK + d], kj, aq);
                ak = fmaf(sK[i * KK + d], kj, ak);
            }
            aq = warp_sum(aq);
            ak = warp_sum(ak);
            if (lane == 0) {
                U[Lo.aqk + i * kBT + j] = p.scale * aq;
                sL[i * kBT + j] = (i > j) ? sB[i] * ak : 0.f;
            }
        }
    }
    for (int idx = tid; idx < kBT * kBT; idx += kThreads) {
        const int i = idx / kBT, j = idx % kBT;
        if (j > i) {
            U[Lo.aqk + idx] = 0.f;
            sL[idx] = 0.f;
        }
        sA[idx] = (i == j) ? 1.f : 0.f;
    }
    __syncthreads();

    // qg, kg, decay; then sQ becomes beta * 2^g2 * k (the right operand of w).
    for (int idx = tid; idx < kBT * KK; idx += kThreads) {
        const int i = idx / KK, d = idx % KK;
        const float gi = sG[idx], G = sG[(kBT - 1) * KK + d];
        const float e = exp2f(gi);
        U[Lo.qg + idx] = p.scale * sQ[idx] * e;
        U[Lo.kg + idx] = sK[idx] * exp2f(G - gi);
        sQ[idx] = sB[i] * sK[idx] * e;
    }
    for (int d = tid; d < KK; d += kThreads) U[Lo.dec + d] = exp2f(sG[(kBT - 1) * KK + d]);

    // Akk = (I + L)^-1 by forward substitution, one row at a time.
    for (int i = 1; i < kBT; ++i) {
        __syncthreads();
        if (tid < i) {
            const int j = tid;
            float s = 0.f;
            for (int m = j; m < i; ++m) s = fmaf(sL[i * kBT + m], sA[m * kBT + j], s);
            sA[i * kBT + j] = -s;
        }
    }
    __syncthreads();

    // w = Akk (beta 2^g2 k),  u = Akk (beta v)
    for (int idx = tid; idx < kBT * KK; idx += kThreads) {
        const int i = idx / KK, d = idx % KK;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc = fmaf(sA[i * kBT + j], sQ[j * KK + d], acc);
        U[Lo.w + idx] = acc;
    }
    for (int idx = tid; idx < kBT * p.V; idx += kThreads) {
        const int i = idx / p.V, c = idx % p.V;
        float acc = 0.f;
        const int jmax = min(i, nr - 1);
        for (int j = 0; j <= jmax; ++j)
            acc = fmaf(sA[i * kBT + j] * sB[j], to_f32(v[((row0 + j) * p.HV + hv) * p.V + c]), acc);
        U[Lo.u + idx] = acc;
    }
}

template <typename T, int KK>
__global__ void __launch_bounds__(kThreads) chunk_scan_kernel(ChunkArgs p) {
    extern __shared__ float sm[];
    float *sH = sm;                    // [KK][BV]  state slice
    float *sW = sH + KK * kScanBV;     // [64][KK]
    float *sQG = sW + kBT * KK;        // [64][KK]
    float *sKG = sQG + kBT * KK;       // [64][KK]
    float *sAqk = sKG + kBT * KK;      // [64][64]
    float *sU = sAqk + kBT * kBT;      // [64][BV]
    float *sVp = sU + kBT * kScanBV;   // [64][BV]
    float *sDec = sVp + kBT * kScanBV; // [KK]

    const int nvb = (p.V + kScanBV - 1) / kScanBV;
    const int64_t bid = blockIdx.x;
    const int vb = (int)(bid % nvb);
    const int hv = (int)((bid / nvb) % p.HV);
    const int n = (int)(bid / ((int64_t)nvb * p.HV));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cb = vb * kScanBV;
    const int c = lane;
    const bool col_ok = cb + c < p.V;

    int b, bos, eos, nc;
    int64_t gc0;
    if (p.cu) {
        if (!p.ctrl->valid) return;
        b = 0;
        bos = p.cu[n];
        eos = p.cu[n + 1];
        nc = (eos - bos + kBT - 1) / kBT;
        gc0 = p.chunk_start[n];
    } else {
        b = n;
        bos = 0;
        eos = p.T;
        nc = (p.T + kBT - 1) / kBT;
        gc0 = (int64_t)n * nc;
    }
    const UnitLayout Lo = unit_layout(KK, p.V);
    const size_t sbase = ((size_t)n * p.HV + hv) * (size_t)KK * p.V;
    T *o = static_cast<T *>(p.o);

    for (int idx = tid; idx < KK * kScanBV; idx += kThreads) {
        const int d = idx / kScanBV, cc = idx % kScanBV;
        sH[idx] = (p.h0 && cb + cc < p.V) ? p.h0[sbase + (size_t)d * p.V + cb + cc] : 0.f;
    }

    for (int ci = 0; ci < nc; ++ci) {
        const float *U = static_cast<const float *>(p.units) + ((gc0 + ci) * p.HV + hv) * Lo.stride;
        const int r0 = bos + ci * kBT;
        const int nr = min(kBT, eos - r0);
        __syncthreads();
        for (int idx = tid; idx < kBT * KK; idx += kThreads) {
            sW[idx] = U[Lo.w + idx];
            sQG[idx] = U[Lo.qg + idx];
            sKG[idx] = U[Lo.kg + idx];
        }
        for (int idx = tid; idx < kBT * kBT; idx += kThreads) sAqk[idx] = U[Lo.aqk + idx];
        for (int idx = tid; idx < kBT * kScanBV; idx += kThreads) {
            const int i = idx / kScanBV, cc = idx % kScanBV;
            sU[idx] = (cb + cc < p.V) ? U[Lo.u + (int64_t)i * p.V + cb + cc] : 0.f;
        }
        for (int d = tid; d < KK; d += kThreads) sDec[d] = U[Lo.dec + d];
        __syncthreads();

        float oq[kBT / 8];
#pragma unroll
        for (int m = 0; m < kBT / 8; ++m) {
            const int i = warp + 8 * m;
            float wh = 0.f, qh = 0.f;
            for (int d = 0; d < KK; ++d) {
                const float hd = sH[d * kScanBV + c];
                wh = fmaf(sW[i * KK + d], hd, wh);
                qh = fmaf(sQG[i * KK + d], hd, qh);
            }
            sVp[i * kScanBV + c] = sU[i * kScanBV + c] - wh;
            oq[m] = qh;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kBT / 8; ++m) {
            const int i = warp + 8 * m;
            float acc = oq[m];
            for (int j = 0; j <= i; ++j) acc = fmaf(sAqk[i * kBT + j], sVp[j * kScanBV + c], acc);
            if (i < nr && col_ok)
                o[(((size_t)b * p.T + r0 + i) * p.HV + hv) * p.V + cb + c] = from_f32<T>(acc);
        }
        for (int d = warp; d < KK; d += 8) {
            float acc = sDec[d] * sH[d * kScanBV + c];
            for (int i = 0; i < kBT; ++i) acc = fmaf(sKG[i * KK + d], sVp[i * kScanBV + c], acc);
            sH[d * kScanBV + c] = acc;
        }
    }
    __syncthreads();
    if (p.ht) {
        for (int idx = tid; idx < KK * kScanBV; idx += kThreads) {
            const int d = idx / kScanBV, cc = idx % kScanBV;
            if (cb + cc < p.V) p.ht[sbase + (size_t)d * p.V + cb + cc] = sH[idx];
        }
    }
}

template <typename T, int KK>
cudaError_t launch_kk(const ChunkArgs &a, cudaStream_t st) {
    const size_t prep_smem = sizeof(float) * (3 * kBT * KK + 2 * kBT * kBT + 3 * kBT);
    const size_t scan_smem = sizeof(float) * (KK * kScanBV + 3 * kBT * KK + kBT * kBT +
                                              2 * kBT * kScanBV + KK);
    cudaError_t e;
    static DeviceOnce once;
    int dev = 0;
    e = once.run(&dev, [&](int) {
        cudaError_t r = cudaFuncSetAttribute(chunk_prep_kernel<T, KK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(chunk_scan_kernel<T, KK>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem);
        return r;
    });
    if (e != cudaSuccess) return e;
    if (a.slots > 0) {
        dim3 grid((unsigned)a.slots, a.HV);
        prof_begin("chunk_prep_simt", st);
        chunk_prep_kernel<T, KK><<<grid, kThreads, prep_smem, st>>>(a);
        prof_end(st);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int nvb = (a.V + kScanBV - 1) / kScanBV;
    const int64_t blocks = (int64_t)a.N * a.HV * nvb;
    if (blocks > 0) {
        prof_begin("chunk_scan_simt", st);
        chunk_scan_kernel<T, KK><<<(unsigned)blocks, kThreads, scan_smem, st>>>(a);
        prof_end(st);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_typed(const ChunkArgs &a, cudaStream_t st) {
    if (a.K == 64) return launch_kk<T, 64>(a, st);
    return launch_kk<T, 128>(a, st);
}

}  // namespace

size_t chunk_simt_unit_bytes(int K, int V) { return sizeof(float) * unit_layout(K, V).stride; }

cudaError_t launch_chunk_simt(const ChunkArgs &a, kda_dtype dt, cudaStream_t st) {
    if (dt == KDA_DTYPE_BF16) return launch_typed<__nv_bfloat16>(a, st);
    return launch_typed<float>(a, st);
}

}  // namespace kda

// kda_chunk_tc.cu -- chunked KDA forward for bf16 inputs on the sm_103a tensor
// cores (tcgen05.mma, accumulators in tensor memory, bulk async copies).
//
// kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Forward", per value head and per
// chunk of BT = 64 rows with g2 the chunk-local cumsum (log2) and G its last row:
//
//   prep kernel, one CTA per (chunk, value head), all in parallel:
//     Stage 1     g2, G (fp32, per channel)
//     Stage 2     Aqk = scale * tril(Qg Kb^T),  L = diag(beta) * strictly_tril(Kg Kb^T)
//                 with Qg = q 2^g2, Kg = k 2^g2, Kb = k 2^-g2: the per-channel gate
//                 2^(g2_i - g2_j) split through the chunk start, one tcgen05 MMA
//                 (M = 128: [Qg; Kg] stacked, N = 64, K = dk).  This split keeps
//                 every factor at most 2^R with R = max |g2| over the chunk; when R
//                 exceeds kSafeRange the grams are formed exactly in fp32 SIMT with
//                 one exp2 per (i, j, d), exponent g2_i - g2_j <= 0 (ALGORITHM.md,
//                 "The numerics law").
//                 Akk = (I + L)^-1: blocked unit-lower-triangular inverse in fp32
//                 (16 x 16 diagonal blocks by substitution, off-diagonal blocks
//                 level by level).
//                 w = Akk diag(beta) Kg,  u = Akk diag(beta) v    (tcgen05, N = dk / dv)
//                 kg = k 2^(G - g2),  qg = scale q 2^g2,  decay = 2^G
//     The results go to the workspace as ready-made MMA operand tiles.
//
//   scan kernel, one CTA per (sequence, value head, 32 value columns):
//     Stage 3+4   v' = u - w h;   o = qg h + Aqk v';   h = Diag(2^G) h + kg^T v'
//                 [w; qg] h    : one MMA, M = 128, N = 32, K = dk
//                 kg^T v'      : one MMA, M = 128 (= dk, zero-padded for dk = 64)
//                 Aqk v'       : accumulated onto the qg h rows of the first MMA
//     h stays in registers in fp32 (thread d owns row d); a bf16 copy in shared
//     memory is the next chunk's MMA operand.  Operand tiles of the next chunks
//     stream in by bulk async copies while the current chunk computes.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kBV = 32;               // value columns per scan CTA
constexpr int kStages = 3;            // scan pipeline depth
constexpr float kSafeRange = 60.f;    // max |g2| (log2) for the split grams
constexpr uint64_t kWaitNs = 1000000000ull;

// Byte layout of one workspace unit (chunk, value head).
struct TcLayout {
    uint32_t aw;      // [128][dk] tile: rows 0..63 w, rows 64..127 scale * qg
    uint32_t kgt;     // [128][64] tile: kg^T (rows >= dk zero)
    uint32_t aqk;     // [64][64] tile: Aqk (scale inside)
    uint32_t u;       // [dv / 32][64][32] bf16 row-major blocks
    uint32_t dec;     // [128] fp32: 2^G (0 beyond dk)
    uint32_t stride;  // unit size, 256-byte multiple
    uint32_t head;    // bytes of aw + kgt + aqk (one contiguous copy)
};

__host__ __device__ inline TcLayout tc_layout(int K, int V) {
    TcLayout L;
    uint32_t off = 0;
    L.aw = off;  off += 128u * K * 2;
    L.kgt = off; off += 128u * 64 * 2;
    L.aqk = off; off += 64u * 64 * 2;
    L.head = off;
    L.u = off;   off += 64u * V * 2;
    L.dec = off; off += 128u * 4;
    L.stride = (uint32_t)align_up(off, 256);
    return L;
}

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

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
}
__device__ __forceinline__ uint4 pack8_at(const float *f) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
}

// ============================================================== prep kernel
template <int KK, int VV>
struct PrepSmem {
    static constexpr int kGStride = KK + 4;                       // padded fp32 row of g2
    static constexpr uint32_t ag = 0;                             // [128][KK] bf16 tile
    static constexpr uint32_t kb = ag + 128 * KK * 2;             // [64][KK] tile / scratch
    static constexpr uint32_t kb_bytes = (64 * KK * 2 > 16384) ? 64 * KK * 2 : 16384;
    static constexpr uint32_t ab = kb + kb_bytes;                 // [64][64] tile Akk diag(beta)
    static constexpr uint32_t v = ab + 64 * 64 * 2;               // [64][VV] tile
    static constexpr uint32_t g = v + 64 * VV * 2;                // g2 fp32, later L and Akk
    static constexpr uint32_t g_bytes0 = 64 * kGStride * 4;
    static constexpr uint32_t g_bytes = g_bytes0 > 2 * 64 * 65 * 4 ? g_bytes0 : 2 * 64 * 65 * 4;
    static constexpr uint32_t used = g + g_bytes;
    // Floor so that at most two CTAs (256 TMEM columns each) or one (512) share an SM.
    static constexpr uint32_t floor_bytes = (KK + VV <= 256) ? 80 * 1024 : 120 * 1024;
    static constexpr uint32_t total = used > floor_bytes ? used : floor_bytes;
};
constexpr int kLS = 65;  // padded row stride of L and Akk (fp32)

template <int KK, int VV>
__global__ void __launch_bounds__(128) chunk_prep_tc_kernel(ChunkArgs p) {
    using S = PrepSmem<KK, VV>;
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ float sBeta[64];
    __shared__ float sGlast[128];
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    __shared__ float sRange;

    const int64_t gc = blockIdx.x;
    const int hv = blockIdx.y;
    int b, r0, nr;
    if (!locate_chunk(p, gc, b, r0, nr)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = hv / (p.HV / p.H);
    constexpr uint32_t kTmemCols = (KK + VV <= 256) ? 256 : 512;

    unsigned char *sAG = sm + S::ag;
    unsigned char *sKB = sm + S::kb;
    unsigned char *sAB = sm + S::ab;
    unsigned char *sV = sm + S::v;
    float *sG = reinterpret_cast<float *>(sm + S::g);
    float *sL = sG;                 // after the elementwise phase: L [64][kLS]
    float *sA = sG + 64 * kLS;      //                             Akk [64][kLS]
    float *sT = reinterpret_cast<float *>(sKB);  // solve scratch (after the grams)

    const TcLayout Lo = tc_layout(KK, VV);
    unsigned char *U = static_cast<unsigned char *>(p.units) + (gc * p.HV + hv) * Lo.stride;

    if (warp == 0) {
        tmem_alloc(&tslot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }

    // ---- 1. inputs -> shared memory (q, k, v as operand tiles; g row-major)
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(p.beta);
    const size_t row0 = (size_t)b * p.T + r0;
    constexpr int KG8 = KK / 8, VG8 = VV / 8, KG4 = KK / 4;
    for (int idx = tid; idx < 64 * KG8; idx += 128) {
        const int i = idx / KG8, c = (idx % KG8) * 8;
        void *dq = sAG + tile_off(i, c, KK);
        void *dk = sAG + tile_off(64 + i, c, KK);
        if (i < nr) {
            const size_t src = ((row0 + i) * p.H + h) * KK + c;
            cp_async16(dq, q + src);
            cp_async16(dk, k + src);
        } else {
            *reinterpret_cast<uint4 *>(dq) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(dk) = make_uint4(0, 0, 0, 0);
        }
    }
    for (int idx = tid; idx < 64 * VG8; idx += 128) {
        const int i = idx / VG8, c = (idx % VG8) * 8;
        void *dv = sV + tile_off(i, c, VV);
        if (i < nr)
            cp_async16(dv, v + ((row0 + i) * p.HV + hv) * VV + c);
        else
            *reinterpret_cast<uint4 *>(dv) = make_uint4(0, 0, 0, 0);
    }
    for (int idx = tid; idx < 64 * KG4; idx += 128) {
        const int i = idx / KG4, c = (idx % KG4) * 4;
        float *dg = sG + i * S::kGStride + c;
        if (i < nr)
            cp_async16(dg, p.g + ((row0 + i) * p.HV + hv) * KK + c);
        else
            *reinterpret_cast<float4 *>(dg) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < 64) sBeta[tid] = tid < nr ? to_f32(beta[(row0 + tid) * p.HV + hv]) : 0.f;
    cp_async_wait_all();
    __syncthreads();

    // ---- optional L2 normalisation of the q and k rows (thread r: row r of [q; k])
    if (p.l2norm) {
        float ss = 0.f;
        for (int c = 0; c < KK; c += 8) {
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(sAG + tile_off(tid, c, KK)), f);
#pragma unroll
            for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
        }
        const float rs = 1.f / sqrtf(ss + 1e-6f);
        for (int c = 0; c < KK; c += 8) {
            uint4 *ptr = reinterpret_cast<uint4 *>(sAG + tile_off(tid, c, KK));
            float f[8];
            unpack8(*ptr, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] *= rs;
            *ptr = pack8(f);
        }
    }

    // ---- 2. Stage 1: chunk-local cumsum, thread d owns channel d
    {
        float rng = 0.f;
        if (tid < KK) {
            float acc = 0.f;
            for (int i = 0; i < nr; ++i) {
                const float gv = sG[i * S::kGStride + tid];
                acc = p.g_is_cumsum ? gv : fmaf(p.g_scale, gv, acc);
                sG[i * S::kGStride + tid] = acc;
                rng = fmaxf(rng, fabsf(acc));
            }
            for (int i = nr; i < 64; ++i) sG[i * S::kGStride + tid] = acc;
            sGlast[tid] = acc;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) rng = fmaxf(rng, __shfl_xor_sync(0xffffffffu, rng, off));
        if (tid == 0) sRange = 0.f;
        __syncthreads();
        if (lane == 0) atomicMax(reinterpret_cast<int *>(&sRange), __float_as_int(rng));
        __syncthreads();
    }
    const bool fast = sRange <= kSafeRange;
    uint32_t phase = 0;  // completed phases of `bar`

    // ---- exact grams for chunks whose gate range is too wide to split
    if (!fast) {
        float *sLx = reinterpret_cast<float *>(sKB);  // [64][64] fp32 L (16 KB)
        for (int i = warp; i < 64; i += 4) {
            for (int j = 0; j <= i; ++j) {
                float aq = 0.f, ak = 0.f;
                for (int d = lane; d < KK; d += 32) {
                    const float e = exp2f(sG[i * S::kGStride + d] - sG[j * S::kGStride + d]);
                    const float qi = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                        sAG + tile_off(i, d, KK)));
                    const float ki = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                        sAG + tile_off(64 + i, d, KK)));
                    const float kj = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                        sAG + tile_off(64 + j, d, KK))) * e;
                    aq = fmaf(qi, kj, aq);
                    ak = fmaf(ki, kj, ak);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    aq += __shfl_xor_sync(0xffffffffu, aq, off);
                    ak += __shfl_xor_sync(0xffffffffu, ak, off);
                }
                if (lane == 0) {
                    *reinterpret_cast<__nv_bfloat16 *>(U + Lo.aqk + tile_off(i, j, 64)) =
                        __float2bfloat16_rn(p.scale * aq);
                    sLx[i * 64 + j] = (i > j) ? sBeta[i] * ak : 0.f;
                }
            }
            for (int j = i + 1 + lane; j < 64; j += 32) {
                *reinterpret_cast<__nv_bfloat16 *>(U + Lo.aqk + tile_off(i, j, 64)) =
                    __float2bfloat16_rn(0.f);
                sLx[i * 64 + j] = 0.f;
            }
        }
    }
    __syncthreads();

    // ---- 3. elementwise: qg, kg (in place), kb, scale*qg -> workspace, kg^T -> workspace
    // idx -> (row i = idx % 64, 8-column group): a warp covers 32 rows of one group.
    for (int idx = tid; idx < 64 * KG8; idx += 128) {
        const int i = idx & 63, c = (idx >> 6) * 8;
        uint4 *pq = reinterpret_cast<uint4 *>(sAG + tile_off(i, c, KK));
        uint4 *pk = reinterpret_cast<uint4 *>(sAG + tile_off(64 + i, c, KK));
        float fq[8], fk[8], qg[8], kgm[8], kb[8], kg[8], qs[8];
        unpack8(*pq, fq);
        unpack8(*pk, fk);
        const float *gr = sG + i * S::kGStride + c;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float gam = gr[j];
            const float e = exp2f(gam);
            qg[j] = fq[j] * e;
            kgm[j] = fk[j] * e;
            kb[j] = fast ? fk[j] * exp2f(-gam) : 0.f;
            kg[j] = fk[j] * exp2f(sGlast[c + j] - gam);
            qs[j] = p.scale * qg[j];
        }
        *pq = pack8(qg);
        *pk = pack8(kgm);
        if (fast) *reinterpret_cast<uint4 *>(sKB + tile_off(i, c, KK)) = pack8(kb);
        *reinterpret_cast<uint4 *>(U + Lo.aw + tile_off(64 + i, c, KK)) = pack8(qs);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<__nv_bfloat16 *>(U + Lo.kgt + tile_off(c + j, i, 64)) =
                __float2bfloat16_rn(kg[j]);
    }
    if (KK < 128) {  // zero rows dk..127 of kg^T
        for (int idx = tid; idx < (128 - KK) * 8; idx += 128) {
            const int d = KK + idx / 8, c = (idx % 8) * 8;
            *reinterpret_cast<uint4 *>(U + Lo.kgt + tile_off(d, c, 64)) = make_uint4(0, 0, 0, 0);
        }
    }
    reinterpret_cast<float *>(U + Lo.dec)[tid] = tid < KK ? exp2f(sGlast[tid]) : 0.f;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;

    // ---- 4. grams on the tensor cores: D[0:128, 0:64] = [Qg; Kg] Kb^T
    if (fast) {
        if (tid == 0) {
            mma_bf16_k(tmem, smem_addr(sAG), 128, KK * 16, smem_addr(sKB), 128, KK * 16,
                       idesc_bf16(128, 64, false, false), KK / 16, 0);
            mma_commit(&bar);
        }
        __syncwarp();
        if (!mbar_wait(&bar, phase & 1, kWaitNs) && tid == 0) report(p.status, KDA_DEVICE_TIMEOUT);
        ++phase;
        tc_fence_after();
        float d[16];
        const int i = tid & 63;
        for (int c0 = 0; c0 < 64; c0 += 16) {
            tmem_ld16(tmem_at(tmem, warp * 32, c0), d);
            if (tid < 64) {  // Aqk row i
                float a[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) a[j] = (c0 + j <= i) ? p.scale * d[j] : 0.f;
                *reinterpret_cast<uint4 *>(U + Lo.aqk + tile_off(i, c0, 64)) = pack8_at(a);
                *reinterpret_cast<uint4 *>(U + Lo.aqk + tile_off(i, c0 + 8, 64)) = pack8_at(a + 8);
            } else {  // L row i
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    sL[i * kLS + c0 + j] = (c0 + j < i) ? sBeta[i] * d[j] : 0.f;
            }
        }
        tc_fence_before();
    } else {
        const float *sLx = reinterpret_cast<const float *>(sKB);
        for (int idx = tid; idx < 64 * 64; idx += 128) sL[(idx >> 6) * kLS + (idx & 63)] = sLx[idx];
    }
    __syncthreads();

    // ---- 5. Akk = (I + L)^-1
    for (int idx = tid; idx < 64 * 64; idx += 128) sA[(idx >> 6) * kLS + (idx & 63)] = 0.f;
    __syncthreads();
    if (tid < 64) {  // diagonal 16 x 16 blocks, one column per thread
        const int I = tid >> 4, c = tid & 15, o = 16 * I;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) s = fmaf(sL[(o + r) * kLS + o + m], x[m], s);
            if (r > c) x[r] = -s;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sA[(o + r) * kLS + o + c] = x[r];
    }
    __syncthreads();
    for (int lvl = 1; lvl < 4; ++lvl) {
        const int nblk = 4 - lvl;
        // T_IJ = sum_{M=J}^{I-1} L_IM A_MJ   for I = J + lvl
        for (int e = tid; e < nblk * 256; e += 128) {
            const int J = e >> 8, I = J + lvl, r = (e >> 4) & 15, c = e & 15;
            float s = 0.f;
            for (int M = J; M < I; ++M) {
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    s = fmaf(sL[(16 * I + r) * kLS + 16 * M + m], sA[(16 * M + m) * kLS + 16 * J + c], s);
            }
            sT[e] = s;
        }
        __syncthreads();
        // A_IJ = -A_II T_IJ
        for (int e = tid; e < nblk * 256; e += 128) {
            const int J = e >> 8, I = J + lvl, r = (e >> 4) & 15, c = e & 15;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                s = fmaf(sA[(16 * I + r) * kLS + 16 * I + m], sT[(J << 8) + m * 16 + c], s);
            sA[(16 * I + r) * kLS + 16 * J + c] = -s;
        }
        __syncthreads();
    }
    // Akk diag(beta) as a bf16 operand tile
    for (int idx = tid; idx < 64 * 8; idx += 128) {
        const int i = idx >> 3, c = (idx & 7) * 8;
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = sA[i * kLS + c + j] * sBeta[c + j];
        *reinterpret_cast<uint4 *>(sAB + tile_off(i, c, 64)) = pack8(f);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 6. w = Akk diag(beta) Kg,  u = Akk diag(beta) v  (valid rows: TMEM lanes 64..127)
    if (tid == 0) {
        const uint32_t a = smem_addr(sAB) - 8 * 1024;  // rows 64..127 of the M = 128 operand
        mma_bf16_k(tmem, a, 128, 1024, smem_addr(sAG) + 64 * KK * 2, KK * 16, 128,
                   idesc_bf16(128, KK, false, true), 4, 0);
        mma_bf16_k(tmem + KK, a, 128, 1024, smem_addr(sV), VV * 16, 128,
                   idesc_bf16(128, VV, false, true), 4, 0);
        mma_commit(&bar);
    }
    __syncwarp();
    if (!mbar_wait(&bar, phase & 1, kWaitNs) && tid == 0) report(p.status, KDA_DEVICE_TIMEOUT);
    tc_fence_after();
    if (warp >= 2) {
        const int i = tid - 64;
        float d[16];
        for (int c0 = 0; c0 < KK; c0 += 16) {
            tmem_ld16(tmem_at(tmem, warp * 32, c0), d);
            *reinterpret_cast<uint4 *>(U + Lo.aw + tile_off(i, c0, KK)) = pack8_at(d);
            *reinterpret_cast<uint4 *>(U + Lo.aw + tile_off(i, c0 + 8, KK)) = pack8_at(d + 8);
        }
        for (int c0 = 0; c0 < VV; c0 += 16) {
            tmem_ld16(tmem_at(tmem, warp * 32, KK + c0), d);
            unsigned char *ub = U + Lo.u + (size_t)(c0 / kBV) * 64 * kBV * 2 +
                                ((size_t)i * kBV + (c0 % kBV)) * 2;
            *reinterpret_cast<uint4 *>(ub) = pack8_at(d);
            *reinterpret_cast<uint4 *>(ub + 16) = pack8_at(d + 8);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ============================================================== scan kernel
template <int KK>
struct ScanSmem {
    static constexpr uint32_t head = 128 * KK * 2 + 128 * 64 * 2 + 64 * 64 * 2;
    static constexpr uint32_t stage = head + 64 * kBV * 2 + 128 * 4;
    static constexpr uint32_t stage_stride = (stage + 1023) / 1024 * 1024;
    static constexpr uint32_t hs = kStages * stage_stride;   // [KK][kBV] bf16 tile
    static constexpr uint32_t vp = hs + KK * kBV * 2;        // [64][kBV] bf16 tile
    static constexpr uint32_t total = vp + 64 * kBV * 2;
};

__device__ __forceinline__ int read_flag(const int *f) { return *reinterpret_cast<const volatile int *>(f); }

template <int KK>
__global__ void __launch_bounds__(160) chunk_scan_tc_kernel(ChunkArgs p) {
    using S = ScanSmem<KK>;
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint64_t full[kStages], empty[kStages];
    __shared__ uint64_t bar_d1[2], bar_d2, bar_d3[2], h_ready, vp_ready;
    __shared__ uint32_t tslot;
    __shared__ int abort_flag;

    const int nvb = p.V / kBV;
    const int64_t bid = blockIdx.x;
    const int vb = (int)(bid % nvb);
    const int hv = (int)((bid / nvb) % p.HV);
    const int n = (int)(bid / ((int64_t)nvb * p.HV));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

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
    const TcLayout Lo = tc_layout(KK, p.V);
    const size_t sbase = ((size_t)n * p.HV + hv) * (size_t)KK * p.V + (size_t)vb * kBV;

    if (warp == 0) {
        tmem_alloc(&tslot, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&bar_d1[0], 1);
        mbar_init(&bar_d1[1], 1);
        mbar_init(&bar_d2, 1);
        mbar_init(&bar_d3[0], 1);
        mbar_init(&bar_d3[1], 1);
        mbar_init(&h_ready, 128);
        mbar_init(&vp_ready, 64);
        mbar_fence_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    // columns: D1 double buffer at 0 / kBV, D2 at 2 kBV
    unsigned char *sH = sm + S::hs;
    unsigned char *sVp = sm + S::vp;
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);

    if (warp == 4) {
        // ------------------------------------------------ producer: bulk loads
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nc; ++c) {
                const int s = c % kStages;
                if (c >= kStages && !mbar_wait(&empty[s], ((c / kStages) - 1) & 1, kWaitNs)) {
                    atomicExch(&abort_flag, 1);
                    report(p.status, KDA_DEVICE_TIMEOUT);
                    break;
                }
                if (read_flag(&abort_flag)) break;
                issued = c + 1;
                const unsigned char *U =
                    static_cast<const unsigned char *>(p.units) + ((gc0 + c) * p.HV + hv) * Lo.stride;
                unsigned char *st = sm + s * S::stage_stride;
                const uint32_t ubytes = 64 * kBV * 2;
                mbar_arrive_expect_tx(&full[s], S::head + ubytes + 512);
                for (uint32_t off = 0; off < S::head; off += 16384) {
                    const uint32_t len = S::head - off < 16384 ? S::head - off : 16384;
                    bulk_g2s(st + off, U + off, len, &full[s]);
                }
                bulk_g2s(st + S::head, U + Lo.u + (size_t)vb * ubytes, ubytes, &full[s]);
                bulk_g2s(st + S::head + ubytes, U + Lo.dec, 512, &full[s]);
            }
            // Copies still in flight must land before the CTA exits (bounded).
            for (int c = issued - kStages > 0 ? issued - kStages : 0; c < issued; ++c)
                mbar_wait(&full[c % kStages], (c / kStages) & 1, kWaitNs);
        }
    } else {
        // ------------------------------------- epilogue warps 0..3 (+ MMA issue by tid 0)
        const int r = tid;  // TMEM lane / state row d / chunk row
        float hreg[kBV];
        const bool has_row = r < KK;
#pragma unroll
        for (int j = 0; j < kBV; ++j) hreg[j] = 0.f;
        if (has_row && p.h0) {
            const float4 *src = reinterpret_cast<const float4 *>(p.h0 + sbase + (size_t)r * p.V);
#pragma unroll
            for (int j = 0; j < kBV / 4; ++j) {
                const float4 x = src[j];
                hreg[4 * j] = x.x; hreg[4 * j + 1] = x.y; hreg[4 * j + 2] = x.z; hreg[4 * j + 3] = x.w;
            }
        }
        auto write_h = [&]() {
            if (has_row) {
#pragma unroll
                for (int j = 0; j < kBV; j += 8)
                    *reinterpret_cast<uint4 *>(sH + tile_off(r, j, kBV)) = pack8_at(hreg + j);
            }
            fence_async_smem();
            mbar_arrive(&h_ready);
        };
        write_h();

        const uint32_t id_m1 = idesc_bf16(128, kBV, false, true);
        for (int c = 0; c < nc; ++c) {
            const int s = c % kStages;
            const uint32_t fpar = (c / kStages) & 1;
            const unsigned char *st = sm + s * S::stage_stride;
            const uint32_t d1 = tmem + (c & 1) * kBV, d2 = tmem + 2 * kBV;
            bool ok = true;
            if (tid == 0) {
                // MMA issue for chunk c: [w; qg] h  ->  D1[c % 2]
                ok = mbar_wait(&full[s], fpar, kWaitNs) && mbar_wait(&h_ready, c & 1, kWaitNs);
                if (ok) {
                    tc_fence_after();
                    mma_bf16_k(d1, smem_addr(st), 128, KK * 16, smem_addr(sH), kBV * 16, 128,
                               id_m1, KK / 16, 0);
                    mma_commit(&bar_d1[c & 1]);
                    if (c >= 1) mma_commit(&empty[(c - 1) % kStages]);
                } else {
                    atomicExch(&abort_flag, 1);
                    report(p.status, KDA_DEVICE_TIMEOUT);
                }
            }
            __syncwarp();
            // all epilogue threads need the stage (u rows and decay)
            if (!mbar_wait(&full[s], fpar, kWaitNs)) { atomicExch(&abort_flag, 1); }
            const float dec = has_row ? reinterpret_cast<const float *>(st + S::head + 64 * kBV * 2)[r] : 0.f;
            if (warp < 2) {
                // v' = u - w h for chunk row r
                float uu[kBV];
                const unsigned char *ur = st + S::head + (size_t)r * kBV * 2;
#pragma unroll
                for (int j = 0; j < kBV; j += 8) {
                    float f[8];
                    unpack8(*reinterpret_cast<const uint4 *>(ur + j * 2), f);
#pragma unroll
                    for (int t = 0; t < 8; ++t) uu[j + t] = f[t];
                }
                if (!mbar_wait(&bar_d1[c & 1], (c >> 1) & 1, kWaitNs)) atomicExch(&abort_flag, 1);
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < kBV; j += 16) {
                    float d[16];
                    tmem_ld16(tmem_at(d1, warp * 32, j), d);
#pragma unroll
                    for (int t = 0; t < 16; ++t) uu[j + t] -= d[t];
                }
#pragma unroll
                for (int j = 0; j < kBV; j += 8)
                    *reinterpret_cast<uint4 *>(sVp + tile_off(r, j, kBV)) = pack8_at(uu + j);
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(&vp_ready);
            }
            if (tid == 0 && ok) {
                // kg^T v' -> D2 ;  Aqk v' accumulated onto rows 64..127 of D1[c % 2]
                ok = mbar_wait(&vp_ready, c & 1, kWaitNs);
                if (ok) {
                    tc_fence_after();
                    mma_bf16_k(d2, smem_addr(st + 128 * KK * 2), 128, 1024, smem_addr(sVp),
                               kBV * 16, 128, id_m1, 4, 0);
                    mma_commit(&bar_d2);
                    mma_bf16_k(d1, smem_addr(st + 128 * KK * 2 + 128 * 64 * 2) - 8 * 1024, 128,
                               1024, smem_addr(sVp), kBV * 16, 128, id_m1, 4, 1);
                    mma_commit(&bar_d3[c & 1]);
                } else {
                    atomicExch(&abort_flag, 1);
                    report(p.status, KDA_DEVICE_TIMEOUT);
                }
            }
            __syncwarp();
            // h = Diag(2^G) h + kg^T v'
            if (!mbar_wait(&bar_d2, c & 1, kWaitNs)) atomicExch(&abort_flag, 1);
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < kBV; j += 16) {
                float d[16];
                tmem_ld16(tmem_at(d2, warp * 32, j), d);
#pragma unroll
                for (int t = 0; t < 16; ++t) hreg[j + t] = fmaf(dec, hreg[j + t], d[t]);
            }
            tc_fence_before();
            if (warp >= 2) {
                // o rows (chunk row r - 64): qg h + Aqk v' from D1[c % 2]
                if (!mbar_wait(&bar_d3[c & 1], (c >> 1) & 1, kWaitNs)) atomicExch(&abort_flag, 1);
                tc_fence_after();
                const int i = r - 64;
                const int row = bos + c * kBT + i;
                const bool store = row < eos && !read_flag(&abort_flag);
                __nv_bfloat16 *orow = o + (((size_t)b * p.T + row) * p.HV + hv) * p.V + vb * kBV;
#pragma unroll
                for (int j = 0; j < kBV; j += 16) {
                    float d[16];
                    tmem_ld16(tmem_at(d1, warp * 32, j), d);
                    if (store) {
                        *reinterpret_cast<uint4 *>(orow + j) = pack8_at(d);
                        *reinterpret_cast<uint4 *>(orow + j + 8) = pack8_at(d + 8);
                    }
                }
                tc_fence_before();
            }
            if (c + 1 < nc) write_h();
            if (read_flag(&abort_flag)) break;
        }
        if (p.ht && has_row && !read_flag(&abort_flag)) {
            float4 *dst = reinterpret_cast<float4 *>(p.ht + sbase + (size_t)r * p.V);
#pragma unroll
            for (int j = 0; j < kBV / 4; ++j)
                dst[j] = make_float4(hreg[4 * j], hreg[4 * j + 1], hreg[4 * j + 2], hreg[4 * j + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

template <int KK, int VV>
cudaError_t launch_prep(const ChunkArgs &a, cudaStream_t st) {
    using S = PrepSmem<KK, VV>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(chunk_prep_tc_kernel<KK, VV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::total);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid((unsigned)a.slots, a.HV);
    prof_begin("chunk_prep_tc", st);
    chunk_prep_tc_kernel<KK, VV><<<grid, 128, S::total, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

template <int KK>
cudaError_t launch_scan(const ChunkArgs &a, cudaStream_t st) {
    using S = ScanSmem<KK>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(chunk_scan_tc_kernel<KK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::total);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int64_t blocks = (int64_t)a.N * a.HV * (a.V / kBV);
    if (blocks == 0) return cudaSuccess;
    prof_begin("chunk_scan_tc", st);
    chunk_scan_tc_kernel<KK><<<(unsigned)blocks, 160, S::total, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

template <int KK>
cudaError_t launch_k(const ChunkArgs &a, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (a.slots > 0) {
        switch (a.V) {
            case 32: e = launch_prep<KK, 32>(a, st); break;
            case 64: e = launch_prep<KK, 64>(a, st); break;
            case 96: e = launch_prep<KK, 96>(a, st); break;
            case 128: e = launch_prep<KK, 128>(a, st); break;
            case 160: e = launch_prep<KK, 160>(a, st); break;
            case 192: e = launch_prep<KK, 192>(a, st); break;
            case 224: e = launch_prep<KK, 224>(a, st); break;
            case 256: e = launch_prep<KK, 256>(a, st); break;
            default: return cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
    }
    return launch_scan<KK>(a, st);
}

}  // namespace

bool chunk_tc_supported(int K, int V) {
    return (K == 64 || K == 128) && V >= kBV && V <= 256 && V % kBV == 0;
}

size_t chunk_tc_unit_bytes(int K, int V) { return tc_layout(K, V).stride; }

cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st) {
    if (a.K == 64) return launch_k<64>(a, st);
    return launch_k<128>(a, st);
}

}  // namespace kda

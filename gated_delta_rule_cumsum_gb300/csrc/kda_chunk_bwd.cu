// kda_chunk_bwd.cu -- chunked KDA backward for bf16 inputs on the sm_103a tensor
// cores (tcgen05.mma with accumulators in tensor memory, bulk async copies).
//
// kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Backward" (the seven launches:
// recompute, re-scan, dAv, dhu, wy_dqkg, intra, dg cumsum), per value head and
// chunk of BT = 64 rows, g2 the chunk-local cumsum of g_scale g (log2), G its
// last row, qg = q 2^g2, kg = k 2^(G - g2), kp = k 2^g2, kn = k 2^-g2, Aqk the
// unscaled q-k gram (o = scale (qg h + Aqk v')), Akk = (I + L)^-1 with
// L = diag(beta) strictly_tril(kp kn^T) =: diag(beta) P, w = Akk diag(beta) kp:
//
//   1, 2  the forward's prep and scan run again and also store, per unit, w and
//         Akk (prep) and the state h_c at the start of the chunk and v'_c (scan);
//   4     dhu, one CTA per (sequence, value head, 32 value columns), chunks in
//         reverse (chunk_dhu_tc_kernel):
//           dv'_c = scale Aqk^T do_c + kg_c dh_{c+1}
//           dh_c  = 2^G dh_{c+1} + scale qg_c^T do_c - w_c^T dv'_c
//         storing dh_{c+1} and dv'_c per unit;
//   3, 5, 6, 7  one CTA per (chunk, value head), all in parallel
//         (chunk_bwd_unit_tc_kernel): with dA = scale tril(do v'^T)
//           dq  = scale (do h^T) 2^g2 + (dA kn) 2^g2
//           dk  = (v' dh^T) 2^(G - g2) + diag(beta) (Akk^T dw) 2^g2
//                 + (dP kn) 2^g2 + (dP^T kp + dA^T qp) 2^-g2,   dw = -dv' h^T
//           dv  = diag(beta) Akk^T dv'
//           dP  = diag(beta) dL,  dL = -strictly_tril(Akk^T dAkk Akk^T),
//           dAkk = (dv' v^T + dw kp^T) diag(beta)
//           dbeta = rowsum(Akk^T dv' . v) + rowsum(Akk^T dw . kp) + rowsum(dL . P)
//           dg2 = ln2 [ scale (do h^T) . qg - (v' dh^T) . kg + diag(beta)(Akk^T dw) . kp
//                      + (dP kn) . kp + (dA kn) . qp - (dP^T kp + dA^T qp) . kn ]
//                 plus, on the last row, ln2 2^G rowsum(h . dh_{c+1}) + ln2 colsum((v' dh^T) . kg)
//           dg  = g_scale x the reverse cumsum of dg2 over the chunk's rows.
//         The gated grams are split through the chunk start (kp, kn), as in the
//         forward's prep; chunks whose gate range max |g2| exceeds kBwdRange are not
//         computed and raise KDA_DEVICE_GATE_RANGE.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_chunk_layout.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr float kLn2 = 0.69314718055994531f;
// Largest chunk gate range (log2) the split grams of the backward take: kn reaches
// 2^range, and its products with dP stay well inside fp32.
constexpr float kBwdRange = 100.f;

// L2 prefetch of a contiguous range (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void bulk_prefetch(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ int read_flag(const int *f) {
    return *reinterpret_cast<const volatile int *>(f);
}
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// ============================================================== dhu kernel
// Rounds i = 0 .. nc - 1 of one (sequence, value head, SBV value columns) take the
// chunks c = nc - 1 - i in reverse.  dh_{c+1} (fp32, thread d of the dh warps owns
// row d) enters as a bf16 operand tile; per round
//   D1a = Aqk_c^T do_c,  D2a = qg_c^T do_c     (off the chain, issued first)
//   D1b = kg_c dh_{c+1}                         ->  dv'_c = scale D1a + D1b
//   D2b = w_c^T dv'_c                           ->  dh_c = 2^G_c dh_{c+1} + scale D2a - D2b
// Aqk, qg and w are read as MN-major operands of the tiles the forward stored.
template <int KK, int SBV>
struct DhuSmem {
    static constexpr int kStages = 3;
    static constexpr uint32_t kg = 0;                        // [64][KK] kg_c
    static constexpr uint32_t wq = kg + 64 * KK * 2;         // [128][KK]: w_c; qg_c
    static constexpr uint32_t aqk = wq + 128 * KK * 2;       // [64][64] Aqk_c
    static constexpr uint32_t dec = aqk + 64 * 64 * 2;       // [128] fp32 2^G_c
    static constexpr uint32_t stage = dec + 512;
    static constexpr uint32_t stage_stride = (stage + 1023) / 1024 * 1024;
    static constexpr uint32_t dh = kStages * stage_stride;   // [KK][SBV] bf16 tile
    static constexpr int kDoBufs = 3;                        // do of chunks c, c - 1, c - 2
    static constexpr uint32_t dout = dh + KK * SBV * 2;      // kDoBufs [64][SBV] tiles
    static constexpr uint32_t dvp = dout + kDoBufs * 64 * SBV * 2;  // [64][SBV] tile
    static constexpr uint32_t total = dvp + 64 * SBV * 2;
    // TMEM columns: D1a at 0 / SBV, D1b at 2 SBV, D2a at 3 SBV / 4 SBV, D2b at 5 SBV.
    static constexpr uint32_t tmem_cols = 6 * SBV <= 256 ? 256 : 512;
};
constexpr int kDhuBarH = 1;  // dh_{c+1} written: the 4 dh warps arrive, the MMA warp syncs
constexpr int kDhuBarV = 2;  // dv'_c written: the 4 dv' warps arrive, the MMA warp syncs

struct BwdArgs {
    ChunkArgs c;           // the forward's arguments, bwd set, its checkpoints
    const void *dout;      // [B,T,HV,V] bf16
    const float *dht;      // [N,HV,K,V] or null
    float *dq, *dk;        // [B,T,H,K]: stored, or with HV > H added (zeroed first)
    float *dv, *dg;        // [B,T,HV,V], [B,T,HV,K]
    float *dbeta;          // [B,T,HV]
    float *dh0;            // [N,HV,K,V] or null
    void *dhn, *dvp;       // per unit: [K][V] tile dL/dh_{c+1}, [64][V] tile dL/dv'_c
    const float *hend;     // [N,HV,K,V]: the final states, stored by the forward re-run
    float *dgs;            // per unit [V/32][K]: sum over 32 value columns of h_{c+1} dh_{c+1}
    // Pipelined launches (dense input): the reverse scan of chunks [pipe_m, nc) of every
    // sequence (part 1: from dht, its last state gradient to dhm) runs first, then that
    // of [0, pipe_m) (part 2: from dhm) beside the gradients of the first part's chunks.
    int dhu_part;          // 0: every chunk; 1 or 2 as above
    int pipe_m;
    float *dhm;            // [N,HV,K,V] fp32
    int unit_c0, unit_c1;  // the gradient kernel's chunks in every sequence (c1 <= c0: all units)
};

// Warp roles: 0..3 dh (rows 32 w .. 32 w + 31), 4..7 dv' (M = 64 rows 16 (w % 4) ..
// + 15 in TMEM lanes 32 (w % 4) .. + 15) and the do tiles, 8 bulk copies, 9 MMA issue.
template <int KK, int SBV>
__global__ void __launch_bounds__(320, 1) chunk_dhu_tc_kernel(BwdArgs a) {
    using S = DhuSmem<KK, SBV>;
    constexpr int kStages = S::kStages;
    const ChunkArgs &p = a.c;
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint64_t full[kStages], empty[kStages], do_full[S::kDoBufs], bar_d1, bar_d2, bar_fin;
    __shared__ uint32_t tslot;
    __shared__ int abort_flag;

    const int nvb = p.V / SBV;
    const int vb = (int)(blockIdx.x % nvb);
    const int hv = (int)((blockIdx.x / nvb) % p.HV);
    const int n = (int)(blockIdx.x / ((int64_t)nvb * p.HV));
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
    // this launch's chunks [c_lo, c_hi), taken in reverse
    const int c_lo = a.dhu_part == 2 ? 0 : (a.dhu_part == 1 ? min(a.pipe_m, nc) : 0);
    const int c_hi = a.dhu_part == 2 ? min(a.pipe_m, nc) : nc;
    const int ncs = c_hi - c_lo;
    const float *dh_in = a.dhu_part == 2 ? a.dhm : a.dht;
    float *dh_out = a.dhu_part == 1 ? a.dhm : a.dh0;
    const TcLayout Lo = tc_layout(KK, p.V, true);
    const unsigned char *units = static_cast<const unsigned char *>(p.units);

    if (warp == 0) {
        tmem_alloc(&tslot, S::tmem_cols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 4);  // MMA commit + the dh warps (they read 2^G)
        }
        for (int x = 0; x < S::kDoBufs; ++x) mbar_init(&do_full[x], 4);
        mbar_init(&bar_d1, 1);
        mbar_init(&bar_d2, 1);
        mbar_init(&bar_fin, 1);
        mbar_fence_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    unsigned char *sDh = sm + S::dh;
    unsigned char *sDo = sm + S::dout;
    unsigned char *sDvp = sm + S::dvp;
    auto fail = [&]() {
        atomicExch(&abort_flag, 1);
        report(p.status, KDA_DEVICE_TIMEOUT);
    };
    auto wait_copy = [&](uint64_t *bar, uint32_t parity) {
        if (read_flag(&abort_flag)) return;
        if (!mbar_wait(bar, parity, kWaitNs)) fail();
    };
    auto wait_mma = [&](uint64_t *bar, uint32_t parity) {
        if (!mbar_wait(bar, parity, kWaitNs)) fail();
    };
    auto stage = [&](int i) { return sm + (i % kStages) * S::stage_stride; };
    auto uidx = [&](int c) { return unit_index(p, gc0 + c, hv); };

    if (warp == 8) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < ncs; ++i) {
                const int s = i % kStages;
                if (i >= kStages) wait_copy(&empty[s], ((i / kStages) - 1) & 1);
                if (read_flag(&abort_flag)) break;
                unsigned char *st = stage(i);
                const unsigned char *U = units + uidx(c_hi - 1 - i) * (int64_t)Lo.stride;
                mbar_arrive_expect_tx(&full[s], 3 * 64 * KK * 2 + 64 * 64 * 2 + 512);
                bulk_g2s(st + S::kg, U + Lo.kgt, 64 * KK * 2, &full[s]);
                bulk_g2s(st + S::wq, U + Lo.wb, 64 * KK * 2, &full[s]);
                bulk_g2s(st + S::wq + 64 * KK * 2, U + Lo.aw + 64 * KK * 2, 64 * KK * 2, &full[s]);
                bulk_g2s(st + S::aqk, U + Lo.aqk, 64 * 64 * 2, &full[s]);
                bulk_g2s(st + S::dec, U + Lo.dec, 512, &full[s]);
                issued = i + 1;
            }
            for (int i = issued - kStages > 0 ? issued - kStages : 0; i < issued; ++i)
                mbar_wait(&full[i % kStages], (i / kStages) & 1, kWaitNs);
        }
    } else if (warp == 9) {
        // ----------------------------------------------------- MMA issuer
        const uint32_t id_d1a = idesc_bf16(64, SBV, true, true);    // Aqk^T (MN-major), do
        const uint32_t id_d1b = idesc_bf16(64, SBV, false, true);   // kg (K-major), dh
        const uint32_t id_d2 = idesc_bf16(128, SBV, true, true);    // qg^T / w^T, do / dv'
        constexpr uint32_t binc = 2 * SBV * 16 / 16;
        const uint64_t ddh = sdesc(smem_addr(sDh), SBV * 16, 128);
        const uint64_t ddv = sdesc(smem_addr(sDvp), SBV * 16, 128);
        for (int i = 0; i < ncs; ++i) {
            const int s = i % kStages;
            const uint32_t st = smem_addr(stage(i));
            const uint64_t ddo = sdesc(smem_addr(sDo) + (i % S::kDoBufs) * 64 * SBV * 2, SBV * 16, 128);
            wait_copy(&full[s], (i / kStages) & 1);
            wait_copy(&do_full[i % S::kDoBufs], (i / S::kDoBufs) & 1);
            __syncwarp();
            bool go = !read_flag(&abort_flag);
            if (elect_one()) {
                tc_fence_after();
                if (go) {
                    mma_bf16_seq<4, false>(tmem + (i & 1) * SBV, sdesc(st + S::aqk, 64 * 16, 128),
                                           2 * 64 * 16 / 16, ddo, binc, id_d1a);
                    mma_bf16_seq<4, false>(tmem + (3 + (i & 1)) * SBV,
                                           sdesc(st + S::wq + 64 * KK * 2, KK * 16, 128),
                                           2 * KK * 16 / 16, ddo, binc, id_d2);
                }
            }
            __syncwarp();
            named_sync(kDhuBarH, 128 + 32);
            go = !read_flag(&abort_flag);
            if (elect_one()) {
                tc_fence_after();
                if (go)
                    mma_bf16_seq<KK / 16, false>(tmem + 2 * SBV, sdesc(st + S::kg, 128, KK * 16), 16,
                                                 ddh, binc, id_d1b);
                mma_commit(&bar_d1);
            }
            __syncwarp();
            named_sync(kDhuBarV, 128 + 32);
            go = !read_flag(&abort_flag);
            if (elect_one()) {
                tc_fence_after();
                if (go)
                    mma_bf16_seq<4, false>(tmem + 5 * SBV, sdesc(st + S::wq, KK * 16, 128),
                                           2 * KK * 16 / 16, ddv, binc, id_d2);
                mma_commit(&bar_d2);
                mma_commit(&empty[s]);
            }
            __syncwarp();
        }
        if (elect_one()) {
            mma_commit(&bar_fin);
            mbar_wait(&bar_fin, 0, kWaitNs);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------ dh warps: the state gradient
        const int row = warp * 32 + lane;
        const bool glob_row = row < p.K;
        const uint32_t lanebase = (uint32_t)(warp * 32) << 16;
        float dh[SBV];
#pragma unroll
        for (int j = 0; j < SBV; ++j) dh[j] = 0.f;
        if (dh_in && glob_row) {
            const float4 *src = reinterpret_cast<const float4 *>(
                dh_in + (((size_t)n * p.HV + hv) * p.K + row) * (size_t)p.V + (size_t)vb * SBV);
#pragma unroll
            for (int j = 0; j < SBV / 4; ++j) {
                const float4 x = src[j];
                dh[4 * j] = x.x; dh[4 * j + 1] = x.y; dh[4 * j + 2] = x.z; dh[4 * j + 3] = x.w;
            }
        }
        // The decay's gradient needs sum_j h_{c+1} dh_{c+1} per row: the state at the
        // end of chunk c against its gradient (the two terms the chain rule gives,
        // 2^G h_c . dh_{c+1} and colsum(dkg . kg), add up to it since kg^T v'_c =
        // h_{c+1} - 2^G h_c).  h_{c+1} is chunk c + 1's checkpoint, loaded a round
        // ahead; for the last chunk it is the final state.
        uint4 hnext[SBV / 8];
        for (int i = 0; i < ncs; ++i) {
            const int c = c_hi - 1 - i;
            // dh_{c+1}: the D1b operand and chunk c's dL/dh_{c+1} tile
            unsigned char *t = static_cast<unsigned char *>(a.dhn) +
                               uidx(c) * (int64_t)(KK * p.V * 2);
#pragma unroll
            for (int cc = 0; cc < SBV; cc += 8) {
                const uint4 v8 = pack8_at(dh + cc);
                *reinterpret_cast<uint4 *>(sDh + tile_off(row, cc, SBV)) = v8;
                *reinterpret_cast<uint4 *>(t + tile_off(row, vb * SBV + cc, p.V)) = v8;
            }
            fence_async_smem();
            __syncwarp();
            named_arrive(kDhuBarH, 128 + 32);
            // off the chain: dh_{c+1} stays in registers until the update below
            {
                float dot = 0.f;
                if (i == 0 && c + 1 < nc) {  // a part-2 launch: chunk c + 1's checkpoint
                    const unsigned char *hc = static_cast<const unsigned char *>(p.ck_h) +
                                              uidx(c + 1) * (int64_t)(KK * p.V * 2) +
                                              tile_off(row, vb * SBV, p.V);
#pragma unroll
                    for (int j = 0; j < SBV / 8; ++j)
                        hnext[j] = *reinterpret_cast<const uint4 *>(hc + j * 128);
                }
                if (i == 0 && c + 1 == nc) {
                    if (glob_row) {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            a.hend + (((size_t)n * p.HV + hv) * p.K + row) * (size_t)p.V + (size_t)vb * SBV);
#pragma unroll
                        for (int j = 0; j < SBV / 4; ++j) {
                            const float4 x = src[j];
                            dot = fmaf(x.x, dh[4 * j], fmaf(x.y, dh[4 * j + 1],
                                  fmaf(x.z, dh[4 * j + 2], fmaf(x.w, dh[4 * j + 3], dot))));
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < SBV / 8; ++j) {
                        float f[8];
                        unpack8(hnext[j], f);
#pragma unroll
                        for (int t = 0; t < 8; ++t) dot = fmaf(f[t], dh[8 * j + t], dot);
                    }
                }
                a.dgs[(uidx(c) * (p.V / SBV) + vb) * KK + row] = dot;
                if (c > c_lo) {  // chunk c's checkpoint is h_{c} = the next round's h_{c'+1}
                    const unsigned char *hc = static_cast<const unsigned char *>(p.ck_h) +
                                              uidx(c) * (int64_t)(KK * p.V * 2) +
                                              tile_off(row, vb * SBV, p.V);
#pragma unroll
                    for (int j = 0; j < SBV / 8; ++j)
                        hnext[j] = *reinterpret_cast<const uint4 *>(hc + j * 128);
                }
            }
            float dec = 0.f;
            wait_copy(&full[i % kStages], (i / kStages) & 1);
            if (!read_flag(&abort_flag)) dec = reinterpret_cast<const float *>(stage(i) + S::dec)[row];
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[i % kStages]);
            wait_mma(&bar_d2, i & 1);
            tc_fence_after();
            float d2a[SBV], d2b[SBV];
            if constexpr (SBV == 32) {
                tmem_ld32(tmem + lanebase + (3 + (i & 1)) * SBV, d2a);
                tmem_ld32(tmem + lanebase + 5 * SBV, d2b);
            } else {
                tmem_ld16(tmem + lanebase + (3 + (i & 1)) * SBV, d2a);
                tmem_ld16(tmem + lanebase + 5 * SBV, d2b);
            }
#pragma unroll
            for (int j = 0; j < SBV; ++j) dh[j] = fmaf(dec, dh[j], fmaf(p.scale, d2a[j], -d2b[j]));
            tc_fence_before();
        }
        if (dh_out && glob_row && !read_flag(&abort_flag)) {
            float4 *dst = reinterpret_cast<float4 *>(
                dh_out + (((size_t)n * p.HV + hv) * p.K + row) * (size_t)p.V + (size_t)vb * SBV);
#pragma unroll
            for (int j = 0; j < SBV / 4; ++j)
                dst[j] = make_float4(dh[4 * j], dh[4 * j + 1], dh[4 * j + 2], dh[4 * j + 3]);
        }
    } else {
        // ------------------------------------- dv' warps: dv'_c = scale D1a + D1b
        const int q = warp & 3, t128 = tid - 128;
        const int r = 16 * q + (lane & 15);
        const uint32_t lanebase = (uint32_t)(32 * q) << 16;
        const __nv_bfloat16 *dout = static_cast<const __nv_bfloat16 *>(a.dout);
        // do rows of chunk c into tile buf by 16-byte cp.async (zero fill past the
        // sequence), one commit group per chunk; issued two rounds ahead so that the
        // loads' latency stays off the chain
        auto issue_do = [&](int c, int buf) {
            if (c >= c_lo) {
                const int row0 = bos + c * kBT;
                const int nr = min(kBT, eos - row0);
                unsigned char *dst = sDo + buf * 64 * SBV * 2;
                for (int pc = t128; pc < 64 * (SBV / 8); pc += 128) {
                    const int rr = pc / (SBV / 8), ch = (pc % (SBV / 8)) * 8;
                    const __nv_bfloat16 *src =
                        dout + (((size_t)b * p.T + row0 + (rr < nr ? rr : 0)) * p.HV + hv) * p.V +
                        vb * SBV + ch;
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                                     smem_addr(dst + tile_off(rr, ch, SBV))),
                                 "l"(src), "r"(rr < nr ? 16 : 0)
                                 : "memory");
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        // the oldest group in flight (chunk c's) has landed: hand its tile to the MMAs
        auto publish_do = [&](int buf) {
            asm volatile("cp.async.wait_group 1;" ::: "memory");
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&do_full[buf]);
        };
        issue_do(c_hi - 1, 0);
        issue_do(c_hi - 2, 1);
        if (ncs > 0) publish_do(0);
        for (int i = 0; i < ncs; ++i) {
            const int c = c_hi - 1 - i;
            wait_mma(&bar_d1, i & 1);
            tc_fence_after();
            float d1a[SBV], d1b[SBV];
            if constexpr (SBV == 32) {
                tmem_ld32(tmem + lanebase + (i & 1) * SBV, d1a);
                tmem_ld32(tmem + lanebase + 2 * SBV, d1b);
            } else {
                tmem_ld16(tmem + lanebase + (i & 1) * SBV, d1a);
                tmem_ld16(tmem + lanebase + 2 * SBV, d1b);
            }
            tc_fence_before();
            if (lane < 16) {
                unsigned char *t = static_cast<unsigned char *>(a.dvp) +
                                   uidx(c) * (int64_t)(64 * p.V * 2);
#pragma unroll
                for (int j = 0; j < SBV; ++j) d1a[j] = fmaf(p.scale, d1a[j], d1b[j]);
#pragma unroll
                for (int cc = 0; cc < SBV; cc += 8) {
                    const uint4 v8 = pack8_at(d1a + cc);
                    *reinterpret_cast<uint4 *>(sDvp + tile_off(r, cc, SBV)) = v8;
                    *reinterpret_cast<uint4 *>(t + tile_off(r, vb * SBV + cc, p.V)) = v8;
                }
            }
            fence_async_smem();
            __syncwarp();
            named_arrive(kDhuBarV, 128 + 32);
            // tile (i + 2) % 3 was last read by round i - 1's MMAs, complete once
            // bar_d1 of round i fired
            issue_do(c - 2, (i + 2) % S::kDoBufs);
            if (i + 1 < ncs) publish_do((i + 1) % S::kDoBufs);
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, S::tmem_cols);
}

// ============================================================ unit kernel
// Shared memory of one (chunk, value head) unit.  Operand tiles in the no-swizzle
// core-matrix layout (tile_off); g2 fp32 with 16-byte column groups XORed by row.
template <int KK, int VV>
struct UnitSmem {
    static constexpr uint32_t g2 = 0;                         // fp32 [64][KK]
    static constexpr uint32_t kp = g2 + 64 * KK * 4;          // [64][KK] k 2^g2
    static constexpr uint32_t kn = kp + 64 * KK * 2;          // [64][KK] k 2^-g2
    static constexpr uint32_t qp = kn + 64 * KK * 2;          // [64][KK] q 2^g2
    static constexpr uint32_t vt = qp + 64 * KK * 2;          // [64][VV] v
    static constexpr uint32_t akk = vt + 64 * VV * 2;         // [64][64] Akk
    static constexpr uint32_t dout = akk + 64 * 64 * 2;       // [64][VV] do; later [dP; dA] [128][64]
    static constexpr uint32_t dvp = dout + 64 * VV * 2;       // [64][VV] dv' (right below do)
    static constexpr uint32_t vp = dvp + 64 * VV * 2;         // [64][VV] v'
    static constexpr uint32_t h = vp + 64 * VV * 2;           // [KK][VV] h_c
    static constexpr uint32_t dhn = h + KK * VV * 2;          // [KK][VV] dh_{c+1}
    static constexpr uint32_t misc = dhn + KK * VV * 2;
    // over h once the first MMAs have read it, and over dh_{c+1} once the second have
    static constexpr uint32_t dw = h;                         // [64][KK]
    static constexpr uint32_t dakk = dw + 64 * KK * 2;        // [64][64]
    static constexpr uint32_t xt = dakk + 64 * 64 * 2;        // [64][64] Akk^T dAkk
    static constexpr uint32_t dg2 = g2;                       // fp32 [64][KK], for the final cumsum
    static constexpr uint32_t dap = dout;                     // [128][64]: dP; dA
    static constexpr uint32_t beta = misc;                    // fp32 [64]
    static constexpr uint32_t gl = beta + 64 * 4;             // fp32 [KK]: G
    static constexpr uint32_t dG = gl + KK * 4;               // fp32 [KK]
    static constexpr uint32_t egl = dG + KK * 4;              // fp32 [KK]: 2^G
    static constexpr uint32_t seg = egl + KK * 4;             // fp32 [4][KK]: cumsum segment totals
    static constexpr uint32_t total = seg + 4 * KK * 4;
    static_assert(xt + 64 * 64 * 2 <= dhn, "tiles over h");
    static_assert(128 * 64 * 2 <= 64 * VV * 2, "[dP; dA] fits over do");
};

template <int W>
__device__ __forceinline__ int fsw(int r, int c) {
    return r * W + ((((c >> 2) ^ r) & 7) | ((c >> 2) & ~7)) * 4 + (c & 3);
}
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void unpack8(const unsigned char *p, float (&f)[8]) {
    unpack8(*reinterpret_cast<const uint4 *>(p), f);
}
// fp32 accumulation into a gradient in global memory (several CTAs may add to
// the same q / k row when value heads share it).
__device__ __forceinline__ void add8(float *dst, const float (&x)[8]) {
    atomicAdd(reinterpret_cast<float4 *>(dst), make_float4(x[0], x[1], x[2], x[3]));
    atomicAdd(reinterpret_cast<float4 *>(dst + 4), make_float4(x[4], x[5], x[6], x[7]));
}

// One CTA of 16 warps per (chunk, value head).  Epilogue threads read accumulators
// with 32-lane TMEM loads: warp w reaches lanes 32 (w % 4) .. + 31 and the four
// warps of a lane quadrant take a quarter of the columns each.  For an M = 128
// result that is rows 32 (w % 4) .. + 31; for an M = 64 result row r sits in lane
// 32 (r / 16) + r % 16, so lanes 0..15 of every warp hold a row.
constexpr int kUnitThreads = 512;

template <int KK, int VV>
__global__ void __launch_bounds__(kUnitThreads, 1) chunk_bwd_unit_tc_kernel(BwdArgs a) {
    using S = UnitSmem<KK, VV>;
    constexpr int NT = kUnitThreads;
    const ChunkArgs &p = a.c;
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tslot;
    __shared__ int range_bad;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, part = warp >> 2;
    const TcLayout Lo = tc_layout(KK, VV, true);
    float *sG = reinterpret_cast<float *>(sm + S::g2);
    float *sBeta = reinterpret_cast<float *>(sm + S::beta);
    float *sGl = reinterpret_cast<float *>(sm + S::gl);
    float *sDG = reinterpret_cast<float *>(sm + S::dG);
    float *sDg2 = reinterpret_cast<float *>(sm + S::dg2);

    if (warp == 0) {
        tmem_alloc(&tslot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    const uint32_t s0 = smem_addr(sm);
    uint32_t phase = 0, ld_phase = 0;
    // this launch's units: every chunk slot of every value head, or (a pipelined
    // launch's part, dense input) chunks [unit_c0, unit_c1) of every sequence
    const bool ranged = a.unit_c1 > a.unit_c0;
    const int uw = a.unit_c1 - a.unit_c0, ntc = (p.T + kBT - 1) / kBT;
    const int64_t per_hv = ranged ? (int64_t)p.B * uw : p.slots;
    const int64_t units = per_hv * p.HV;
    auto unit_at = [&](int64_t it, int &uhv, int64_t &ugc) {
        uhv = (int)(it / per_hv);
        const int64_t r = it - uhv * per_hv;
        ugc = ranged ? (r / uw) * ntc + a.unit_c0 + (r % uw) : r;
    };
    // A unit's inputs into L2: one thread bulk-prefetches the five tiles (one TMA
    // operation each); the 64 rows of q, k, g, v and do, 12 lines of 128 bytes a row
    // at K = V = 128, take a line prefetch per thread (a bulk prefetch per row was
    // measured to hold its warp for ~16K cycles).
    auto prefetch_unit = [&](int64_t u) {
        if (u >= units) return;
        int uhv;
        int64_t ugc;
        unit_at(u, uhv, ugc);
        int ub, ur0, unr, ucl;
        if (!locate_chunk(p, ugc, ub, ur0, unr, ucl)) return;
        const int64_t uui = unit_index(p, ugc, uhv);
        const int uhq = uhv / (p.HV / p.H);
        const size_t urb = (size_t)ub * p.T + ur0;
        if (tid == 32) {
            bulk_prefetch(static_cast<const unsigned char *>(p.ck_h) + uui * (int64_t)(KK * VV * 2), KK * VV * 2);
            bulk_prefetch(static_cast<const unsigned char *>(a.dhn) + uui * (int64_t)(KK * VV * 2), KK * VV * 2);
            bulk_prefetch(static_cast<const unsigned char *>(p.ck_vp) + uui * (int64_t)(64 * VV * 2), 64 * VV * 2);
            bulk_prefetch(static_cast<const unsigned char *>(a.dvp) + uui * (int64_t)(64 * VV * 2), 64 * VV * 2);
            bulk_prefetch(static_cast<const unsigned char *>(p.units) + uui * (int64_t)Lo.stride + Lo.akk,
                          64 * 64 * 2);
        }
        constexpr int kLines = KK * 2 / 128 * 2 + KK * 4 / 128 + VV * 2 / 128 * 2;  // per row
        for (int li = tid; li < unr * kLines; li += NT) {
            const int r = li / kLines, j = li % kLines;
            const char *ptr;
            if (j < 2 * (KK * 2 / 128)) {
                const int t = j / (KK * 2 / 128), o = j % (KK * 2 / 128);
                ptr = reinterpret_cast<const char *>(static_cast<const __nv_bfloat16 *>(t ? p.k : p.q) +
                                                     ((urb + r) * p.H + uhq) * p.K) + 128 * o;
            } else if (j < 2 * (KK * 2 / 128) + KK * 4 / 128) {
                const int o = j - 2 * (KK * 2 / 128);
                ptr = reinterpret_cast<const char *>(p.g + ((urb + r) * p.HV + uhv) * p.K) + 128 * o;
            } else {
                const int jj = j - 2 * (KK * 2 / 128) - KK * 4 / 128;
                const int t = jj / (VV * 2 / 128), o = jj % (VV * 2 / 128);
                ptr = reinterpret_cast<const char *>(static_cast<const __nv_bfloat16 *>(t ? a.dout : p.v) +
                                                     ((urb + r) * p.HV + uhv) * p.V) + 128 * o;
            }
            asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
        }
    };

    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    int hv;
    int64_t gc;
    unit_at(unit, hv, gc);
    int b, row0, nr, cl;
    if (!locate_chunk(p, gc, b, row0, nr, cl)) continue;
    const int hq = hv / (p.HV / p.H);
    const int64_t ui = unit_index(p, gc, hv);
    if (tid == 0) {
        range_bad = 0;
        // the previous unit's reads of these buffers precede the copies' writes
        fence_async_smem();
        // the forward's and the dhu's tiles of this unit
        mbar_arrive_expect_tx(&bar_ld, 2 * KK * VV * 2 + 2 * 64 * VV * 2 + 64 * 64 * 2);
        bulk_g2s(sm + S::h, static_cast<const unsigned char *>(p.ck_h) + ui * (int64_t)(KK * VV * 2),
                 KK * VV * 2, &bar_ld);
        bulk_g2s(sm + S::dhn, static_cast<const unsigned char *>(a.dhn) + ui * (int64_t)(KK * VV * 2),
                 KK * VV * 2, &bar_ld);
        bulk_g2s(sm + S::vp, static_cast<const unsigned char *>(p.ck_vp) + ui * (int64_t)(64 * VV * 2),
                 64 * VV * 2, &bar_ld);
        bulk_g2s(sm + S::dvp, static_cast<const unsigned char *>(a.dvp) + ui * (int64_t)(64 * VV * 2),
                 64 * VV * 2, &bar_ld);
        bulk_g2s(sm + S::akk, static_cast<const unsigned char *>(p.units) + ui * (int64_t)Lo.stride + Lo.akk,
                 64 * 64 * 2, &bar_ld);
    }
    const size_t rowbase = (size_t)b * p.T + row0;
    // Input rows: every load of a thread is issued before its first store, so that
    // their latencies overlap; q and k stay in registers across the cumsum.
    constexpr int kQkIt = 64 * (KK / 8) / NT;
    uint4 qraw[kQkIt], kraw[kQkIt];
    {
        const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
        const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
#pragma unroll
        for (int it = 0; it < kQkIt; ++it) {
            const int pc = tid + it * NT, r = pc / (KK / 8), c = (pc % (KK / 8)) * 8;
            qraw[it] = kraw[it] = make_uint4(0, 0, 0, 0);
            if (r < nr && c < p.K) {
                const size_t off = ((rowbase + r) * p.H + hq) * p.K + c;
                qraw[it] = *reinterpret_cast<const uint4 *>(q + off);
                kraw[it] = *reinterpret_cast<const uint4 *>(k + off);
            }
        }
    }
    {
        constexpr int kGIt = 64 * (KK / 4) / NT, kVIt = 64 * (VV / 8) / NT;
        const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
        const __nv_bfloat16 *dout = static_cast<const __nv_bfloat16 *>(a.dout);
        float4 x[kGIt];
        uint4 y[kVIt], z[kVIt];
#pragma unroll
        for (int it = 0; it < kGIt; ++it) {
            const int pc = tid + it * NT, r = pc / (KK / 4), c = (pc % (KK / 4)) * 4;
            x[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < nr && c < p.K)
                x[it] = *reinterpret_cast<const float4 *>(p.g + ((rowbase + r) * p.HV + hv) * p.K + c);
        }
        if (p.act.A_log) {  // the activated gate -exp(A_log) softplus(g + dt_bias), as the forward
            const float na = gate_neg_a(p.act, hv);
#pragma unroll
            for (int it = 0; it < kGIt; ++it) {
                const int pc = tid + it * NT, r = pc / (KK / 4), c = (pc % (KK / 4)) * 4;
                if (r < nr && c < p.K) {
                    float *e = reinterpret_cast<float *>(&x[it]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) e[j] = na * softplus_f(e[j] + gate_bias(p.act, hv, c + j, p.K));
                }
            }
        }
#pragma unroll
        for (int it = 0; it < kVIt; ++it) {
            const int pc = tid + it * NT, r = pc / (VV / 8), c = (pc % (VV / 8)) * 8;
            y[it] = z[it] = make_uint4(0, 0, 0, 0);
            if (r < nr) {
                const size_t off = ((rowbase + r) * p.HV + hv) * p.V + c;
                y[it] = *reinterpret_cast<const uint4 *>(v + off);
                z[it] = *reinterpret_cast<const uint4 *>(dout + off);
            }
        }
        if (tid < 64) {
            float bt = 0.f;
            if (tid < nr) {
                bt = to_f32(static_cast<const __nv_bfloat16 *>(p.beta)[(rowbase + tid) * p.HV + hv]);
                if (p.act.beta_scale > 0.f) bt = beta_activate<__nv_bfloat16>(bt, p.act.beta_scale);
            }
            sBeta[tid] = bt;
        }
#pragma unroll
        for (int it = 0; it < kGIt; ++it) {
            const int pc = tid + it * NT, r = pc / (KK / 4), c = (pc % (KK / 4)) * 4;
            *reinterpret_cast<float4 *>(sG + fsw<KK>(r, c)) = x[it];
        }
#pragma unroll
        for (int it = 0; it < kVIt; ++it) {
            const int pc = tid + it * NT, r = pc / (VV / 8), c = (pc % (VV / 8)) * 8;
            *reinterpret_cast<uint4 *>(sm + S::vt + tile_off(r, c, VV)) = y[it];
            *reinterpret_cast<uint4 *>(sm + S::dout + tile_off(r, c, VV)) = z[it];
        }
    }
    __syncthreads();
    // chunk-local cumsum of g_scale g (rows past the chunk hold zeros, so they keep
    // the last row's value): per channel four threads take 16 rows each, then add
    // the totals of the segments before theirs.  The decay's gradient: ln2 times the
    // reverse scan's per-column-block sums of h_{c+1} dh_{c+1}.
    float *sSeg = reinterpret_cast<float *>(sm + S::seg);
    const int cd = tid & (KK - 1), cs = tid / KK;  // channel, 16-row segment
    float gsum[16];
    if (cs < 4) {
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            acc = fmaf(p.g_scale, sG[fsw<KK>(16 * cs + r, cd)], acc);
            gsum[r] = acc;
        }
        sSeg[cs * KK + cd] = acc;
    }
    if (tid < KK) {
        float x = 0.f;
        for (int vb = 0; vb < VV / 32; ++vb) x += a.dgs[(ui * (VV / 32) + vb) * KK + tid];
        sDG[tid] = kLn2 * x;
    }
    __syncthreads();
    if (cs < 4) {
        float off = 0.f;
        for (int t = 0; t < cs; ++t) off += sSeg[t * KK + cd];
        bool bad = false;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float g2 = gsum[r] + off;
            sG[fsw<KK>(16 * cs + r, cd)] = g2;
            bad |= !(fabsf(g2) <= kBwdRange);  // also NaN
        }
        if (cs == 3) {
            sGl[cd] = gsum[15] + off;
            reinterpret_cast<float *>(sm + S::egl)[cd] = ex2f(gsum[15] + off);
        }
        if (bad) range_bad = 1;
    }
    __syncthreads();
    if (range_bad) {
        // refused: the chunk's gradients are zero (the status word tells the caller)
        if (tid == 0) report(p.status, KDA_DEVICE_GATE_RANGE);
        for (int i = tid; i < nr * (KK / 4); i += NT) {
            const int r = i / (KK / 4), c = (i % (KK / 4)) * 4;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p.H == p.HV) {
                *reinterpret_cast<float4 *>(a.dq + ((rowbase + r) * p.H + hq) * p.K + c) = z;
                *reinterpret_cast<float4 *>(a.dk + ((rowbase + r) * p.H + hq) * p.K + c) = z;
            }
            *reinterpret_cast<float4 *>(a.dg + ((rowbase + r) * p.HV + hv) * p.K + c) = z;
            *reinterpret_cast<float4 *>(a.dv + ((rowbase + r) * p.HV + hv) * p.V + c) = z;
        }
        if (tid < nr) a.dbeta[(rowbase + tid) * p.HV + hv] = 0.f;
        if (tid == 0) mbar_wait(&bar_ld, ld_phase & 1, kWaitNs);  // the copies land first
        ++ld_phase;
        __syncthreads();
        continue;
    }
    // q, k rows -> kp, kn, qp tiles
#pragma unroll
    for (int it = 0; it < kQkIt; ++it) {
        const int pc = tid + it * NT, r = pc / (KK / 8), c = (pc % (KK / 8)) * 8;
        float fq[8], fk[8];
        unpack8(qraw[it], fq);
        unpack8(kraw[it], fk);
        if (p.l2norm) {  // q / sqrt(sum q^2 + 1e-6) per row, as the forward: 16 threads a row
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                sq = fmaf(fq[j], fq[j], sq);
                sk = fmaf(fk[j], fk[j], sk);
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            const float rq = 1.f / sqrtf(sq + 1e-6f), rk = 1.f / sqrtf(sk + 1e-6f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                fq[j] *= rq;
                fk[j] *= rk;
            }
        }
        const float4 g0 = *reinterpret_cast<const float4 *>(sG + fsw<KK>(r, c));
        const float4 g1 = *reinterpret_cast<const float4 *>(sG + fsw<KK>(r, c + 4));
        const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        float kp[8], kn[8], qp[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float e = ex2f(gg[j]), ei = ex2f(-gg[j]);
            kp[j] = fk[j] * e;
            kn[j] = fk[j] * ei;
            qp[j] = fq[j] * e;
        }
        *reinterpret_cast<uint4 *>(sm + S::kp + tile_off(r, c, KK)) = pack8(kp);
        *reinterpret_cast<uint4 *>(sm + S::kn + tile_off(r, c, KK)) = pack8(kn);
        *reinterpret_cast<uint4 *>(sm + S::qp + tile_off(r, c, KK)) = pack8(qp);
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0 && !mbar_wait(&bar_ld, ld_phase & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
    ++ld_phase;
    __syncthreads();
    tc_fence_after();
    prefetch_unit(unit + gridDim.x);  // this CTA's next unit, into L2 while this one computes

    auto mma_wait = [&]() {
        if (!mbar_wait(&bar_mma, phase & 1, kWaitNs) && tid == 0) report(p.status, KDA_DEVICE_TIMEOUT);
        ++phase;
        tc_fence_after();
    };
    // K-major tile [rows][C]: per K = 16 step +256 bytes; MN-major: +2 C * 16 bytes.
    auto kmaj = [&](uint32_t off, int C) { return sdesc(s0 + off, 128, C * 16); };
    auto mnmaj = [&](uint32_t off, int C) { return sdesc(s0 + off, C * 16, 128); };
    auto tl = [&](uint32_t col) { return tmem_at(tmem, 32 * quad, col); };

    // ---- P = kp kn^T, dA = do v'^T, Qd = do h^T, Wd = dv' h^T (all M = 64)
    if (tid == 0) {
        mma_bf16_seq<KK / 16, false>(tmem + 0, kmaj(S::kp, KK), 16, kmaj(S::kn, KK), 16,
                                     idesc_bf16(64, 64, false, false));
        mma_bf16_seq<VV / 16, false>(tmem + 64, kmaj(S::dout, VV), 16, kmaj(S::vp, VV), 16,
                                     idesc_bf16(64, 64, false, false));
        mma_bf16_seq<VV / 16, false>(tmem + 128, kmaj(S::dout, VV), 16, kmaj(S::h, VV), 16,
                                     idesc_bf16(64, KK, false, false));
        mma_bf16_seq<VV / 16, false>(tmem + 256, kmaj(S::dvp, VV), 16, kmaj(S::h, VV), 16,
                                     idesc_bf16(64, KK, false, false));
        mma_commit(&bar_mma);
    }
    mma_wait();
    __syncthreads();

    const float scale = p.scale;
    auto grow = [&](float *base, int r) { return base + ((rowbase + r) * p.H + hq) * p.K; };
    auto g2v = [&](int r, int c, float (&o)[8]) {
        const float4 x = *reinterpret_cast<const float4 *>(sG + fsw<KK>(r, c));
        const float4 y = *reinterpret_cast<const float4 *>(sG + fsw<KK>(r, c + 4));
        o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w; o[4] = y.x; o[5] = y.y; o[6] = y.z; o[7] = y.w;
    };
    // Every result here is M = 64, read with the 16x32bx2 shape: this thread holds row
    // r64 and, of a result N wide, the N / 8 columns from c64(N) (the two half-warps
    // on adjacent column blocks).  Its dq and dk elements (16 each) accumulate in its
    // own TMEM lane, which no M = 64 result uses, and reach global memory once.
    const int r64 = 16 * quad + (lane & 15), hs = lane >> 4;
    auto col0 = [&](int N) { return part * (N / 4); };
    auto c64 = [&](int N) { return part * (N / 4) + hs * (N / 8); };
    const uint32_t acc_dq = tl(384 + part * 16), acc_dk = tl(448 + part * 16);
    // this thread's 16 elements of dg2 (the gradient with respect to the cumsum), in
    // registers until the final reverse cumsum
    float dgr[16];
    const bool excl = p.H == p.HV;  // no other CTA adds to these q / k rows

    // ---- dq <- scale Qd 2^g2 (its dg2 term, ln2 scale Qd . qp = ln2 dq . qp 2^-g2, is
    // added with the last terms: dg2 lives over dh_{c+1}, which the next MMAs read);
    // dw = -Wd; dA = scale tril(do v'^T)
#pragma unroll
    for (int c8 = 0; c8 < 16; c8 += 8) {
        const int c0 = c64(KK) + c8;
        float d[8], gg[8], acc[8];
        tmem_ld16x2_8<16>(tl(128 + col0(KK) + c8), d);
        g2v(r64, c0, gg);
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[t] = scale * d[t] * ex2f(gg[t]);
        tmem_st8(acc_dq + c8, acc);
        tmem_ld16x2_8<16>(tl(256 + col0(KK) + c8), d);
#pragma unroll
        for (int t = 0; t < 8; ++t) d[t] = -d[t];
        *reinterpret_cast<uint4 *>(sm + S::dw + tile_off(r64, c0, KK)) = pack8_at(d);
    }
    {
        const int c0 = c64(64);
        float d[8];
        tmem_ld16x2_8<8>(tl(64 + col0(64)), d);
#pragma unroll
        for (int t = 0; t < 8; ++t) d[t] = (c0 + t <= r64) ? scale * d[t] : 0.f;
        *reinterpret_cast<uint4 *>(sm + S::dap + tile_off(64 + r64, c0, 64)) = pack8_at(d);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- dkg = v' dh^T; dAkk = dv' v^T + dw kp^T (columns scaled by beta below)
    if (tid == 0) {
        mma_bf16_seq<VV / 16, false>(tmem + 128, kmaj(S::vp, VV), 16, kmaj(S::dhn, VV), 16,
                                     idesc_bf16(64, KK, false, false));
        mma_bf16_seq<VV / 16, false>(tmem + 64, kmaj(S::dvp, VV), 16, kmaj(S::vt, VV), 16,
                                     idesc_bf16(64, 64, false, false));
        mma_bf16_seq<KK / 16, true>(tmem + 64, kmaj(S::dw, KK), 16, kmaj(S::kp, KK), 16,
                                    idesc_bf16(64, 64, false, false));
        mma_commit(&bar_mma);
    }
    mma_wait();
    // ---- dk <- dkg 2^(G - g2); dg2 -= ln2 dkg . kg, kg = kn 2^G
    {
        const float *sEgl = reinterpret_cast<const float *>(sm + S::egl);
#pragma unroll
        for (int c8 = 0; c8 < 16; c8 += 8) {
            const int c0 = c64(KK) + c8;
            float d[8], gg[8], kn[8], acc[8], dg8[8];
            tmem_ld16x2_8<16>(tl(128 + col0(KK) + c8), d);
            g2v(r64, c0, gg);
            unpack8(sm + S::kn + tile_off(r64, c0, KK), kn);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                acc[t] = d[t] * ex2f(sGl[c0 + t] - gg[t]);
                dg8[t] = -kLn2 * d[t] * kn[t] * sEgl[c0 + t];
            }
            tmem_st8(acc_dk + c8, acc);
#pragma unroll
            for (int t = 0; t < 8; ++t) dgr[c8 + t] = dg8[t];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- Akk^T [dv' | dw]
    if (tid == 0) {
        mma_bf16_seq<4, false>(tmem + 128, mnmaj(S::akk, 64), 2 * 64, mnmaj(S::dvp, VV), 2 * VV,
                               idesc_bf16(64, VV, true, true));
        mma_bf16_seq<4, false>(tmem + 256, mnmaj(S::akk, 64), 2 * 64, mnmaj(S::dw, KK), 2 * KK,
                               idesc_bf16(64, KK, true, true));
        mma_commit(&bar_mma);
    }
    mma_wait();
    // ---- dv = diag(beta) Akk^T dv'; dk += diag(beta) (Akk^T dw) 2^g2; dbeta; dAkk tile
    // (this thread's part of dbeta stays in dbp until the dL terms join it)
    float dbp = 0.f;
    {
        const float br = sBeta[r64];
        float db = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < 16; c8 += 8) {
            const int c0 = c64(VV) + c8;
            float d[8], vv[8];
            tmem_ld16x2_8<16>(tl(128 + col0(VV) + c8), d);
            unpack8(sm + S::vt + tile_off(r64, c0, VV), vv);
#pragma unroll
            for (int t = 0; t < 8; ++t) db = fmaf(d[t], vv[t], db);
            if (r64 < nr) {
                float *dvr = a.dv + ((rowbase + r64) * p.HV + hv) * p.V + c0;
                *reinterpret_cast<float4 *>(dvr) = make_float4(br * d[0], br * d[1], br * d[2], br * d[3]);
                *reinterpret_cast<float4 *>(dvr + 4) = make_float4(br * d[4], br * d[5], br * d[6], br * d[7]);
            }
        }
#pragma unroll
        for (int c8 = 0; c8 < 16; c8 += 8) {
            const int c0 = c64(KK) + c8;
            float d[8], gg[8], kp[8], acc[8], dg8[8];
            tmem_ld16x2_8<16>(tl(256 + col0(KK) + c8), d);
            tmem_ld8(acc_dk + c8, acc);
            g2v(r64, c0, gg);
            unpack8(sm + S::kp + tile_off(r64, c0, KK), kp);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                db = fmaf(d[t], kp[t], db);
                const float x = br * d[t];
                acc[t] = fmaf(x, ex2f(gg[t]), acc[t]);
                dg8[t] = kLn2 * x * kp[t];
            }
            tmem_st8(acc_dk + c8, acc);
#pragma unroll
            for (int t = 0; t < 8; ++t) dgr[c8 + t] += dg8[t];
        }
        {
            const int c0 = c64(64);
            float d[8];
            tmem_ld16x2_8<8>(tl(64 + col0(64)), d);
#pragma unroll
            for (int t = 0; t < 8; ++t) d[t] *= sBeta[c0 + t];
            *reinterpret_cast<uint4 *>(sm + S::dakk + tile_off(r64, c0, 64)) = pack8_at(d);
            dbp = db;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- X = Akk^T dAkk
    if (tid == 0) {
        mma_bf16_seq<4, false>(tmem + 128, mnmaj(S::akk, 64), 2 * 64, mnmaj(S::dakk, 64), 2 * 64,
                               idesc_bf16(64, 64, true, true));
        mma_commit(&bar_mma);
    }
    mma_wait();
    {
        const int c0 = c64(64);
        float d[8];
        tmem_ld16x2_8<8>(tl(128 + col0(64)), d);
        *reinterpret_cast<uint4 *>(sm + S::xt + tile_off(r64, c0, 64)) = pack8_at(d);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- Y = X Akk^T
    if (tid == 0) {
        mma_bf16_seq<4, false>(tmem + 192, kmaj(S::xt, 64), 16, kmaj(S::akk, 64), 16,
                               idesc_bf16(64, 64, false, false));
        mma_commit(&bar_mma);
    }
    mma_wait();
    // ---- dL = -strictly_tril(Y); dbeta += rowsum(dL . P); dP = diag(beta) dL
    {
        const int c0 = c64(64);
        float y[8], pp[8];
        tmem_ld16x2_8<8>(tl(192 + col0(64)), y);
        tmem_ld16x2_8<8>(tl(0 + col0(64)), pp);
        const float br = sBeta[r64];
        float db = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float dl = (c0 + t < r64) ? -y[t] : 0.f;
            db = fmaf(dl, pp[t], db);
            y[t] = br * dl;
        }
        *reinterpret_cast<uint4 *>(sm + S::dap + tile_off(r64, c0, 64)) = pack8_at(y);
        // the eight threads of a row put their parts in fixed slots over the X tile (the
        // Y MMA that read it has completed): summed in order below, so dbeta does not
        // depend on timing
        reinterpret_cast<float *>(sm + S::xt)[r64 * 8 + part * 2 + hs] = dbp + db;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- dP kn, dA kn, dP^T kp + dA^T qp
    if (tid == 0) {
        mma_bf16_seq<4, false>(tmem + 0, kmaj(S::dap, 64), 16, mnmaj(S::kn, KK), 2 * KK,
                               idesc_bf16(64, KK, false, true));
        mma_bf16_seq<4, false>(tmem + 128, kmaj(S::dap + 64 * 64 * 2, 64), 16, mnmaj(S::kn, KK),
                               2 * KK, idesc_bf16(64, KK, false, true));
        mma_bf16_seq<4, false>(tmem + 256, mnmaj(S::dap, 64), 2 * 64, mnmaj(S::kp, KK), 2 * KK,
                               idesc_bf16(64, KK, true, true));
        mma_bf16_seq<4, true>(tmem + 256, mnmaj(S::dap + 64 * 64 * 2, 64), 2 * 64, mnmaj(S::qp, KK),
                              2 * KK, idesc_bf16(64, KK, true, true));
        mma_commit(&bar_mma);
    }
    mma_wait();
    // ---- dk += (dP kn) 2^g2 + (dP^T kp + dA^T qp) 2^-g2, dq += (dA kn) 2^g2, their
    // dg2 terms; dq and dk to global memory
#pragma unroll
    for (int c8 = 0; c8 < 16; c8 += 8) {
        const int c0 = c64(KK) + c8;
        float t1[8], t3[8], t9[8], ak[8], aq[8], gg[8], dg8[8];
        tmem_ld16x2_8<16>(tl(0 + col0(KK) + c8), t1);
        tmem_ld16x2_8<16>(tl(128 + col0(KK) + c8), t3);
        tmem_ld16x2_8<16>(tl(256 + col0(KK) + c8), t9);
        tmem_ld8(acc_dk + c8, ak);
        tmem_ld8(acc_dq + c8, aq);
        g2v(r64, c0, gg);
        {
            float f[8];
            unpack8(sm + S::kp + tile_off(r64, c0, KK), f);
#pragma unroll
            for (int t = 0; t < 8; ++t) dg8[t] = t1[t] * f[t];
            unpack8(sm + S::qp + tile_off(r64, c0, KK), f);
#pragma unroll
            for (int t = 0; t < 8; ++t)  // (dA kn) . qp, and the first dq term's ln2 dq . qp 2^-g2
                dg8[t] = fmaf(fmaf(aq[t], ex2f(-gg[t]), t3[t]), f[t], dg8[t]);
            unpack8(sm + S::kn + tile_off(r64, c0, KK), f);
#pragma unroll
            for (int t = 0; t < 8; ++t) dg8[t] = kLn2 * fmaf(-t9[t], f[t], dg8[t]);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float e = ex2f(gg[t]), ei = ex2f(-gg[t]);
            ak[t] = fmaf(t1[t], e, fmaf(t9[t], ei, ak[t]));
            aq[t] = fmaf(t3[t], e, aq[t]);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) dgr[c8 + t] += dg8[t];
        if (r64 < nr && c0 < p.K) {
            float *qd = grow(a.dq, r64) + c0, *kd = grow(a.dk, r64) + c0;
            if (excl) {
                *reinterpret_cast<float4 *>(qd) = make_float4(aq[0], aq[1], aq[2], aq[3]);
                *reinterpret_cast<float4 *>(qd + 4) = make_float4(aq[4], aq[5], aq[6], aq[7]);
                *reinterpret_cast<float4 *>(kd) = make_float4(ak[0], ak[1], ak[2], ak[3]);
                *reinterpret_cast<float4 *>(kd + 4) = make_float4(ak[4], ak[5], ak[6], ak[7]);
            } else {
                add8(qd, aq);
                add8(kd, ak);
            }
        }
    }
    // dg2 over g2, whose last reader was the loop above
    __syncthreads();
#pragma unroll
    for (int c4 = 0; c4 < 16; c4 += 4)
        *reinterpret_cast<float4 *>(sDg2 + fsw<KK>(r64, c64(KK) + c4)) =
            make_float4(dgr[c4], dgr[c4 + 1], dgr[c4 + 2], dgr[c4 + 3]);
    tc_fence_before();
    __syncthreads();
    // ---- dg: g_scale x reverse cumsum of dg2 (G's gradient on the last row), per
    // channel in four 16-row segments; dbeta
    if (cs < 4) {
        float acc = 0.f;
#pragma unroll
        for (int r = 15; r >= 0; --r) {
            const int rr = 16 * cs + r;
            float x = rr < nr ? sDg2[fsw<KK>(rr, cd)] : 0.f;
            if (rr == nr - 1) x += sDG[cd];
            acc += x;
            gsum[r] = acc;
        }
        sSeg[cs * KK + cd] = acc;
    }
    __syncthreads();
    if (cs < 4) {
        float off = 0.f;
        for (int t = cs + 1; t < 4; ++t) off += sSeg[t * KK + cd];
        if (cd < p.K) {
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int rr = 16 * cs + r;
                if (rr < nr) a.dg[((rowbase + rr) * p.HV + hv) * p.K + cd] = p.g_scale * (gsum[r] + off);
            }
        }
    }
    if (tid < nr && tid < 64) {
        const float *slot = reinterpret_cast<const float *>(sm + S::xt) + tid * 8;
        float x = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) x += slot[j];
        a.dbeta[(rowbase + tid) * p.HV + hv] = x;
    }
    tc_fence_before();
    __syncthreads();
    }
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int KK, int SBV>
cudaError_t launch_dhu(const BwdArgs &a, cudaStream_t st) {
    using S = DhuSmem<KK, SBV>;
    static DeviceOnce once;
    int dev = 0;
    cudaError_t e = once.run(&dev, [](int) {
        return cudaFuncSetAttribute(chunk_dhu_tc_kernel<KK, SBV>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::total);
    });
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.c.N * a.c.HV * (a.c.V / SBV);
    if (blocks == 0) return cudaSuccess;
    prof_begin("chunk_dhu_tc", st);
    chunk_dhu_tc_kernel<KK, SBV><<<(unsigned)blocks, 320, S::total, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

template <int KK, int VV>
cudaError_t launch_unit(const BwdArgs &a, cudaStream_t st, int cta_cap = 0) {
    using S = UnitSmem<KK, VV>;
    static DeviceOnce once;
    static int sms[64];
    int dev = 0;
    cudaError_t e = once.run(&dev, [](int d) {
        cudaError_t r = cudaFuncSetAttribute(chunk_bwd_unit_tc_kernel<KK, VV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)S::total);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms[d], cudaDevAttrMultiProcessorCount, d);
        return r;
    });
    if (e != cudaSuccess) return e;
    const int64_t units = a.unit_c1 > a.unit_c0 ? (int64_t)a.c.B * (a.unit_c1 - a.unit_c0) * a.c.HV
                                                : a.c.slots * a.c.HV;
    if (units == 0) return cudaSuccess;
    // persistent: one CTA per SM (its shared memory allows no second), units strided
    const int ctas = cta_cap > 0 && cta_cap < sms[dev] ? cta_cap : sms[dev];
    const unsigned grid = (unsigned)(units < ctas ? units : ctas);
    prof_begin("chunk_bwd_unit_tc", st);
    chunk_bwd_unit_tc_kernel<KK, VV><<<grid, kUnitThreads, S::total, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

// The library's own stream for a pipelined backward's first gradient launch and
// the events that fork it from the caller's stream and join it back, per device.
struct BwdStreams {
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_bwd_mu;

cudaError_t bwd_streams(BwdStreams **out) {
    static BwdStreams per_dev[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    BwdStreams &bs = per_dev[dev];
    if (!bs.side) {
        if ((e = cudaEventCreateWithFlags(&bs.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&bs.join, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&bs.side, cudaStreamNonBlocking)) != cudaSuccess) return e;
    }
    *out = &bs;
    return cudaSuccess;
}

}  // namespace

bool chunk_bwd_tc_supported(int K, int V) { return K == 128 && V == 128; }

int chunk_bwd_pipe_m(int B, int HV, int V, int T, int sms) {
    // Cost model in reverse-scan rounds: a gradient unit takes about 16 rounds of an
    // SM (18 us against 1.13 us at K = V = 128, measured).  Serial: 1 round per chunk,
    // then every unit on all SMs.  Pipelined at m: the rounds of [m, nc), then the
    // longer of the rounds of [0, m) and the units of [m, nc) on the SMs the scan
    // leaves free, then the units of [0, m) on all SMs.
    constexpr int64_t kUnit = 16;
    const int64_t nc = (T + kBT - 1) / kBT;
    const int64_t scan_ctas = (int64_t)B * HV * (V / 32);
    if (nc < 16 || B <= 0 || HV <= 0 || 2 * scan_ctas > sms) return 0;
    const int64_t hb = (int64_t)B * HV, free_sms = sms - scan_ctas;
    auto waves = [](int64_t units, int64_t ctas) { return (units + ctas - 1) / ctas; };
    int64_t best = nc + waves(hb * nc, sms) * kUnit;
    int best_m = 0;
    for (int64_t m = nc / 4; m + 4 <= nc; ++m) {
        const int64_t side = waves(hb * (nc - m), free_sms) * kUnit;
        const int64_t cost = (nc - m) + (m > side ? m : side) + waves(hb * m, sms) * kUnit;
        if (cost < best) {
            best = cost;
            best_m = (int)m;
        }
    }
    return best_m;
}

cudaError_t launch_chunk_bwd_tc(const ChunkArgs &c, const void *dout, const float *dht, float *dq,
                                float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                                void *dhn, void *dvp, float *hend, float *dgs, float *dhm,
                                bool serial, bool rerun, cudaStream_t st) {
    if (!chunk_bwd_tc_supported(c.K, c.V)) return cudaErrorInvalidValue;
    BwdArgs a;
    a.c = c;
    a.c.ht = hend;  // the re-run forward stores the final states there
    a.hend = hend;
    a.dgs = dgs;
    a.dout = dout;
    a.dht = dht;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dg = dg;
    a.dbeta = dbeta;
    a.dh0 = dh0;
    a.dhn = dhn;
    a.dvp = dvp;
    a.dhu_part = 0;
    a.pipe_m = 0;
    a.dhm = dhm;
    a.unit_c0 = a.unit_c1 = 0;
    cudaError_t e = cudaSuccess;
    if (rerun && (e = launch_chunk_tc(a.c, st)) != cudaSuccess)  // recompute and re-scan
        return e;
    static DeviceOnce once;
    static int sms[64];
    int dev = 0;
    if ((e = once.run(&dev, [](int d) {
             return cudaDeviceGetAttribute(&sms[d], cudaDevAttrMultiProcessorCount, d);
         })) != cudaSuccess)
        return e;
    const int m = (!c.cu && !serial && dhm) ? chunk_bwd_pipe_m(c.B, c.HV, c.V, c.T, sms[dev]) : 0;
    if (m == 0) {
        if ((e = launch_dhu<128, 32>(a, st)) != cudaSuccess) return e;
        return launch_unit<128, 128>(a, st);
    }
    // Pipelined: the reverse scan of [m, nc), then on the caller's stream that of
    // [0, m) while the side stream forms the gradients of [m, nc) on the SMs the scan
    // leaves free; the gradients of [0, m) once both are done.  No kernel waits for
    // another: the streams and events order whole launches.
    std::lock_guard<std::mutex> lock(g_bwd_mu);
    BwdStreams *bs = nullptr;
    if ((e = bwd_streams(&bs)) != cudaSuccess) return e;
    const int nc = (c.T + kBT - 1) / kBT;
    BwdArgs s1 = a, s2 = a, u1 = a, u2 = a;
    s1.dhu_part = 1;
    s2.dhu_part = 2;
    s1.pipe_m = s2.pipe_m = m;
    u1.unit_c0 = m;
    u1.unit_c1 = nc;
    u2.unit_c0 = 0;
    u2.unit_c1 = m;
    const int scan_ctas = c.B * c.HV * (c.V / 32);
    if ((e = launch_dhu<128, 32>(s1, st)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(bs->fork, st)) != cudaSuccess) return e;
    if ((e = launch_dhu<128, 32>(s2, st)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(bs->side, bs->fork, 0)) != cudaSuccess) return e;
    if ((e = launch_unit<128, 128>(u1, bs->side, sms[dev] - scan_ctas)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(bs->join, bs->side)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(st, bs->join, 0)) != cudaSuccess) return e;
    return launch_unit<128, 128>(u2, st);
}

}  // namespace kda

// kda_chunk_tc.cu -- chunked KDA forward for bf16 inputs on the sm_103a tensor
// cores (tcgen05.mma, accumulators in tensor memory, bulk async copies).
//
// kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Forward", per value head and per
// chunk of BT = 64 rows with g2 the chunk-local cumsum (log2) and G its last row:
//
//   prep kernel, one CTA per (chunk, value head), all in parallel:
//     Stage 1     g2, G (fp32, per channel)
//     Stage 2     Aqk = tril(Qg Kb^T),  L = diag(beta) * strictly_tril(Kg Kb^T)
//                 with Qg = q 2^g2, Kg = k 2^g2, Kb = k 2^-g2: the per-channel gate
//                 2^(g2_i - g2_j) split through the chunk start, one tcgen05 MMA
//                 (M = 128: [Qg; Kg] stacked, N = 64, K = dk).  This split keeps
//                 every factor at most 2^R with R = max |g2| over the chunk; when R
//                 exceeds kSafeRange (100) the grams are formed exactly in fp32 SIMT
//                 with one exp2 per (i, j, d), exponent g2_i - g2_j <= 0 (ALGORITHM.md,
//                 "The numerics law").
//                 Akk = (I + L)^-1: blocked unit-lower-triangular inverse in fp32
//                 (16 x 16 diagonal blocks by substitution, then two doubling
//                 steps to 32 x 32 and 64 x 64).
//                 w = Akk diag(beta) Kg,  u = Akk diag(beta) v    (tcgen05, N = dk / dv)
//                 kg = k 2^(G - g2),  qg = q 2^g2,  decay = 2^G
//     The results go to the workspace as ready-made MMA operand tiles.
//
//   scan kernel, one CTA per (sequence, value head, 32 value columns):
//     Stage 3+4   v' = u - w h;   o = scale (qg h + Aqk v');   h = Diag(2^G) h + kg^T v'
//                 [w; qg] h    : one MMA, M = 128, N = 32, K = dk
//                 kg^T v'      : one MMA, M = 128 (= dk, zero-padded for dk = 64)
//                 Aqk v'       : accumulated onto the qg h rows of the first MMA
//     h stays in registers in fp32 (thread d owns row d); a bf16 copy in shared
//     memory is the next chunk's MMA operand.  Operand tiles of the next chunks
//     stream in by bulk async copies while the current chunk computes.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_chunk_layout.cuh"

#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>

namespace kda {
namespace {

using namespace tc;

// Whether a chunk continues the scan of the chunk before it: not a sequence's
// first chunk, nor the first chunk of the second segment of a split launch or of
// a pipelined launch's part (those scans start from a given state).  A prep
// launch of a pipelined call covers one part, which starts at prep_c0.
__device__ __forceinline__ bool continues(const ChunkArgs &p, int cl, int seq_chunks) {
    return cl > 0 && !(p.split && cl == (seq_chunks + 1) / 2) &&
           !(p.pipe.parts > 0 && cl == p.prep_c0);
}

// A prep launch's units: every chunk slot of every value head, or (a pipelined
// launch's part, dense input) chunks [prep_c0, prep_c1) of every sequence.
// Units run value head by value head, chunks in order within a sequence.
__host__ __device__ __forceinline__ int64_t prep_units(const ChunkArgs &p) {
    const int64_t per_hv = p.prep_c1 > p.prep_c0 ? (int64_t)p.B * (p.prep_c1 - p.prep_c0) : p.slots;
    return per_hv * p.HV;
}
__device__ __forceinline__ void prep_unit(const ChunkArgs &p, int64_t unit, int &hv, int64_t &gc) {
    if (p.prep_c1 > p.prep_c0) {
        const int w = p.prep_c1 - p.prep_c0;
        const int64_t per_hv = (int64_t)p.B * w;
        hv = (int)(unit / per_hv);
        const int64_t r = unit - hv * per_hv;
        gc = (r / w) * ((p.T + kBT - 1) / kBT) + p.prep_c0 + (r % w);
    } else {
        hv = (int)(unit / p.slots);
        gc = unit % p.slots;
    }
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}


// ============================================================== prep kernel
// Shared memory of the prep kernel.  The kernel declares no static shared
// memory, so the dynamic region starts 1024-byte aligned (checked at run time)
// and every offset below is a constant.
//
// Inputs arrive by TMA tensor copies with 128-byte swizzling, directly in the
// layout the tensor cores read (sdesc_sw128): the [q; k] tile ("ag") and the
// [kb; kg of the previous chunk] tile ("kbx") each hold 128 rows in KK / 64
// column blocks of 16 KB (rows 0..63 in the first 8 KB, rows 64..127 in the
// second), and g lands in g2 as KK / 32 boxes of [64 rows][32 fp32].  The
// elementwise pass then works in place.
// With dk = 128 the solve's fp32 matrices are stored split by rows: L (rows 0..31
// and 32..63) in the two kb pieces of kbx (which the split grams of a chunk with
// a wide gate range never read), T and P in the two previous-kg pieces once the
// gram MMA has read them, Akk in the two q pieces of ag.
// Buffer plan when dk = 128 and dv <= 128 ("pref"): after the elementwise pass
// v goes into the second half of g2 and the next unit's g channels 0..63 into the
// first half; Akk diag(beta) goes over the second q piece.  The k rows of ag are
// free after the W MMA (the next unit's k goes there), the q rows and v after the
// u MMA (the next unit's q and its g channels 64..127).  Otherwise v and
// Akk diag(beta) sit in g2 and every copy of the next unit starts after the u
// MMA.
template <int KK>
struct PrepSmem {
    static constexpr uint32_t kBlk = 16384;                     // column block of ag / kbx
    static constexpr uint32_t beta = 0;                         // fp32 [64]
    static constexpr uint32_t dprev = beta + 64 * 4;            // fp32 [128]: 2^G of the previous chunk
    static constexpr uint32_t eg = dprev + 128 * 4;             // fp32 [128]: 2^G
    static constexpr uint32_t gv = eg + 128 * 4;                // fp32 [128]: G
    static constexpr uint32_t bars = gv + 128 * 4;              // 4 mbarriers
    static constexpr uint32_t misc = bars + 4 * 8;              // tslot, range bits
    static constexpr uint32_t cur = 1856;                       // two unit cursors (UnitCur, 40 B)
    static constexpr uint32_t ag = 2048;                        // [q; k] tile
    static constexpr uint32_t kbx = ag + (KK / 64) * kBlk;      // [kb; previous kg] tile
    static constexpr uint32_t g = kbx + (KK / 64) * kBlk;       // fp32 [64][KK] g2 (swizzled); later v + AB
    static constexpr uint32_t g_need0 = 64 * KK * 4;
    // the exact grams' B operand (32 k rows, 128-byte swizzled), right after g2: dead
    // space then (v and the tiles after g2 are written later in the unit)
    static constexpr uint32_t khat = g + g_need0;
    static constexpr uint32_t khat_end = khat + 32 * KK * 2;
    static_assert(misc + 8 <= cur && cur + 96 <= ag && g % 1024 == 0 && khat % 1024 == 0,
                  "prep layout");
    __host__ __device__ static constexpr uint32_t g_bytes(int VV) {
        return g_need0 > 64u * VV * 2 + 64 * 64 * 2 ? g_need0 : 64u * VV * 2 + 64 * 64 * 2;
    }
    __host__ __device__ static constexpr uint32_t extra(int VV) { return g + g_bytes(VV); }
    // L fp32 [64][64], T fp32 [32][32], P bf16 tile [64][64], Akk fp32 [64][64].
    // dk = 128 reuses kbx and the q pieces of ag for them (L and Akk split by rows,
    // the second half kBlk further on); dk = 64 keeps them after g2.
    static constexpr bool big = KK == 128;
    __host__ __device__ static constexpr uint32_t lbuf(int VV) { return big ? kbx : extra(VV); }
    __host__ __device__ static constexpr uint32_t tbuf(int VV) {
        return big ? kbx + 8192 : lbuf(VV) + 64 * 64 * 4;
    }
    __host__ __device__ static constexpr uint32_t pbuf(int VV) {
        return big ? kbx + kBlk + 8192 : tbuf(VV) + 32 * 32 * 4;
    }
    __host__ __device__ static constexpr uint32_t abuf(int VV) {
        return big ? ag : pbuf(VV) + 64 * 64 * 2;
    }
    __host__ __device__ static constexpr uint32_t used(int VV) {
        return big ? (extra(VV) > khat_end ? extra(VV) : khat_end)
                   : (abuf(VV) + 64 * 64 * 4 > khat_end ? abuf(VV) + 64 * 64 * 4 : khat_end);
    }
    // Floor so that at most two CTAs (256 TMEM columns each) share an SM.
    __host__ __device__ static constexpr uint32_t total(int VV) {
        return used(VV) > 80 * 1024 ? used(VV) : 80 * 1024;
    }
};

// Where a prep unit is: written by thread 0 for the next unit while the current
// one runs (two slots, alternating), read by every thread.
struct UnitCur {
    long long unit, gc;
    int hv, b, r0, nr, cl, ncs;
};
static_assert(sizeof(UnitCur) <= 48, "two cursors fit their area");

// The TMA descriptors of one prep launch: q and k as [B*T rows][H][K] bf16 with
// 64 x 64 boxes, g as [B*T rows][HV][K] fp32 with 64 x 32 boxes, v as
// [B*T rows][HV][V] bf16 with 64 x 64 boxes (encoded when dv is 64 or 128, unused
// otherwise), 128-byte swizzle.
struct PrepMaps {
    CUtensorMap q, k, g, v;
};

// One 3-D tensor-map tile load into shared memory, completion counted in bytes
// on `bar` (coordinates innermost first: channel, head, row).
__device__ __forceinline__ void tma_load3(void *dst, const CUtensorMap *map, int c0, int c1,
                                          int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

// fp32 index of g2 element (r, c): box c / 32 of [64][32] fp32, 128-byte rows,
// 16-byte chunk (c % 32) / 4 stored at chunk position ((c % 32) / 4) ^ (r % 8).
__device__ __forceinline__ int gsw(int r, int c) {
    return (c >> 5) * 2048 + r * 32 + ((((c >> 2) & 7) ^ (r & 7)) << 2) + (c & 3);
}
// Byte offset of element (r, c) / of the 16-byte chunk holding channels
// c .. c + 7 (c a multiple of 8) in the ag and kbx tiles.
__device__ __forceinline__ uint32_t qk_off(int r, int c) { return sw128_off(r, c, 16384); }

// fp32 [rows][W] with the 16-byte column group XORed by (row & 7): eight
// consecutive rows at the same columns fall in distinct banks.
template <int W>
__device__ __forceinline__ int fsw(int r, int c) {
    return r * W + ((((c >> 2) ^ r) & 7) | ((c >> 2) & ~7)) * 4 + (c & 3);
}
template <int W>
__device__ __forceinline__ float4 ld4(const float *b, int r, int c) {
    return *reinterpret_cast<const float4 *>(b + fsw<W>(r, c));
}
template <int W>
__device__ __forceinline__ void st4(float *b, int r, int c, float4 v) {
    *reinterpret_cast<float4 *>(b + fsw<W>(r, c)) = v;
}
__device__ __forceinline__ void fma4(float4 &s, float a, const float4 &x) {
    s.x = fmaf(a, x.x, s.x);
    s.y = fmaf(a, x.y, s.y);
    s.z = fmaf(a, x.z, s.z);
    s.w = fmaf(a, x.w, s.w);
}

__device__ __forceinline__ float4 neg4(float4 v) { return make_float4(-v.x, -v.y, -v.z, -v.w); }

// L and Akk (fp32 [64][64], fsw<64> layout) with dk = 128 are split by rows: rows
// 0..31 at +0, rows 32..63 at +16 KB (two 8 KB pieces of kbx or ag).  Float index
// of (r, c).
template <bool SPLIT>
__device__ __forceinline__ int akk_idx(int r, int c) {
    return fsw<64>(r, c) + (SPLIT ? (r >> 5) * 2048 : 0);
}
template <bool SPLIT>
__device__ __forceinline__ float4 lda4(const float *A, int r, int c) {
    return *reinterpret_cast<const float4 *>(A + akk_idx<SPLIT>(r, c));
}
template <bool SPLIT>
__device__ __forceinline__ void sta4(float *A, int r, int c, float4 v) {
    *reinterpret_cast<float4 *>(A + akk_idx<SPLIT>(r, c)) = v;
}
// s += P[r][m] Q[m][c..c+3] over 16 columns m, P = L (64 wide) or Akk, Q = Akk or
// T (32 wide): the strip products of the blocked solve.
template <bool SPLIT>
__device__ __forceinline__ void strip_la(float4 &s, const float *L, int pr, int pc, const float *A,
                                         int qr, int qc) {
#pragma unroll
    for (int m4 = 0; m4 < 16; m4 += 4) {
        const float4 a = lda4<SPLIT>(L, pr, pc + m4);
        fma4(s, a.x, lda4<SPLIT>(A, qr + m4, qc));
        fma4(s, a.y, lda4<SPLIT>(A, qr + m4 + 1, qc));
        fma4(s, a.z, lda4<SPLIT>(A, qr + m4 + 2, qc));
        fma4(s, a.w, lda4<SPLIT>(A, qr + m4 + 3, qc));
    }
}
template <bool SPLIT>
__device__ __forceinline__ void strip_at(float4 &s, const float *A, int pr, int pc, const float *T,
                                         int qr, int qc) {
#pragma unroll
    for (int m4 = 0; m4 < 16; m4 += 4) {
        const float4 a = lda4<SPLIT>(A, pr, pc + m4);
        fma4(s, a.x, ld4<32>(T, qr + m4, qc));
        fma4(s, a.y, ld4<32>(T, qr + m4 + 1, qc));
        fma4(s, a.z, ld4<32>(T, qr + m4 + 2, qc));
        fma4(s, a.w, ld4<32>(T, qr + m4 + 3, qc));
    }
}

// The exact gated grams of a chunk whose gate range is too wide to split (the comment
// above its call site), out of line: cold code kept away from the prep's hot path.
// Pairs j < i in different 4-row blocks: the gate is split at a block boundary e
// between them, 2^(g2_i - g2_e) 2^(g2_e - g2_j), both exponents <= 0, so the pair is
// the product of two bounded operands and goes to the tensor cores.  Four M = 64,
// N = 32 MMAs, one per level of a halving of the chunk: level s (32, 16, 8, 4) pairs
// the rows of the second half of every 2s-row block (A: their q rows, then their k
// rows, scaled to the block's midpoint e) with the rows of its first half (B: k rows
// scaled from e).  A lives in rows 0..63 of kbx (free in this path until L is written
// there), B in khat.  Products of rows and columns of different blocks are formed
// too and discarded (every factor is at most 1, so they stay finite).  What is left,
// the 4 x 4 diagonal blocks, takes 2^(g2_i - g2_j) itself per channel on the CUDA
// cores.
// aqk: the unit's Aqk tile; sL: L (fp32, akk_idx layout); sKB: kbx; sKH: khat;
// tmem: the CTA's accumulator (columns 0..127 used here); bar, phase: the MMA
// barrier and its phase (four completions consumed).
template <int KK, bool kSplitA>
__device__ __noinline__ void exact_grams(const unsigned char *sAG, const float *sG2,
                                         const float *sBeta, float *sL, unsigned char *sKB,
                                         unsigned char *sKH, unsigned char *aqk,
                                         const uint32_t tmem, uint64_t *bar, uint32_t phase,
                                         int32_t *status, const int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    // ---- the pairs in different 4-row blocks, one MMA per level
#pragma unroll 1
    for (int grp = 0; grp < 4; ++grp) {
        const int lg = 5 - grp, hsz = 1 << lg;  // level: half-blocks of hsz rows
        // A rows r: side r / 32 (q, then k); row i of the chunk: the second half of
        // block rr / hsz; boundary e: that block's midpoint
#pragma unroll 1
        for (int it = 0; it < KK / 32; ++it) {
            const int idx = tid + it * 256, l = idx & 31, w = idx >> 5;
            const int r = (w & 7) * 8 + (l & 7), c = ((w >> 3) * 4 + (l >> 3)) * 8;
            const int rr = r & 31;
            const int e = ((rr >> lg) << (lg + 1)) + hsz, i = e + (rr & (hsz - 1));
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(sAG + qk_off((r >> 5) * 64 + i, c)), f);
            const float4 gi0 = *reinterpret_cast<const float4 *>(sG2 + gsw(i, c));
            const float4 gi1 = *reinterpret_cast<const float4 *>(sG2 + gsw(i, c + 4));
            const float4 ge0 = *reinterpret_cast<const float4 *>(sG2 + gsw(e, c));
            const float4 ge1 = *reinterpret_cast<const float4 *>(sG2 + gsw(e, c + 4));
            f[0] *= ex2_ftz(gi0.x - ge0.x); f[1] *= ex2_ftz(gi0.y - ge0.y);
            f[2] *= ex2_ftz(gi0.z - ge0.z); f[3] *= ex2_ftz(gi0.w - ge0.w);
            f[4] *= ex2_ftz(gi1.x - ge1.x); f[5] *= ex2_ftz(gi1.y - ge1.y);
            f[6] *= ex2_ftz(gi1.z - ge1.z); f[7] *= ex2_ftz(gi1.w - ge1.w);
            *reinterpret_cast<uint4 *>(sKB + qk_off(r, c)) = pack8(f);
        }
        // B rows n: k row j of the first half of block n / hsz, boundary e its midpoint
#pragma unroll 1
        for (int it = 0; it < KK / 64; ++it) {
            const int idx = tid + it * 256, l = idx & 31, w = idx >> 5;
            const int n = (w & 3) * 8 + (l & 7), c = ((w >> 2) * 4 + (l >> 3)) * 8;
            const int e = ((n >> lg) << (lg + 1)) + hsz, j = e - hsz + (n & (hsz - 1));
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(sAG + qk_off(64 + j, c)), f);
            const float4 gj0 = *reinterpret_cast<const float4 *>(sG2 + gsw(j, c));
            const float4 gj1 = *reinterpret_cast<const float4 *>(sG2 + gsw(j, c + 4));
            const float4 ge0 = *reinterpret_cast<const float4 *>(sG2 + gsw(e, c));
            const float4 ge1 = *reinterpret_cast<const float4 *>(sG2 + gsw(e, c + 4));
            f[0] *= ex2_ftz(ge0.x - gj0.x); f[1] *= ex2_ftz(ge0.y - gj0.y);
            f[2] *= ex2_ftz(ge0.z - gj0.z); f[3] *= ex2_ftz(ge0.w - gj0.w);
            f[4] *= ex2_ftz(ge1.x - gj1.x); f[5] *= ex2_ftz(ge1.y - gj1.y);
            f[6] *= ex2_ftz(ge1.z - gj1.z); f[7] *= ex2_ftz(ge1.w - gj1.w);
            *reinterpret_cast<uint4 *>(sKH + sw128_off(n, c, 32 * 128)) = pack8(f);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t a0 = smem_addr(sKB), b0 = smem_addr(sKH);
            const uint32_t idn = idesc_bf16(64, 32, false, false);
#pragma unroll 1
            for (int kk = 0; kk < KK / 16; ++kk) {
                const uint32_t ko = (kk & 3) * 32;
                mma_bf16(tmem + 32 * grp, sdesc_sw128(a0 + (kk >> 2) * 16384 + ko, 16, 1024),
                         sdesc_sw128(b0 + (kk >> 2) * (32 * 128) + ko, 16, 1024), idn, kk > 0);
            }
            mma_commit(bar);
            if (!mbar_wait(bar, phase & 1, kWaitNs)) report(status, KDA_DEVICE_TIMEOUT);
        }
        ++phase;
        __syncthreads();
        tc_fence_after();
    }
    // ---- their results (L's place in kbx is free now).  An M = 64 result's row r sits
    // in TMEM lane 32 (r / 16) + r % 16; this thread holds row r, columns 16 hs .. + 15
    // of levels w / 4 and w / 4 + 2, and stores the columns of its own block, four at
    // a time (contiguous in j)
    {
        const int quad = warp & 3, hs = lane >> 4;
        const int r = 16 * quad + (lane & 15), rr = r & 31;
#pragma unroll 1
        for (int g2 = 0; g2 < 2; ++g2) {
            const int grp = (warp >> 2) + 2 * g2, lg = 5 - grp, hsz = 1 << lg;
            float d[16];
            tmem_ld16x2_16<16>(tmem_at(tmem, 32 * quad, 32 * grp), d);
            const int e = ((rr >> lg) << (lg + 1)) + hsz, i = e + (rr & (hsz - 1));
#pragma unroll
            for (int t = 0; t < 16; t += 4) {
                const int n = 16 * hs + t;
                if ((n >> lg) != (rr >> lg)) continue;
                const int j = e - hsz + (n & (hsz - 1));
                if (quad < 2) {
                    __nv_bfloat162 h2[2] = {__floats2bfloat162_rn(d[t], d[t + 1]),
                                            __floats2bfloat162_rn(d[t + 2], d[t + 3])};
                    *reinterpret_cast<uint2 *>(aqk + tile_off(i, j, 64)) =
                        *reinterpret_cast<const uint2 *>(h2);
                } else {
                    const float b = sBeta[i];
                    sta4<kSplitA>(sL, i, j, make_float4(b * d[t], b * d[t + 1], b * d[t + 2], b * d[t + 3]));
                }
            }
        }
    }
    // ---- the diagonal blocks.  lane l holds the channel pairs (2 l + 64 m, 2 l + 64 m
    // + 1), m < dk / 64.  Its shared-memory offsets, from the swizzles: the q/k tile
    // (qk_off) at m * 16 KB + r * 128 + ((((l / 4) % 8) ^ (r % 8)) << 4) + 4 (l % 4), the
    // k rows 8 KB further; g2 (gsw) at (l / 16 + 2 m) * 8 KB + 4 r (32 r floats) + the
    // 16-byte chunk ((l / 2) % 8) ^ (r % 8) + 8 (l % 2) bytes.  Addressed in the shared
    // window.
    constexpr int CP = KK / 64;
    const uint32_t ag = (uint32_t)__cvta_generic_to_shared(sAG);
    const uint32_t g2b = (uint32_t)__cvta_generic_to_shared(sG2);
    const int L1 = (lane >> 2) & 7, L0 = (lane & 3) * 4;
    const int G1 = (lane >> 1) & 7, G0 = (lane & 1) * 8 + (lane >> 4) * 8192;
    const auto qrow = [&](int r) { return ag + (uint32_t)(r * 128 + ((L1 ^ (r & 7)) << 4) + L0); };
    const auto grow = [&](int r) { return g2b + (uint32_t)(r * 128 + ((G1 ^ (r & 7)) << 4) + G0); };
    const auto bf2 = [](uint32_t a) {
        uint32_t x;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(x) : "r"(a));
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x));
    };
    const auto f2 = [](uint32_t a) {
        float2 x;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(x.x), "=f"(x.y) : "r"(a));
        return x;
    };
    // the reduction and the store of row i, columns j0 .. j0 + 3: the eight sums (Aqk
    // and the k gram of the four columns) reduced over the warp by halving exchanges
    // (nine shuffles), lane 4 o ending with sum o
    const auto emit = [&](int i, int j0, const float (&v)[8]) {
        const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
        float w[4], x[2];
#pragma unroll
        for (int t = 0; t < 4; ++t)
            w[t] = (b4 ? v[4 + t] : v[t]) + __shfl_xor_sync(0xffffffffu, b4 ? v[t] : v[4 + t], 16);
#pragma unroll
        for (int t = 0; t < 2; ++t)
            x[t] = (b3 ? w[2 + t] : w[t]) + __shfl_xor_sync(0xffffffffu, b3 ? w[t] : w[2 + t], 8);
        float y = (b2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, b2 ? x[0] : x[1], 4);
        y += __shfl_xor_sync(0xffffffffu, y, 2);
        y += __shfl_xor_sync(0xffffffffu, y, 1);
        if ((lane & 3) == 0) {
            const int j = j0 + 2 * b3 + b2;  // sum 4 b4 + 2 b3 + b2
            if (!b4)
                *reinterpret_cast<__nv_bfloat16 *>(aqk + tile_off(i, j, 64)) =
                    __float2bfloat16_rn(j <= i ? y : 0.f);
            else
                sL[akk_idx<kSplitA>(i, j)] = j < i ? sBeta[i] * y : 0.f;
        }
    };
    // warp w takes rows 8 b + w, b < 8, the row's channels in registers, columns
    // 4 floor(i / 4) .. i of its 4-row block; zeros above the diagonal
#pragma unroll 1
    for (int s = 0; s < 8; ++s) {
        const int i = 8 * s + warp;
        float2 qi[CP], ki[CP], gi[CP];
        const uint32_t qa = qrow(i), ga = grow(i);
#pragma unroll
        for (int m = 0; m < CP; ++m) {
            qi[m] = bf2(qa + m * 16384);
            ki[m] = bf2(qa + 8192 + m * 16384);
            gi[m] = f2(ga + m * 16384);
        }
#pragma unroll 1
        {
            const int j0 = i & ~3;
            float v[8];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                float aq = 0.f, ak = 0.f;
                const uint32_t kja = qrow(j0 + jj) + 8192, gja = grow(j0 + jj);
#pragma unroll
                for (int m = 0; m < CP; ++m) {
                    // columns past i may overflow here; their sums are never stored
                    const float2 k2 = bf2(kja + m * 16384), g2 = f2(gja + m * 16384);
                    const float kx = k2.x * ex2_ftz(gi[m].x - g2.x);
                    const float ky = k2.y * ex2_ftz(gi[m].y - g2.y);
                    aq = fmaf(qi[m].y, ky, fmaf(qi[m].x, kx, aq));
                    ak = fmaf(ki[m].y, ky, fmaf(ki[m].x, kx, ak));
                }
                v[jj] = aq;
                v[4 + jj] = ak;
            }
            emit(i, j0, v);
        }
        for (int j = i + 1 + lane; j < 64; j += 32) {
            *reinterpret_cast<__nv_bfloat16 *>(aqk + tile_off(i, j, 64)) = __float2bfloat16_rn(0.f);
            sL[akk_idx<kSplitA>(i, j)] = 0.f;
        }
    }
}

// ACT: the gate activation (kda_activation.A_log) is compiled in.
// PADK: K < dk, the channels past K are zero (TMA fills them; otherwise K == dk
// and the channel count is a compile-time constant).
template <int KK, bool ACT, bool PADK>
__global__ void __launch_bounds__(256, 2)
    chunk_prep_tc_kernel(ChunkArgs p, const __grid_constant__ PrepMaps maps) {
    const int Kc = PADK ? p.K : KK;  // the input's channels
    using S = PrepSmem<KK>;
    constexpr bool kSplitA = S::big;
    const int VV = p.V;
    extern __shared__ __align__(1024) unsigned char sm[];
    float *sBeta = reinterpret_cast<float *>(sm + S::beta);
    float *sDprev = reinterpret_cast<float *>(sm + S::dprev);
    float *sEG = reinterpret_cast<float *>(sm + S::eg);   // 2^G per channel
    float *sGv = reinterpret_cast<float *>(sm + S::gv);   // G per channel
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::bars);
    uint64_t &bar = bars[0], &bar_g = bars[1], &bar_qk = bars[2], &bar_v = bars[3];
    uint32_t &tslot = *reinterpret_cast<uint32_t *>(sm + S::misc);
    int &sRangeBits = *reinterpret_cast<int *>(sm + S::misc + 4);
    UnitCur *curs = reinterpret_cast<UnitCur *>(sm + S::cur);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr uint32_t kCols = 256;
    // The swizzled TMA destinations need a 1024-byte aligned base, which a kernel
    // without static shared memory has; checked once, never assumed silently.
    if (smem_addr(sm) & 1023u) {
        if (tid == 0) report(p.status, KDA_DEVICE_INTERNAL);
        return;
    }
    const bool pref = KK == 128 && VV <= 128;  // see PrepSmem
    // v by TMA (64 x 64 boxes, 128-byte swizzle) when dv is 64 or 128 with the pref
    // plan; 16-byte cp.async copies into the plain core-matrix layout otherwise
    const bool vtma = pref && (VV & 63) == 0;

    unsigned char *sAG = sm + S::ag;
    unsigned char *sKB = sm + S::kbx;
    float *sG2 = reinterpret_cast<float *>(sm + S::g);
    // v: with the pref plan in the second half of g2
    unsigned char *sV = pref ? sm + S::g + 64 * 64 * 4 : sm + S::g;
    constexpr uint32_t v_half = 0;  // extra gap before v's rows 32..63 (none)
    // Akk diag(beta), twice (rows 0..63 and 64..127 of the M = 128 A operand), in
    // L's place once the solve is done with L and T
    unsigned char *sAB = sm + S::lbuf(VV);
    float *sL = reinterpret_cast<float *>(sm + S::lbuf(VV));    // after the gram MMA
    float *sT = reinterpret_cast<float *>(sm + S::tbuf(VV));
    unsigned char *sPB = sm + S::pbuf(VV);
    float *sA = reinterpret_cast<float *>(sm + S::abuf(VV));

    const TcLayout Lo = tc_layout(KK, VV, p.bwd);
    if (warp == 0) {
        tmem_alloc(&tslot, kCols);
        tmem_relinquish();
    }
    // Persistent: the CTA takes a contiguous range of units in (value head,
    // chunk) order, so consecutive units are usually consecutive chunks of one
    // head.  The previous chunk's kg tile and 2^G then stay in shared memory
    // ("carry") instead of being re-derived from its k and g.
    const int64_t total = prep_units(p);
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t ubeg = (int64_t)blockIdx.x * per;
    const int64_t uend = ubeg + per < total ? ubeg + per : total;
    // Thread 0 only: the first unit at or after u that has rows, into *c.
    auto find = [&](int64_t u, UnitCur *c) {
        for (; u < uend; ++u) {
            int hv_, b_, r0_, nr_, cl_, ns_, nc_;
            int64_t gc_;
            prep_unit(p, u, hv_, gc_);
            if (locate_chunk(p, gc_, b_, r0_, nr_, cl_, &ns_, &nc_)) {
                c->unit = u; c->gc = gc_; c->hv = hv_; c->b = b_; c->r0 = r0_; c->nr = nr_;
                c->cl = cl_; c->ncs = nc_;
                return;
            }
        }
        c->unit = uend;
    };
    // Thread 0 only: the unit after *c.  Dense inputs step without divisions:
    // chunk cl of sequence b runs over [c0, c1) (a pipelined part) or all chunks.
    auto advance = [&](const UnitCur *c, UnitCur *n) {
        if (c->unit + 1 >= uend) {
            n->unit = uend;
            return;
        }
        if (__builtin_expect(p.cu != nullptr, 0)) {
            find(c->unit + 1, n);
            return;
        }
        const int ntc = (p.T + kBT - 1) / kBT;
        const int c0 = p.prep_c1 > p.prep_c0 ? p.prep_c0 : 0;
        const int c1 = p.prep_c1 > p.prep_c0 ? p.prep_c1 : ntc;
        int hv_ = c->hv, b_ = c->b, cl_ = c->cl + 1;
        if (cl_ >= c1) {
            cl_ = c0;
            if (++b_ >= p.B) {
                b_ = 0;
                ++hv_;
            }
        }
        n->unit = c->unit + 1;
        n->gc = (int64_t)b_ * ntc + cl_;
        n->hv = hv_; n->b = b_; n->cl = cl_; n->ncs = ntc;
        n->r0 = cl_ * kBT;
        n->nr = min(kBT, p.T - n->r0);
    };
    // TMA copies of a unit's g rows (into g2) and q / k rows (into ag); issued by
    // thread 0 after a fence that orders the buffers' earlier generic-proxy
    // accesses before the copies' writes.
    // g goes in two halves of KK / 64 boxes each (two arrivals on bar_g per unit).
    auto issue = [&](const UnitCur *c, bool do_g_lo, bool do_g_hi, bool do_q, bool do_k) {
        const int row = c->b * p.T + c->r0;
        const int h_ = c->hv / (p.HV / p.H);
        fence_async_smem();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (half ? !do_g_hi : !do_g_lo) continue;
            mbar_arrive_expect_tx(&bar_g, 64 * KK * 2);
#pragma unroll
            for (int x = half * (KK / 64); x < (half + 1) * (KK / 64); ++x)
                tma_load3(sm + S::g + x * 8192, &maps.g, x * 32, c->hv, row, &bar_g);
        }
        if (do_q) {
            mbar_arrive_expect_tx(&bar_qk, 64 * KK * 2);
#pragma unroll
            for (int x = 0; x < KK / 64; ++x)
                tma_load3(sAG + x * S::kBlk, &maps.q, x * 64, h_, row, &bar_qk);
        }
        if (do_k) {
            mbar_arrive_expect_tx(&bar_qk, 64 * KK * 2);
#pragma unroll
            for (int x = 0; x < KK / 64; ++x)
                tma_load3(sAG + x * S::kBlk + 8192, &maps.k, x * 64, h_, row, &bar_qk);
        }
    };
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init(&bar_g, 2);   // the two halves of g arrive separately
        mbar_init(&bar_qk, 2);  // the q copies and the k copies arrive separately
        mbar_init(&bar_v, 1);
        mbar_fence_init();
        sRangeBits = 0;
        find(ubeg, &curs[0]);
        if (curs[0].unit < uend) issue(&curs[0], true, true, true, true);
    }
    if (PADK && tid < 128) sDprev[tid] = 1.f;  // channels past K keep 1 (their W columns are zero)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    uint32_t phase = 0, ph_in = 0;  // MMA barrier phases; input copies (g and q/k) per unit
    uint32_t ph_v = 0;              // v copies by TMA (one per unit)
    int slot = 0;
    int prev_hv = -1;
    int64_t prev_gc = -1;
    while (true) {
    const UnitCur *cur = &curs[slot];
    const UnitCur *nxt = &curs[slot ^ 1];  // written below by thread 0, read after a barrier
    const int64_t unit = cur->unit;
    if (unit >= uend) break;
    const int hv = cur->hv, b = cur->b, r0 = cur->r0, nr = cur->nr, cl = cur->cl;
    const int64_t gc = cur->gc;
    if (tid == 0) advance(cur, &curs[slot ^ 1]);
    const bool halo = continues(p, cl, cur->ncs);  // the previous chunk's state feeds this one
    const bool carry = halo && prev_hv == hv && prev_gc == gc - 1;
    const int h = hv / (p.HV / p.H);
    unsigned char *U = static_cast<unsigned char *>(p.units) + unit_index(p, gc, hv) * Lo.stride;

    // ---- 1. the previous chunk's k rows when they are not carried over (the
    // run's first unit), 16-byte chunks into the swizzled kbx rows 64..127
    const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(p.beta);
    const size_t row0 = (size_t)b * p.T + r0;
    const int VG8 = VV / 8;
    // beta in a register now, into shared memory after the gates: its load
    // latency overlaps everything up to there
    float bet = (tid < 64 && tid < nr) ? to_f32(beta[(row0 + tid) * p.HV + hv]) : 0.f;
    if (p.act.beta_scale > 0.f && tid < 64 && tid < nr)
        bet = beta_activate<__nv_bfloat16>(bet, p.act.beta_scale);
    // the gate activation's per-channel constants (thread d and 128 + d: channel d)
    constexpr bool gate_act = ACT;
    const float neg_a = gate_act ? gate_neg_a(p.act, hv) : 0.f;
    const float gbias = gate_act && (tid & 127) < Kc ? gate_bias(p.act, hv, tid & 127, Kc) : 0.f;
    if (__builtin_expect(halo && !carry, 0)) {
#pragma unroll 1
        for (int it = 0; it < KK / 32; ++it) {
            const int idx = tid + it * 256, i = idx & 63, c = (idx >> 6) * 8;
            if (c < Kc)
                cp_async16(sKB + qk_off(64 + i, c), k + ((row0 - 64 + i) * p.H + h) * Kc + c);
            else
                *reinterpret_cast<uint4 *>(sKB + qk_off(64 + i, c)) = make_uint4(0, 0, 0, 0);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");

    // ---- 2. Stage 1.  While the copies are in flight, the previous chunk's gate
    // rows are prefetched into L2; once its k rows have landed, thread 128 + d
    // turns channel d of them into kg' = k' 2^(G' - g2'_j) (a reverse running sum)
    // and records 2^G'.  Thread d < dk then forms g2 for channel d in place in
    // shared memory (rows past the end keep G).
    const size_t grs = (size_t)p.HV * Kc;
    const int dh = tid - 128;
    const bool halo_thread = halo && !carry && tid >= 128 && dh < Kc;
    if (__builtin_expect(halo && !carry, 0) && tid >= 128 && (dh & ~31) < Kc) {
        // the 64 gate rows of this warp's 32 channels into L2 now (two rows per
        // lane, no registers held), read after the barrier below
        const float *gp = p.g + ((row0 - 64) * p.HV + hv) * Kc + (dh & ~31);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(gp + lane * grs));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(gp + (lane + 32) * grs));
    }
    if (tid < 64) sBeta[tid] = bet;
    // One thread polls each completion; the others wait at the barrier after it.
    if (tid == 0 && !mbar_wait(&bar_g, ph_in & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // the previous chunk's k rows, L2-normalised first when asked (threads 128..191,
    // one row each)
    if (__builtin_expect(p.l2norm && halo && !carry, 0)) {
        if (tid >= 128 && tid < 192) {
            const int row = tid - 64;  // rows 64..127 of kbx
            float ss = 0.f;
#pragma unroll 1
            for (int c = 0; c < KK; c += 8) {
                float f[8];
                unpack8(*reinterpret_cast<const uint4 *>(sKB + qk_off(row, c)), f);
#pragma unroll
                for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
            }
            const float rsn = 1.f / sqrtf(ss + 1e-6f);
#pragma unroll 1
            for (int c = 0; c < KK; c += 8) {
                uint4 *at = reinterpret_cast<uint4 *>(sKB + qk_off(row, c));
                float f[8];
                unpack8(*at, f);
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] *= rsn;
                *at = pack8(f);
            }
        }
        __syncthreads();
    }
    if (__builtin_expect(halo_thread, 0)) {
        // ... then it becomes its kg (one channel per halo thread), while threads
        // 0..127 run the cumsum below: row j is scaled by 2^(sum of the gates
        // after it), G' - g2'_j for per-token gates, G' - g'_j for a cumsum input.
        // eight rows at a time from the last, the next eight loaded meanwhile
        const float *gp = p.g + ((row0 - 64) * p.HV + hv) * Kc + dh;
        const float Gc = gate_act ? 0.f : __ldg(gp + 63 * grs);  // G' when g holds the cumsum
        float cur[8], nxt[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) cur[j] = __ldg(gp + (56 + j) * grs);
        float acc = 0.f;
#pragma unroll 1
        for (int j0 = 56; j0 >= 0; j0 -= 8) {
            const int jn = j0 > 0 ? j0 - 8 : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) nxt[j] = __ldg(gp + (jn + j) * grs);
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                __nv_bfloat16 *pk = reinterpret_cast<__nv_bfloat16 *>(sKB + qk_off(64 + j0 + j, dh));
                const float ex = p.g_is_cumsum ? Gc - cur[j] : acc;
                *pk = __float2bfloat16_rn(__bfloat162float(*pk) * ex2_ftz(ex));
                float gj = cur[j];
                if (gate_act) gj = neg_a * softplus_f(gj + gbias);
                acc = fmaf(p.g_scale, gj, acc);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
        }
        sDprev[dh] = ex2_ftz(p.g_is_cumsum ? Gc : acc);
    }
    // thread d < dk: channel d's chunk-local cumsum in place (rows past the end keep
    // G).  Per-token gates: all 64 rows in registers, four independent 16-row
    // running sums, then each quarter offset by the totals before it.  Otherwise
    // (activation or a cumsum input) 16 rows at a time, each block's loads issued
    // before the previous block's stores: a store to the tile between two of its
    // loads would order them and put the shared-memory latency on every row.
    if (tid < KK) {
        float acc = 0.f, rng = 0.f;
        const bool live = tid < Kc;  // channels past K keep a zero gate
        if (!gate_act && !p.g_is_cumsum) {
            float x[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) x[i] = sG2[gsw(i, tid)];
            float tot[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float a = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int i = 16 * q4 + j;
                    a = fmaf(p.g_scale, (i < nr && live) ? x[i] : 0.f, a);
                    x[i] = a;
                }
                tot[q4] = a;
            }
            float off = 0.f;
#pragma unroll
            for (int q4 = 1; q4 < 4; ++q4) {
                off += tot[q4 - 1];
#pragma unroll
                for (int j = 0; j < 16; ++j) x[16 * q4 + j] += off;
            }
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                rng = fmaxf(rng, fabsf(x[i]));
                sG2[gsw(i, tid)] = x[i];
            }
            acc = x[63];
        } else {
            float x[16], y[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = sG2[gsw(j, tid)];
#pragma unroll 1
            for (int i0 = 0; i0 < 64; i0 += 16) {
                if (i0 + 16 < 64) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) y[j] = sG2[gsw(i0 + 16 + j, tid)];
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (i0 + j < nr && live) {
                        float gj = x[j];
                        if (gate_act) gj = neg_a * softplus_f(gj + gbias);
                        acc = p.g_is_cumsum ? gj : fmaf(p.g_scale, gj, acc);
                    }
                    x[j] = acc;
                    rng = fmaxf(rng, fabsf(acc));
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) sG2[gsw(i0 + j, tid)] = x[j];
#pragma unroll
                for (int j = 0; j < 16; ++j) x[j] = y[j];
            }
        }
        const float eG = ex2_ftz(acc);
        sEG[tid] = eG;
        sGv[tid] = acc;
        reinterpret_cast<float *>(U + Lo.dec)[tid] = eG;
        atomicMax(&sRangeBits, __float_as_int(rng));
    } else if (tid < 128) {
        reinterpret_cast<float *>(U + Lo.dec)[tid] = 0.f;
    }
    if (tid == 0 && !mbar_wait(&bar_qk, ph_in & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
    ++ph_in;
    __syncthreads();
    // rows past the chunk's end hold another sequence's rows (or NaN): zero them
    // before anything reads them
    if (__builtin_expect(nr < 64, 0)) {
        for (int idx = tid; idx < (64 - nr) * (KK / 8); idx += 256) {
            const int i = nr + idx / (KK / 8), c = (idx % (KK / 8)) * 8;
            *reinterpret_cast<uint4 *>(sAG + qk_off(i, c)) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(sAG + qk_off(64 + i, c)) = make_uint4(0, 0, 0, 0);
        }
        __syncthreads();
    }

    // ---- optional L2 normalisation of the q and k rows (thread t: row t)
    if (__builtin_expect(p.l2norm != 0, 0)) {
        if (tid < 128) {
            float ss = 0.f;
#pragma unroll 1
            for (int c = 0; c < KK; c += 8) {
                float f[8];
                unpack8(*reinterpret_cast<const uint4 *>(sAG + qk_off(tid, c)), f);
#pragma unroll
                for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
            }
            const float rsn = 1.f / sqrtf(ss + 1e-6f);
#pragma unroll 1
            for (int c = 0; c < KK; c += 8) {
                uint4 *at = reinterpret_cast<uint4 *>(sAG + qk_off(tid, c));
                float f[8];
                unpack8(*at, f);
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] *= rsn;
                *at = pack8(f);
            }
        }
        __syncthreads();
    }
    const bool fast = __int_as_float(sRangeBits) <= kSafeRange;

    // ---- exact grams for chunks whose gate range is too wide to split.  A pair j < i
    // in different 16-row blocks takes the gate through a block boundary e between
    // them, 2^(g2_i - g2_e) 2^(g2_e - g2_j), both exponents <= 0 (ALGORITHM.md, "The
    // numerics law": a boundary between the blocks separates the pair): four small
    // tensor-core products of operands scaled to the boundaries.  The 4 x 4 diagonal
    // blocks take 2^(g2_i - g2_j) itself on the CUDA cores.
    if (__builtin_expect(!fast, 0)) {
        exact_grams<KK, kSplitA>(sAG, sG2, sBeta, sL, sKB, sm + S::khat, U + Lo.aqk, tmem, &bar,
                                 phase, p.status, tid);
        phase += 4;
        __syncthreads();
    }

    // ---- 3. elementwise, in place: 8 channels of one row per thread; lanes 0..7
    // take 8 consecutive rows of one column chunk, which the swizzle spreads over
    // all banks.  qg, kg, kb in place; qg and kg to the workspace.
#pragma unroll 1
    for (int it = 0; it < KK / 32; ++it) {
        const int idx = tid + it * 256, l = idx & 31, w = idx >> 5;
        const int i = (w & 7) * 8 + (l & 7);
        const int c = ((w >> 3) * 4 + (l >> 3)) * 8;
        uint4 *pq = reinterpret_cast<uint4 *>(sAG + qk_off(i, c));
        uint4 *pk = reinterpret_cast<uint4 *>(sAG + qk_off(64 + i, c));
        float fq[8], fk[8], gam[8];
        unpack8(*pq, fq);
        unpack8(*pk, fk);
        *reinterpret_cast<float4 *>(gam) = *reinterpret_cast<const float4 *>(sG2 + gsw(i, c));
        *reinterpret_cast<float4 *>(gam + 4) = *reinterpret_cast<const float4 *>(sG2 + gsw(i, c + 4));
        float qg[8], kgm[8], kb[8], kgv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float e = ex2_ftz(gam[j]);
            qg[j] = fq[j] * e;
            kgm[j] = fk[j] * e;
            if (fast) {
                kb[j] = fk[j] * ex2_ftz(-gam[j]);
                kgv[j] = kb[j] * sEG[c + j];
            } else {
                kgv[j] = fk[j] * ex2_ftz(sGv[c + j] - gam[j]);
            }
        }
        const uint4 qpk = pack8(qg);
        *pq = qpk;
        *pk = pack8(kgm);
        if (fast) *reinterpret_cast<uint4 *>(sKB + qk_off(i, c)) = pack8(kb);
        *reinterpret_cast<uint4 *>(U + Lo.aw + tile_off(64 + i, c, KK)) = qpk;
        *reinterpret_cast<uint4 *>(U + Lo.kgt + tile_off(i, c, KK)) = pack8(kgv);
    }
    if (vtma) {
        // One barrier: the elementwise pass has read g2 and written the gram
        // operands before thread 0 issues v into g2's second half, the next unit's
        // g channels 0..63 into its first half, and the gram MMA.  v is waited for
        // just before the u MMA.
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            fence_async_smem();
            mbar_arrive_expect_tx(&bar_v, 64 * VV * 2);
            for (int x = 0; x < VV / 64; ++x)
                tma_load3(sV + x * 8192, &maps.v, x * 64, hv, b * p.T + r0, &bar_v);
            if (nxt->unit < uend) issue(nxt, true, false, false, false);
        }
    } else {
        __syncthreads();
        // v into the freed g2 buffer (its second half with the pref plan); waited
        // for just before the u MMA
        for (int idx = tid; idx < 64 * VG8; idx += 256) {
            const int l = idx & 31, w = idx >> 5;
            const int i = (w & 7) * 8 + (l & 7);
            const int c = ((w >> 3) * 4 + (l >> 3)) * 8;
            void *dv = sV + tile_off(i, c, VV) + (i >= 32 ? v_half : 0);
            if (i < nr)
                cp_async16(dv, v + ((row0 + i) * p.HV + hv) * VV + c);
            else
                *reinterpret_cast<uint4 *>(dv) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        // with the pref plan the first half of g2 is free for good: the next
        // unit's g channels 0..63
        if (pref && tid == 0 && nxt->unit < uend) issue(nxt, true, false, false, false);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    // ---- 4. grams on the tensor cores.  D[:, 0:64] = [Qg; Kg] Kb^T (split grams),
    // D[:, 64:128] = [Qg; Kg] kgp^T (cross-chunk gram with the previous chunk);
    // Kb and kgp are rows 0..63 and 64..127 of kbx, so both take one MMA series
    // of N = 128.  Both operands K-major, 128-byte swizzled: a K step of 16
    // channels moves 32 bytes inside a column block, every fourth step a block.
    if (tid == 0) {
        const uint32_t a0 = smem_addr(sAG), b0 = smem_addr(sKB) + ((fast || !halo) ? 0 : 8192);
        const uint32_t idn = idesc_bf16(128, (fast && halo) ? 128 : 64, false, false);
        if (fast || halo) {
#pragma unroll 1
            for (int kk = 0; kk < KK / 16; ++kk) {
                const uint32_t ko = (kk >> 2) * S::kBlk + (kk & 3) * 32;
                mma_bf16(tmem + (fast ? 0 : 64), sdesc_sw128(a0 + ko, 16, 1024),
                         sdesc_sw128(b0 + ko, 16, 1024), idn, kk > 0);
            }
        }
        mma_commit(&bar);
    }
    if (tid == 0 && !mbar_wait(&bar, phase & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
    __syncthreads();
    ++phase;
    tc_fence_after();
    {
        const int quad = warp & 3, i = (tid & 127) & 63;
        // 16 columns at a time, the loops kept rolled: code size, not issue slots, is
        // what this kernel runs short of (its 2 x 256 threads wait on instruction fetch)
        if (warp < 4 && fast) {  // Aqk (rows 0..63) and L (rows 64..127) from columns 0..63
            const float bi = sBeta[i];
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 16) {
                float dd[16];
                tmem_ld16(tmem_at(tmem, quad * 32, c0), dd);
                if (tid < 64) {
#pragma unroll
                    for (int h = 0; h < 16; h += 8) {
                        float a8[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) a8[j] = (c0 + h + j <= i) ? dd[h + j] : 0.f;
                        *reinterpret_cast<uint4 *>(U + Lo.aqk + tile_off(i, c0 + h, 64)) = pack8(a8);
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 16; h += 4)
                        sta4<kSplitA>(sL, i, c0 + h,
                                make_float4(c0 + h < i ? bi * dd[h] : 0.f,
                                            c0 + h + 1 < i ? bi * dd[h + 1] : 0.f,
                                            c0 + h + 2 < i ? bi * dd[h + 2] : 0.f,
                                            c0 + h + 3 < i ? bi * dd[h + 3] : 0.f));
                }
            }
        }
        if (warp >= 6 && halo) {  // P = kg_c kgp^T from rows 64..127, columns 64..127
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 16) {
                float dd[16];
                tmem_ld16(tmem_at(tmem, quad * 32, 64 + c0), dd);
                *reinterpret_cast<uint4 *>(sPB + tile_off(i, c0, 64)) = pack8_at(dd);
                *reinterpret_cast<uint4 *>(sPB + tile_off(i, c0 + 8, 64)) = pack8_at(dd + 8);
            }
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---- 5. Akk = (I + L)^-1 in fp32.  The 16 x 16 diagonal blocks X_I by
    // substitution, then two doubling steps: the 32 x 32 diagonal blocks
    // (A_10 = -X_1 L_10 X_0, A_32 = -X_3 L_32 X_2), then the lower-left 32 x 32
    // block -Y_1 L_[23][01] Y_0.  The products run as 1 x 4 strips per thread
    // (row r = lane % 8 + 8 (t / 32), columns 4 (lane / 8) of a 16 x 16 block).
    // Only blocks on or below the diagonal are written; the rest is masked later.
    if (tid < 64) {
        const int I = tid >> 4, c = tid & 15, o = 16 * I;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int m4 = 0; m4 < r; m4 += 4) {
                const float4 l4 = lda4<kSplitA>(sL, o + r, o + m4);
                s0 = fmaf(l4.x, x[m4], s0);
                if (m4 + 1 < r) s1 = fmaf(l4.y, x[m4 + 1], s1);
                if (m4 + 2 < r) s0 = fmaf(l4.z, x[m4 + 2], s0);
                if (m4 + 3 < r) s1 = fmaf(l4.w, x[m4 + 3], s1);
            }
            if (r > c) x[r] = -(s0 + s1);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sA[akk_idx<kSplitA>(o + r, o + c)] = x[r];
    }
    __syncthreads();
    const int sr = (lane & 7) + 8 * ((tid >> 5) & 1), sc = 4 * (lane >> 3), blk = tid >> 6;
    if (tid < 128) {  // T = L_{I,I-1} X_{I-1} for I = 1, 3  -> sT block (blk, blk)
        const int I = 2 * blk + 1;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        strip_la<kSplitA>(s, sL, 16 * I + sr, 16 * (I - 1), sA, 16 * (I - 1), 16 * (I - 1) + sc);
        st4<32>(sT, 16 * blk + sr, 16 * blk + sc, s);
    }
    __syncthreads();
    if (tid < 128) {  // A_{I,I-1} = -X_I T
        const int I = 2 * blk + 1;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        strip_at<kSplitA>(s, sA, 16 * I + sr, 16 * I, sT, 16 * blk, 16 * blk + sc);
        sta4<kSplitA>(sA, 16 * I + sr, 16 * (I - 1) + sc, neg4(s));
    }
    __syncthreads();
    {  // T_IJ = sum_M L_IM Y0_MJ for I = 2, 3 and J = 0, 1  -> sT (I - 2, J)
        const int I = 2 + (blk >> 1), J = blk & 1;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int M = J; M < 2; ++M)
            strip_la<kSplitA>(s, sL, 16 * I + sr, 16 * M, sA, 16 * M, 16 * J + sc);
        st4<32>(sT, 16 * (I - 2) + sr, 16 * J + sc, s);
    }
    __syncthreads();
    {  // A_IJ = -sum_M Y1_IM T_MJ
        const int I = 2 + (blk >> 1), J = blk & 1;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int M = 2; M <= I; ++M)
            strip_at<kSplitA>(s, sA, 16 * I + sr, 16 * M, sT, 16 * (M - 2), 16 * J + sc);
        sta4<kSplitA>(sA, 16 * I + sr, 16 * J + sc, neg4(s));
    }
    __syncthreads();
    // Akk diag(beta) as a bf16 operand tile (Akk is lower triangular), stored twice so
    // that the MMAs below give every result row in both TMEM lane halves.
#pragma unroll 1
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + it * 256, l = idx & 31, w = idx >> 5;
        const int i = (w & 7) * 8 + (l & 7);
        const int c = ((w >> 3) * 4 + (l >> 3)) * 8;
        const float4 a0 = lda4<kSplitA>(sA, i, c), a1 = lda4<kSplitA>(sA, i, c + 4);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = (c + j <= i) ? av[j] * sBeta[c + j] : 0.f;
        const uint4 ab = pack8(f);
        *reinterpret_cast<uint4 *>(sAB + tile_off(i, c, 64)) = ab;
        *reinterpret_cast<uint4 *>(sAB + tile_off(64 + i, c, 64)) = ab;
        if (__builtin_expect(p.bwd, 0)) {  // Akk itself for the backward
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = (c + j <= i) ? av[j] : 0.f;
            *reinterpret_cast<uint4 *>(U + Lo.akk + tile_off(i, c, 64)) = pack8(f);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 6. W = Akk diag(beta) Kg and M = Akk diag(beta) P (TMEM lanes 64..127 repeat
    // lanes 0..63).
    // Kg is an MN-major 128-byte swizzled operand here: a K step (16 rows) moves
    // two 8-row groups (2 KB); its 64-column blocks lie 16 KB apart.
    const uint64_t adesc = sdesc(smem_addr(sAB), 128, 1024);  // [Akk diag(beta); the same]
    if (tid == 0) {
        const uint32_t kg0 = smem_addr(sAG) + 8192;
#pragma unroll 1
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, adesc + (uint64_t)(kk * 16), sdesc_sw128(kg0 + kk * 2048, S::kBlk, 1024),
                     idesc_bf16(128, KK, false, true), kk > 0);
        if (halo)
            mma_bf16_seq<4, false>(tmem + KK, adesc, 16, sdesc(smem_addr(sPB), 64 * 16, 128),
                                   2 * 64 * 16 / 16, idesc_bf16(128, 64, false, true));
        mma_commit(&bar);
    }
    if (tid == 0 && !mbar_wait(&bar, phase & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
    __syncthreads();
    ++phase;
    tc_fence_after();
    // The k rows of ag were the W MMA's last use of them: with the pref plan, the
    // next unit's k rows go there now.
    if (pref && tid == 0 && nxt->unit < uend) issue(nxt, false, false, false, true);
    {
        // W~ = W Diag(2^G_prev) -> rows 0..63 of the [W; qg] tile, and M.  Row i sits in
        // TMEM lanes i and 64 + i; the four warps that reach those lanes (w % 4 = i / 32
        // or 2 + i / 32) take a quarter of its columns each.
        const int quad = warp & 3, i = (tid & 127) & 63, part = (warp >> 2) + 2 * (quad >> 1);
        constexpr int kQ = KK / 4;
        float dd[kQ];
        if constexpr (kQ == 32)
            tmem_ld32(tmem_at(tmem, quad * 32, part * kQ), dd);
        else
            tmem_ld16(tmem_at(tmem, quad * 32, part * kQ), dd);
        if (__builtin_expect(p.bwd, 0)) {  // W itself for the backward
#pragma unroll
            for (int c8 = 0; c8 < kQ; c8 += 8)
                *reinterpret_cast<uint4 *>(U + Lo.wb + tile_off(i, part * kQ + c8, KK)) = pack8_at(dd + c8);
        }
        if (halo) {
#pragma unroll
            for (int j = 0; j < kQ; ++j) dd[j] *= sDprev[part * kQ + j];
        }
#pragma unroll
        for (int c8 = 0; c8 < kQ; c8 += 8)
            *reinterpret_cast<uint4 *>(U + Lo.aw + tile_off(i, part * kQ + c8, KK)) = pack8_at(dd + c8);
        if (halo) {
            float dm[16];
            tmem_ld16(tmem_at(tmem, quad * 32, KK + part * 16), dm);
#pragma unroll
            for (int c8 = 0; c8 < 16; c8 += 8)
                *reinterpret_cast<uint4 *>(U + Lo.mt + tile_off(i, part * 16 + c8, 64)) = pack8_at(dm + c8);
        }
    }
    // v has landed before anyone passes this barrier.  With v by TMA, rows past
    // the chunk's end (another sequence's rows, or NaN) are zeroed once it has.
    if (vtma && __builtin_expect(nr < 64, 0)) {
        if (!mbar_wait(&bar_v, ph_v & 1, kWaitNs) && tid == 0) report(p.status, KDA_DEVICE_TIMEOUT);
        for (int idx = tid; idx < (64 - nr) * (VV / 8); idx += 256) {
            const int i = nr + idx / (VV / 8), c = (idx % (VV / 8)) * 8;
            *reinterpret_cast<uint4 *>(sV + sw128_off(i, c, 8192)) = make_uint4(0, 0, 0, 0);
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid < KK) sDprev[tid] = sEG[tid];  // the next chunk's 2^G_prev (read after this unit)

    // ---- 7. u = Akk diag(beta) v
    if (tid == 0) {
        if (vtma) {
            // v MN-major, 128-byte swizzled: a K step (16 rows) moves 2 KB, its
            // 64-column boxes lie 8 KB apart
            if (!mbar_wait(&bar_v, ph_v & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem, adesc + (uint64_t)(kk * 16),
                         sdesc_sw128(smem_addr(sV) + kk * 2048, 8192, 1024),
                         idesc_bf16(128, VV, false, true), kk > 0);
        } else {
            // K step kk: v rows 16 kk .. 16 kk + 15 (the second half v_half further on)
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem, adesc + (uint64_t)(kk * 16),
                         sdesc(smem_addr(sV) + kk * 2 * VV * 16 + (kk >= 2 ? v_half : 0), VV * 16, 128),
                         idesc_bf16(128, VV, false, true), kk > 0);
        }
        mma_commit(&bar);
    }
    if (vtma) ++ph_v;
    if (tid == 0 && !mbar_wait(&bar, phase & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
    __syncthreads();
    ++phase;
    tc_fence_after();
    // Every operand of this unit has been read: the next unit's remaining copies,
    // and, if it is the next chunk of this sequence, this chunk's kg as its
    // previous-kg rows (waited for at the start of that unit).
    if (nxt->unit < uend) {
        if (tid == 0) issue(nxt, !pref, true, true, !pref);
        if (nxt->hv == hv && nxt->gc == gc + 1 && continues(p, nxt->cl, nxt->ncs)) {
#pragma unroll 1
            for (int it = 0; it < KK / 32; ++it) {
                const int idx = tid + it * 256, i = idx & 63, c = (idx >> 6) * 8;
                cp_async16(sKB + qk_off(64 + i, c), U + Lo.kgt + tile_off(i, c, KK));
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
    }
    {
        // u: the same row split as W, a quarter of the dv columns per warp
        const int quad = warp & 3, i = (tid & 127) & 63, part = (warp >> 2) + 2 * (quad >> 1);
        const int per = VV / 4, cbeg = part * per;  // per: a multiple of 8
        if (per % 16 == 0) {
#pragma unroll 1
            for (int c0 = cbeg; c0 < cbeg + per; c0 += 16) {
                float dd[16];
                tmem_ld16(tmem_at(tmem, quad * 32, c0), dd);
                unsigned char *ub = U + Lo.u + ((size_t)(c0 / kUB) * 64 + i) * kUB * 2;
                *reinterpret_cast<uint4 *>(ub) = pack8_at(dd);
                *reinterpret_cast<uint4 *>(ub + 16) = pack8_at(dd + 8);
            }
        } else {
            for (int c0 = cbeg; c0 < cbeg + per; c0 += 8) {
                float dd[8];
                tmem_ld8(tmem_at(tmem, quad * 32, c0), dd);
                unsigned char *ub =
                    U + Lo.u + ((size_t)(c0 / kUB) * 64 + i) * kUB * 2 + (c0 % kUB) * 2;
                *reinterpret_cast<uint4 *>(ub) = pack8_at(dd);
            }
        }
    }
    tc_fence_before();
    if (tid == 0) sRangeBits = 0;
    __syncthreads();
    tc_fence_after();
    prev_hv = hv;
    prev_gc = gc;
    slot ^= 1;
    }  // unit loop
    // Every copy was waited for, but a wait that gave up may have left its copy
    // in flight: wait for the last ones once more (bounded; immediate when they
    // landed) before the shared memory they write is released.
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (tid == 0 && ph_in > 0) {
        mbar_wait(&bar_g, (ph_in - 1) & 1, kWaitNs);
        mbar_wait(&bar_qk, (ph_in - 1) & 1, kWaitNs);
        if (ph_v > 0) mbar_wait(&bar_v, (ph_v - 1) & 1, kWaitNs);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kCols);
}

// ============================================================== scan kernel
// Rounds r = 0 .. nc of one (sequence, value head, SBV value columns); round r
// finishes chunk c = r - 1 and starts chunk c + 1:
//   A: D1  = [W~_{c+1}; qg_c] h_c        (needs h_c)
//   C: D2  = kg_c^T v'_c                 (needs v'_c)   ->  h_{c+1} = Diag(2^G_c) h_c + D2
//   B: D1 += [M_{c+1}; Aqk_c] v'_c       (needs v'_c)   ->  v'_{c+1} = u_{c+1} - D1[0:64]
//                                                          o_c      = scale D1[64:128]
// where W~_{c+1} = W_{c+1} Diag(2^G_c) and M_{c+1} = W_{c+1} kg_c^T come from the
// prep kernel: v'_{c+1} = u_{c+1} - W_{c+1} h_{c+1} expands into the A and B
// terms.  Issue order A, C, B: the state update (after C) overlaps B, and the
// next round's A can start as soon as h_{c+1} is written.  Round 0 only forms
// v'_0 = u_0 - W_0 h_0.  A tcgen05.mma of these shapes occupies the tensor
// unit for a fixed ~50 cycles whatever N <= 64 is, so 32 columns per CTA cost
// no more MMA time than 16.
//
// Split sequences (context parallel within the GPU).  The state after a segment
// of chunks is an affine function of the state before it: h_end = P h_start + E.
// A split launch runs a sequence's two halves at once: segment 0 from h0 as
// above (its final state E0), segment 1 from a zero state (o partial, final state
// E1) and, in K extra "identity" columns, from the identity matrix with u = 0:
// their readout is Q_c, the response of o_c to the segment's initial state, and
// their final state is P.  The fix kernel then adds Q_c E0 to segment 1's rows
// and forms ht = P E0 + E1.  The prep treats segment 1's first chunk as a
// sequence start (untilded W, no M), which is exactly a scan from a given state.
template <int KK, int SBV>
struct ScanSmem {
    static constexpr int kStages = SBV == 32 ? 3 : 2;
    static constexpr uint32_t top = 0;                         // [128][KK]: W~_{c+1}; qg_c
    static constexpr uint32_t kgt = top + 128 * KK * 2;        // [64][KK]: kg_c
    static constexpr uint32_t bot = kgt + 64 * KK * 2;         // [128][64]: M_{c+1}; Aqk_c
    static constexpr uint32_t u = bot + 128 * 64 * 2;          // [SBV/kUB][64][kUB] bf16: u_{c+1}
    static constexpr uint32_t dec = u + 64 * SBV * 2;          // [128] fp32: 2^G_c
    static constexpr uint32_t stage = dec + 512;
    static constexpr uint32_t stage_stride = (stage + 1023) / 1024 * 1024;
    static constexpr uint32_t hs = kStages * stage_stride;     // [KK][SBV] tile
    static constexpr uint32_t vp = hs + KK * SBV * 2;          // [64][SBV] tile
    static constexpr uint32_t total = vp + 64 * SBV * 2;
    // D1[0], D1[1], D2 at 0, SBV, 2 SBV
    static constexpr uint32_t tmem_cols = SBV == 32 ? 128 : (SBV == 64 ? 256 : 512);
};

__device__ __forceinline__ int read_flag(const int *f) {
    return *reinterpret_cast<const volatile int *>(f);
}

// Hardware named barriers (ids 1 and 2; 0 is __syncthreads).  bar.arrive does
// not block; bar.sync waits for the barrier's full thread count.  Whole warps
// execute both (the instructions are warp-aligned).  A named barrier hands over
// in a few tens of cycles, an mbarrier arrive -> wait in a few hundred.
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// One lane of a converged warp (the same lane every time the warp is converged).
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}
constexpr int kBarH = 1;   // h_c written: the 4 h warps arrive, the MMA warp syncs
constexpr int kBarV = 2;   // v'_c written and D1 read: v' and o warps arrive, the MMA warp syncs
constexpr int kThrH = 128 + 32;
constexpr int kThrV = 128 + 32;


// Work item of a scan CTA.  Without a split: (n, hv, vb) over the V columns.
// With a split, per (n, hv): V/SBV segment-0 blocks, V/SBV segment-1 blocks,
// then KK/SBV segment-1 identity blocks.
struct ScanItem {
    int n, hv, vb, seg;
    bool ident;
};
template <int KK, int SBV>
__device__ __forceinline__ ScanItem scan_item(const ChunkArgs &p, int64_t bid) {
    ScanItem it;
    const int nreal = p.V / SBV;
    const int bpp = p.split ? 2 * nreal + KK / SBV : nreal;
    const int j = (int)(bid % bpp);
    it.hv = (int)((bid / bpp) % p.HV);
    it.n = (int)(bid / ((int64_t)bpp * p.HV));
    it.seg = p.pipe.parts > 0 ? (p.scan_c0 > 0 ? 1 : 0) : (j < nreal ? 0 : 1);
    it.ident = j >= 2 * nreal;
    it.vb = j < nreal ? j : (j < 2 * nreal ? j - nreal : j - 2 * nreal);
    return it;
}

// Warp roles: 0..3 h (state rows 32 w .. 32 w + 31, all SBV columns, in fp32
// registers), 4..5 v' (rows 0..63 of D1), 6..7 o (rows 64..127 of D1), 8 bulk
// copies, 9 MMA issue.  A warp reaches TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31.
template <int KK, int SBV>
__global__ void __launch_bounds__(320, 1) chunk_scan_tc_kernel(ChunkArgs p) {
    using S = ScanSmem<KK, SBV>;
    constexpr int kStages = S::kStages;
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint64_t full[kStages], empty[kStages];
    // bar_v[x]: MMAs writing D1[x] done, one per buffer.
    __shared__ uint64_t bar_v[2], bar_h, bar_fin, bar_never;
    __shared__ uint32_t tslot;
    __shared__ int abort_flag;

    const ScanItem item = scan_item<KK, SBV>(p, blockIdx.x);
    const int n = item.n, hv = item.hv, vb = item.vb;
    const bool ident = item.ident;
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
    // this CTA's chunks [c0, c1) of the sequence
    int c0 = 0, c1 = nc;
    if (p.split) {
        const int m = (nc + 1) / 2;
        if (item.seg == 0) c1 = m; else c0 = m;
    } else if (p.pipe.parts > 0) {
        c0 = min(p.scan_c0, nc);
        c1 = min(p.scan_c1, nc);
    }
    const int ncs = c1 - c0;
    const int R = ncs > 0 ? ncs + 1 : 0;  // rounds
    const TcLayout Lo = tc_layout(KK, p.V, p.bwd);
    const unsigned char *units = static_cast<const unsigned char *>(p.units);

    if (warp == 0) {
        tmem_alloc(&tslot, S::tmem_cols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 6);  // MMA commit + the h and v' warps
        }
        mbar_init(&bar_v[0], 1);
        mbar_init(&bar_v[1], 1);
        mbar_init(&bar_h, 1);
        mbar_init(&bar_fin, 1);
        mbar_init(&bar_never, 1);  // the test hook's barrier: nothing ever arrives on it
        mbar_fence_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;  // D1[0] at +0, D1[1] at +SBV, D2 at +2 SBV
    unsigned char *sH = sm + S::hs;
    unsigned char *sVp = sm + S::vp;
    // A wait that runs out sets the abort flag.  From then on nobody waits for
    // copies (full / empty) and the MMA warp issues no MMAs, but it still commits
    // every round, and every role still takes part in every named barrier: the
    // commits keep the epilogue in step with the MMA warp, so each named-barrier
    // instance gathers exactly one arrival per warp, and the CTA runs through its
    // rounds and exits.
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
    auto stage = [&](int r) { return sm + (r % kStages) * S::stage_stride; };

    if (warp == 8) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int r = 0; r < R; ++r) {
                const int s = r % kStages;
                if (r >= kStages) wait_copy(&empty[s], ((r / kStages) - 1) & 1);
                if (read_flag(&abort_flag)) break;
                unsigned char *st = stage(r);
                const int c = c0 + r - 1;
                const bool nxt = r < ncs, cur = r >= 1;
                uint32_t bytes = 0;
                if (nxt) bytes += 64 * KK * 2 + (ident ? 0 : 64 * SBV * 2) + (cur ? 64 * 64 * 2 : 0);
                if (cur) bytes += 64 * KK * 2 + 64 * KK * 2 + 64 * 64 * 2 + 512;
                mbar_arrive_expect_tx(&full[s], bytes);
                if (nxt) {
                    const unsigned char *U1 = units + unit_index(p, gc0 + c + 1, hv) * (int64_t)Lo.stride;
                    bulk_g2s(st + S::top, U1 + Lo.aw, 64 * KK * 2, &full[s]);
                    if (!ident)
                        bulk_g2s(st + S::u, U1 + Lo.u + (size_t)vb * 64 * SBV * 2, 64 * SBV * 2,
                                 &full[s]);
                    if (cur) bulk_g2s(st + S::bot, U1 + Lo.mt, 64 * 64 * 2, &full[s]);
                }
                if (cur) {
                    const unsigned char *U0 = units + unit_index(p, gc0 + c, hv) * (int64_t)Lo.stride;
                    bulk_g2s(st + S::top + 64 * KK * 2, U0 + Lo.aw + 64 * KK * 2, 64 * KK * 2,
                             &full[s]);
                    bulk_g2s(st + S::kgt, U0 + Lo.kgt, 64 * KK * 2, &full[s]);
                    bulk_g2s(st + S::bot + 64 * 64 * 2, U0 + Lo.aqk, 64 * 64 * 2, &full[s]);
                    bulk_g2s(st + S::dec, U0 + Lo.dec, 512, &full[s]);
                }
                issued = r + 1;
            }
            // Copies in flight must land before the CTA exits (bounded).
            for (int r = issued - kStages > 0 ? issued - kStages : 0; r < issued; ++r)
                mbar_wait(&full[r % kStages], (r / kStages) & 1, kWaitNs);
        }
    } else if (warp == 9) {
        // ----------------------------------------------------- MMA issuer
        const uint32_t idn = idesc_bf16(128, SBV, false, true);
        const uint32_t idc = idesc_bf16(128, SBV, true, true);  // A = kg tile read MN-major
        const uint64_t dh = sdesc(smem_addr(sH), SBV * 16, 128);
        const uint64_t dv = sdesc(smem_addr(sVp), SBV * 16, 128);
        constexpr uint32_t binc = 2 * SBV * 16 / 16;
        if (p.test_timeout) {
            // KDA_FLAG_TEST_WAIT_TIMEOUT: a consumer wait that runs out, on purpose
            if (elect_one() && !mbar_wait(&bar_never, 0, 2000)) fail();
            __syncwarp();
        }
        for (int r = 0; r < R; ++r) {
            const int s = r % kStages;
            const uint32_t st = smem_addr(stage(r));
            const uint32_t d1 = tmem + (r & 1) * SBV;
            wait_copy(&full[s], (r / kStages) & 1);
            __syncwarp();
            named_sync(kBarH, kThrH);
            const bool go = !read_flag(&abort_flag);
            if (elect_one()) {
                tc_fence_after();
                if (go)
                    mma_bf16_seq<KK / 16, false>(d1, sdesc(st + S::top, 128, KK * 16), 16, dh, binc, idn);
            }
            __syncwarp();
            if (r >= 1) {
                named_sync(kBarV, kThrV);
                if (elect_one()) {
                    tc_fence_after();
                    if (go)
                        mma_bf16_seq<4, false>(tmem + 2 * SBV, sdesc(st + S::kgt, KK * 16, 128),
                                               2 * KK * 16 / 16, dv, binc, idc);
                    mma_commit(&bar_h);
                    if (go) mma_bf16_seq<4, true>(d1, sdesc(st + S::bot, 128, 1024), 16, dv, binc, idn);
                }
                __syncwarp();
            }
            if (elect_one()) {
                mma_commit(&bar_v[r & 1]);
                mma_commit(&empty[s]);
            }
            __syncwarp();
        }
        // Every MMA issued has completed before the CTA frees its tensor memory.
        if (elect_one()) {
            mma_commit(&bar_fin);
            mbar_wait(&bar_fin, 0, kWaitNs);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------ h warps: the state
        const int row = warp * 32 + lane;
        const bool has_row = row < KK;
        const bool glob_row = row < p.K;  // rows past K stay zero and are neither read nor stored
        const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + 2 * SBV;
        float h[SBV];
#pragma unroll
        for (int j = 0; j < SBV; ++j) h[j] = 0.f;
        if (ident) {
#pragma unroll
            for (int j = 0; j < SBV; ++j) h[j] = (row == vb * SBV + j) ? 1.f : 0.f;
        } else if (glob_row && (item.seg == 0 ? p.h0 : (p.pipe.parts > 0 ? p.e0 : nullptr))) {
            // a pipelined launch's later parts start from the previous part's final state
            const float *h_init = item.seg == 0 ? p.h0 : p.e0;
            const float4 *src = reinterpret_cast<const float4 *>(
                h_init + (((size_t)n * p.HV + hv) * p.K + row) * (size_t)p.V + (size_t)vb * SBV);
#pragma unroll
            for (int j = 0; j < SBV / 4; ++j) {
                const float4 x = src[j];
                h[4 * j] = x.x; h[4 * j + 1] = x.y; h[4 * j + 2] = x.z; h[4 * j + 3] = x.w;
            }
        }
        // h at the start of chunk cc: the next MMA's operand (and, for the backward,
        // the chunk's checkpoint tile)
        auto write_h = [&](int cc) {
            if (has_row) {
                unsigned char *t = p.ck_h ? static_cast<unsigned char *>(p.ck_h) +
                                                unit_index(p, gc0 + cc, hv) * (int64_t)(KK * p.V * 2) +
                                                tile_off(row, vb * SBV, p.V)
                                          : nullptr;
#pragma unroll
                for (int c = 0; c < SBV; c += 8) {
                    const uint4 v8 = pack8_at(h + c);
                    *reinterpret_cast<uint4 *>(sH + tile_off(row, c, SBV)) = v8;
                    if (t) *reinterpret_cast<uint4 *>(t + c * 16) = v8;  // next 8 columns: +128 B
                }
            }
            fence_async_smem();
            __syncwarp();
            named_arrive(kBarH, kThrH);
        };
        // 2^G of round r's finishing chunk, read one round ahead
        auto fetch = [&](int r) {
            float d = 1.f;
            wait_copy(&full[r % kStages], (r / kStages) & 1);
            if (r >= 1 && has_row) d = reinterpret_cast<const float *>(stage(r) + S::dec)[row];
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[r % kStages]);
            return d;
        };
        if (R > 0) write_h(c0);
        float dec = R > 0 ? fetch(0) : 1.f;
        for (int r = 0; r < R; ++r) {
            const bool nxt = r < ncs;
            if (r >= 1) {
                // h_{c+1} = Diag(2^G_c) h_c + D2  (bar_h also covers A_r's reads of h_c)
                wait_mma(&bar_h, (r - 1) & 1);
                tc_fence_after();
                // D2 a slice at a time (128-column CTAs cannot hold all of D2 beside h)
                constexpr int kSl = SBV == 128 ? 16 : 32;
#pragma unroll
                for (int cb = 0; cb < SBV; cb += kSl) {
                    float d[kSl];
                    if constexpr (kSl == 16)
                        tmem_ld16(taddr + cb, d);
                    else
                        tmem_ld32(taddr + cb, d);
#pragma unroll
                    for (int t = 0; t < kSl; ++t) h[cb + t] = fmaf(dec, h[cb + t], d[t]);
                }
                tc_fence_before();
                if (nxt) write_h(c0 + r);
            } else if (nxt) {
                // Round 0 leaves h_0 in place.  Arrive for round 1 only once round 0's
                // MMA has completed, i.e. after the MMA warp left this barrier's
                // round-0 instance.
                wait_mma(&bar_v[0], 0);
                __syncwarp();
                named_arrive(kBarH, kThrH);
            }
            if (r + 1 < R) dec = fetch(r + 1);
        }
        // final state: ht, or for a split sequence E0 / E1 / P
        float *dst_base = nullptr;
        int width = p.V;
        if (p.pipe.parts > 0) {
            dst_base = c1 >= nc ? p.ht : p.e0;
        } else if (!p.split) {
            dst_base = p.ht;
        } else if (ident) {
            dst_base = p.pm;
            width = KK;
        } else {
            dst_base = item.seg == 0 ? p.e0 : p.e1;
        }
        if (dst_base && glob_row && !read_flag(&abort_flag)) {
            float4 *dst = reinterpret_cast<float4 *>(
                dst_base + (((size_t)n * p.HV + hv) * p.K + row) * (size_t)width + (size_t)vb * SBV);
#pragma unroll
            for (int j = 0; j < SBV / 4; ++j)
                dst[j] = make_float4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
            if (p.split && !ident && item.seg == 0) {
                // E0 again as the fix kernel's bf16 MMA operand ([KK][V] MN-major tile)
                unsigned char *t = static_cast<unsigned char *>(p.e0b) +
                                   ((size_t)n * p.HV + hv) * (size_t)KK * p.V * 2;
#pragma unroll
                for (int c = 0; c < SBV; c += 8)
                    *reinterpret_cast<uint4 *>(t + tile_off(row, vb * SBV + c, p.V)) = pack8_at(h + c);
            }
        }
    } else if (warp < 6) {
        // ------------------------------------- v' warps: v'_{c+1} = u_{c+1} - D1[0:64]
        const int row = (warp - 4) * 32 + lane;
        const uint32_t lanebase = (uint32_t)((warp - 4) * 32) << 16;
        // u_{c+1} of this row, kept as packed bf16 pairs (the registers of 128-column
        // CTAs), unpacked as v' is formed
        uint32_t u2[SBV / 2];
#pragma unroll
        for (int t = 0; t < SBV / 2; ++t) u2[t] = 0u;
        auto fetch = [&](int r) {
            wait_copy(&full[r % kStages], (r / kStages) & 1);
            if (r < ncs && !ident) {
#pragma unroll
                for (int blk = 0; blk < SBV / kUB; ++blk) {
                    const uint4 *ur = reinterpret_cast<const uint4 *>(
                        stage(r) + S::u + ((size_t)blk * 64 + row) * kUB * 2);
                    const uint4 a = ur[0], c = ur[1];
                    u2[blk * 8 + 0] = a.x; u2[blk * 8 + 1] = a.y; u2[blk * 8 + 2] = a.z; u2[blk * 8 + 3] = a.w;
                    u2[blk * 8 + 4] = c.x; u2[blk * 8 + 5] = c.y; u2[blk * 8 + 6] = c.z; u2[blk * 8 + 7] = c.w;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[r % kStages]);
        };
        if (R > 0) fetch(0);
        for (int r = 0; r < ncs; ++r) {
            wait_mma(&bar_v[r & 1], (r >> 1) & 1);
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < SBV; cb += 32) {
                float d[32];
                tmem_ld32(tmem + lanebase + (r & 1) * SBV + cb, d);
#pragma unroll
                for (int t = 0; t < 32; t += 2) {
                    const uint32_t w = u2[(cb + t) / 2];
                    d[t] = __uint_as_float(w << 16) - d[t];
                    d[t + 1] = __uint_as_float(w & 0xffff0000u) - d[t + 1];
                }
#pragma unroll
                for (int c = 0; c < 32; c += 8)
                    *reinterpret_cast<uint4 *>(sVp + tile_off(row, cb + c, SBV)) = pack8_at(d + c);
                if (p.ck_vp) {  // v' of chunk c0 + r for the backward
                    unsigned char *t = static_cast<unsigned char *>(p.ck_vp) +
                                       unit_index(p, gc0 + c0 + r, hv) * (int64_t)(64 * p.V * 2);
#pragma unroll
                    for (int c = 0; c < 32; c += 8)
                        *reinterpret_cast<uint4 *>(t + tile_off(row, vb * SBV + cb + c, p.V)) =
                            pack8_at(d + c);
                }
            }
            tc_fence_before();
            fence_async_smem();
            __syncwarp();
            named_arrive(kBarV, kThrV);
            if (r + 1 < R) fetch(r + 1);
        }
    } else {
        // ------------------------------------- o warps: o_c = scale D1[64:128]
        // (for identity columns: Q_c, segment 1's response to its initial state)
        const int i = (warp - 6) * 32 + lane;  // row within the chunk
        const uint32_t lanebase = (uint32_t)(64 + (warp - 6) * 32) << 16;
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
        for (int r = 0; r < R; ++r) {
            if (r >= 1) {
                wait_mma(&bar_v[r & 1], (r >> 1) & 1);
                tc_fence_after();
                const int c = c0 + r - 1;
                const bool store = !read_flag(&abort_flag) && (ident || o != nullptr);
                const int orow = bos + c * kBT + i;
                unsigned char *qt = ident ? static_cast<unsigned char *>(p.qc) +
                                                ((gc0 + c) * p.HV + hv) * (int64_t)(64 * KK * 2)
                                          : nullptr;
                __nv_bfloat16 *op = o + (((size_t)b * p.T + orow) * p.HV + hv) * p.V + vb * SBV;
                // 32 columns at a time
#pragma unroll
                for (int cb = 0; cb < SBV; cb += 32) {
                    float d[32];
                    tmem_ld32(tmem + lanebase + (r & 1) * SBV + cb, d);
#pragma unroll
                    for (int t = 0; t < 32; ++t) d[t] *= p.scale;
                    if (store && ident) {
#pragma unroll
                        for (int cc = 0; cc < 32; cc += 8)
                            *reinterpret_cast<uint4 *>(qt + tile_off(i, vb * SBV + cb + cc, KK)) =
                                pack8_at(d + cc);
                    } else if (store && orow < eos) {
#pragma unroll
                        for (int cc = 0; cc < 32; cc += 8)
                            *reinterpret_cast<uint4 *>(op + cb + cc) = pack8_at(d + cc);
                    }
                }
                tc_fence_before();
            }
            // D1[r & 1] has been read: the MMA warp may overwrite it two rounds on.
            if (r < ncs) {
                __syncwarp();
                named_arrive(kBarV, kThrV);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, S::tmem_cols);
}

// ============================================================== fix kernel
// For split sequences: o_c += Q_c E0 over segment 1's chunks, and
// ht = P E0 + E1 in fp32.  Blocks [0, n_fix_o) take a pair of adjacent chunk
// slots of one value head: both Q tiles stacked as the 128 rows of one tcgen05
// MMA series against E0 in bf16 (N = dv), one pass per distinct sequence in the
// pair.  The remaining blocks take (sequence, head, 32 columns) of ht.
template <int KK, int VV>
struct FixSmem {
    static constexpr uint32_t e0 = 0;                      // [KK][VV] bf16, MN-major B tile
    static constexpr uint32_t q = e0 + KK * VV * 2;        // [128][KK] bf16: Q of the two chunks
    static constexpr uint32_t ht_need = 16 * KK * 4 + KK * 32 * 4;  // ht units: P rows + E0 block
    static constexpr uint32_t total = q + 128 * KK * 2 > ht_need ? q + 128 * KK * 2 : ht_need;
    static constexpr uint32_t tmem_cols = VV <= 64 ? 64 : (VV <= 128 ? 128 : 256);
};

template <int KK, int VV>
__global__ void __launch_bounds__(256) chunk_fix_tc_kernel(ChunkArgs p) {
    using S = FixSmem<KK, VV>;
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint64_t bar_q, bar_m, bar_e;
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (p.cu && !p.ctrl->valid) return;

    // Persistent over the units: first the (value head, chunk pair) units of
    // o_c += Q_c E0, then the small units of ht = P E0 + E1; CTA b takes units
    // b, b + gridDim.x, ...  Pairs with nothing in segment 1 cost nothing, and the
    // ht units land mostly on CTAs with one pair to fix.
    unsigned char *sE0 = sm + S::e0;
    unsigned char *sQ = sm + S::q;
    if (warp == 0) {
        tmem_alloc(&tslot, S::tmem_cols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_q, 1);
        mbar_init(&bar_m, 1);
        mbar_init(&bar_e, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
    uint32_t ph_e = 0;
    const int quad = warp & 3, half = warp >> 2;
    const int xr = quad >> 1, ir = (quad & 1) * 32 + (tid & 31);  // TMEM lane = row of the pair
    const int64_t pair_units = (int64_t)p.HV * ((p.slots + 1) / 2);
    const int64_t units = pair_units + (p.ht ? (int64_t)p.N * p.HV * (KK / 16) * (VV / 32) : 0);
    uint32_t ph_q = 0, ph_m = 0;
    int e0_key = -1;  // (sequence, head) whose E0 is in shared memory
    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        if (unit >= pair_units) {
            // ------------------------------------------- ht = P E0 + E1
            // unit = (sequence, head, 16-row block, 32-column block); thread: one
            // row, two columns, the full contraction over k.
            const int64_t hu = unit - pair_units;
            const int ncb = VV / 32, nrb = KK / 16;
            const int cb = (int)(hu % ncb);
            const int rb = (int)((hu / ncb) % nrb);
            const int hv = (int)((hu / ((int64_t)ncb * nrb)) % p.HV);
            const int n = (int)(hu / ((int64_t)ncb * nrb * p.HV));
            const size_t base = ((size_t)n * p.HV + hv) * KK;
            const int nc = p.cu ? p.chunk_start[n + 1] - p.chunk_start[n] : (p.T + kBT - 1) / kBT;
            const int d = rb * 16 + (tid >> 4), c = cb * 32 + (tid & 15) * 2;
            if (nc <= 1) {  // segment 1 is empty: P = I, E1 = 0, so ht = E0 exactly
                *reinterpret_cast<float2 *>(p.ht + (base + d) * VV + c) =
                    *reinterpret_cast<const float2 *>(p.e0 + (base + d) * VV + c);
                continue;
            }
            e0_key = -1;  // the shared E0 tile is overwritten here
            float *sP = reinterpret_cast<float *>(sm);   // [16][KK] rows of P
            float *sE = sP + 16 * KK;                    // [KK][32] columns of E0
            for (int idx = tid; idx < 16 * KK / 4; idx += 256) {
                const int r = idx / (KK / 4), k4 = (idx % (KK / 4)) * 4;
                *reinterpret_cast<float4 *>(sP + r * KK + k4) =
                    *reinterpret_cast<const float4 *>(p.pm + (base + rb * 16 + r) * KK + k4);
            }
            for (int idx = tid; idx < KK * 8; idx += 256) {
                const int r = idx >> 3, c4 = (idx & 7) * 4;
                *reinterpret_cast<float4 *>(sE + r * 32 + c4) =
                    *reinterpret_cast<const float4 *>(p.e0 + (base + r) * VV + cb * 32 + c4);
            }
            __syncthreads();
            float2 acc = *reinterpret_cast<const float2 *>(p.e1 + (base + d) * VV + c);
            const float *pr = sP + (tid >> 4) * KK;
            const float *er = sE + (tid & 15) * 2;
#pragma unroll 16
            for (int k = 0; k < KK; ++k) {
                const float pv = pr[k];
                const float2 e = *reinterpret_cast<const float2 *>(er + k * 32);
                acc.x = fmaf(pv, e.x, acc.x);
                acc.y = fmaf(pv, e.y, acc.y);
            }
            *reinterpret_cast<float2 *>(p.ht + (base + d) * VV + c) = acc;
            __syncthreads();
            continue;
        }
        const int64_t pu = unit;
        const int hv = (int)(pu % p.HV);
        const int64_t gpair = (pu / p.HV) * 2;
        int cb_[2], r0_[2], nr_[2], seq_[2];
        bool need[2];
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            int cl, ncn;
            need[x] = gpair + x < p.slots &&
                      locate_chunk(p, gpair + x, cb_[x], r0_[x], nr_[x], cl, &seq_[x], &ncn) &&
                      cl >= (ncn + 1) / 2;  // in segment 1
        }
        if (!need[0] && !need[1]) continue;
        if (tid == 0) {
            uint32_t bytes = 0;
            for (int x = 0; x < 2; ++x)
                if (need[x]) bytes += 64 * KK * 2;
            mbar_arrive_expect_tx(&bar_q, bytes);
            for (int x = 0; x < 2; ++x)
                if (need[x])
                    bulk_g2s(sQ + x * 64 * KK * 2,
                             static_cast<const unsigned char *>(p.qc) +
                                 ((gpair + x) * p.HV + hv) * (int64_t)(64 * KK * 2),
                             64 * KK * 2, &bar_q);
        }
        // this thread's o row segment (half of the columns), loaded now so its
        // latency overlaps E0, the Q copy and the MMA
        const bool has_o = need[xr] && ir < nr_[xr];
        uint4 *orow = reinterpret_cast<uint4 *>(
            o + (((size_t)cb_[xr] * p.T + r0_[xr] + ir) * p.HV + hv) * p.V + half * (VV / 2));
        uint4 ov[VV / 16];
        if (has_o) {
#pragma unroll
            for (int j = 0; j < VV / 16; ++j) ov[j] = orow[j];
        }
        // one pass per distinct sequence among the chunks that need the fix
        const int npass = (need[0] && need[1] && seq_[0] != seq_[1]) ? 2 : 1;
        for (int pass = 0; pass < npass; ++pass) {
            const int seq = npass == 2 ? seq_[pass] : (need[0] ? seq_[0] : seq_[1]);
            const int key = seq * p.HV + hv;
            const bool load_e0 = key != e0_key;  // E0 of this sequence, a bf16 MN-major tile
            if (load_e0 && tid == 0) {
                mbar_arrive_expect_tx(&bar_e, KK * VV * 2);
                bulk_g2s(sE0, static_cast<const unsigned char *>(p.e0b) + (size_t)key * KK * VV * 2,
                         KK * VV * 2, &bar_e);
            }
            e0_key = key;
            if (tid == 0) {
                if (pass == 0 && !mbar_wait(&bar_q, ph_q & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
                if (load_e0 && !mbar_wait(&bar_e, ph_e & 1, kWaitNs)) report(p.status, KDA_DEVICE_TIMEOUT);
                tc_fence_after();
                mma_bf16_seq<KK / 16, false>(tmem, sdesc(smem_addr(sQ), 128, KK * 16), 16,
                                             sdesc(smem_addr(sE0), VV * 16, 128), 2 * VV * 16 / 16,
                                             idesc_bf16(128, VV, false, true));
                mma_commit(&bar_m);
            }
            __syncwarp();
            if (load_e0) ++ph_e;
            if (!mbar_wait(&bar_m, ph_m & 1, kWaitNs) && tid == 0) report(p.status, KDA_DEVICE_TIMEOUT);
            ++ph_m;
            tc_fence_after();
            const bool mine = has_o && seq_[xr] == seq;
#pragma unroll
            for (int cc = 0; cc < VV / 2; cc += 32) {
                float d[32];
                tmem_ld32(tmem_at(tmem, quad * 32, half * (VV / 2) + cc), d);
                if (mine) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float f[8];
                        unpack8(ov[cc / 8 + j], f);
#pragma unroll
                        for (int t = 0; t < 8; ++t) f[t] += d[8 * j + t];
                        orow[cc / 8 + j] = pack8(f);
                    }
                }
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }
        ++ph_q;
    }
    if (warp == 0) tmem_dealloc(tmem, S::tmem_cols);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null when the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// A [rows][mid][inner] row-major tensor as a 3-D map with boxes of
// [64 rows][1][box_inner], 128-byte swizzle, zero fill out of bounds.
cudaError_t encode3(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elem,
                    uint64_t inner, uint64_t mid, uint64_t rows, uint32_t box_inner) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {inner, mid, rows};
    const cuuint64_t strides[2] = {inner * elem, mid * inner * elem};
    const cuuint32_t box[3] = {box_inner, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t prep_maps(const ChunkArgs &a, PrepMaps *m) {
    const uint64_t rows = (uint64_t)a.B * a.T;
    cudaError_t e = encode3(&m->q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K, a.H, rows, 64);
    if (e == cudaSuccess)
        e = encode3(&m->k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K, a.H, rows, 64);
    if (e == cudaSuccess)
        e = encode3(&m->g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.K, a.HV, rows, 32);
    if (e == cudaSuccess && a.V % 64 == 0 && a.V <= 128)
        e = encode3(&m->v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.V, a.HV, rows, 64);
    return e;
}

template <int KK, bool ACT, bool PADK>
cudaError_t launch_prep_t(const ChunkArgs &a, cudaStream_t st, int64_t cta_cap) {
    using S = PrepSmem<KK>;
    // Kernel attributes and the device's limits, set and read once per device.
    struct Info {
        int sms, regs_sm, smem_sm, num_regs, static_smem;
    };
    static DeviceOnce once;
    static Info info[64];
    int dev = 0;
    cudaError_t e = once.run(&dev, [](int d) {
        cudaError_t r = cudaFuncSetAttribute(chunk_prep_tc_kernel<KK, ACT, PADK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)S::total(256));
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(chunk_prep_tc_kernel<KK, ACT, PADK>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        Info x{};
        cudaFuncAttributes fa{};
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&x.sms, cudaDevAttrMultiProcessorCount, d);
        if (r == cudaSuccess)
            r = cudaDeviceGetAttribute(&x.regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, d);
        if (r == cudaSuccess)
            r = cudaDeviceGetAttribute(&x.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d);
        if (r == cudaSuccess) r = cudaFuncGetAttributes(&fa, chunk_prep_tc_kernel<KK, ACT, PADK>);
        if (r == cudaSuccess && fa.numRegs <= 0) r = cudaErrorInvalidDeviceFunction;
        x.num_regs = fa.numRegs;
        x.static_smem = (int)fa.sharedSizeBytes;
        if (r == cudaSuccess) info[d] = x;
        return r;
    });
    if (e != cudaSuccess) return e;
    const Info &I = info[dev];
    // Resident CTAs, from the kernel's registers and this dv's shared memory
    // (TMEM: 256 columns per CTA, at most two per SM).
    const uint32_t smem = S::total(a.V);
    const int sms = I.sms;
    const int by_regs = I.regs_sm / (((I.num_regs + 7) / 8 * 8) * 256);
    const int by_smem = I.smem_sm / (int)(smem + I.static_smem + 1024);
    int per_sm = by_regs < by_smem ? by_regs : by_smem;
    per_sm = per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm);
    int64_t ctas = (int64_t)sms * per_sm;
    if (cta_cap > 0 && cta_cap < ctas) ctas = cta_cap;
    const int64_t units = prep_units(a);
    if (units == 0) return cudaSuccess;
    const unsigned grid = (unsigned)(units < ctas ? units : ctas);
    PrepMaps maps{};
    if ((e = prep_maps(a, &maps)) != cudaSuccess) return e;
    prof_begin("chunk_prep_tc", st);
    chunk_prep_tc_kernel<KK, ACT, PADK><<<grid, 256, smem, st>>>(a, maps);
    prof_end(st);
    return cudaGetLastError();
}

// cta_cap > 0 bounds the grid (a pipelined launch's second part: the SMs the
// concurrent scan leaves free, two CTAs each).
template <int KK>
cudaError_t launch_prep(const ChunkArgs &a, cudaStream_t st, int64_t cta_cap = 0) {
    if (a.K == KK)
        return a.act.A_log ? launch_prep_t<KK, true, false>(a, st, cta_cap)
                           : launch_prep_t<KK, false, false>(a, st, cta_cap);
    return a.act.A_log ? launch_prep_t<KK, true, true>(a, st, cta_cap)
                       : launch_prep_t<KK, false, true>(a, st, cta_cap);
}

template <int KK, int SBV>
cudaError_t launch_scan(const ChunkArgs &a, cudaStream_t st) {
    using S = ScanSmem<KK, SBV>;
    static DeviceOnce once;
    int dev = 0;
    cudaError_t e = once.run(&dev, [](int) {
        return cudaFuncSetAttribute(chunk_scan_tc_kernel<KK, SBV>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::total);
    });
    if (e != cudaSuccess) return e;
    const int64_t per = a.split ? 2 * (a.V / SBV) + KK / SBV : a.V / SBV;
    const int64_t blocks = (int64_t)a.N * a.HV * per;
    if (blocks == 0) return cudaSuccess;
    prof_begin("chunk_scan_tc", st);
    chunk_scan_tc_kernel<KK, SBV><<<(unsigned)blocks, 320, S::total, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

template <int KK, int VV>
cudaError_t launch_fix(const ChunkArgs &a, cudaStream_t st) {
    using S = FixSmem<KK, VV>;
    static DeviceOnce once;
    static int slots[64];  // two resident CTAs per SM
    int dev = 0;
    cudaError_t e = once.run(&dev, [](int d) {
        cudaError_t r = cudaFuncSetAttribute(chunk_fix_tc_kernel<KK, VV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)S::total);
        int sms = 0;
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
        if (r == cudaSuccess) slots[d] = 2 * sms;
        return r;
    });
    if (e != cudaSuccess) return e;
    const int slots_on_device = slots[dev];
    const int64_t units = (a.ht ? (int64_t)a.N * a.HV * (KK / 16) * (VV / 32) : 0) +
                          (int64_t)a.HV * ((a.slots + 1) / 2);
    if (units == 0) return cudaSuccess;
    const unsigned grid = (unsigned)(units < slots_on_device ? units : slots_on_device);
    prof_begin("chunk_fix_tc", st);
    chunk_fix_tc_kernel<KK, VV><<<grid, 256, S::total, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

cudaError_t sm_count(int *out) {
    static DeviceOnce once;
    static int sms[64];
    int dev = 0;
    cudaError_t e = once.run(&dev, [](int d) {
        return cudaDeviceGetAttribute(&sms[d], cudaDevAttrMultiProcessorCount, d);
    });
    if (e != cudaSuccess) return e;
    *out = sms[dev];
    return cudaSuccess;
}

// 32 columns per CTA give the shortest rounds; once that needs more than one wave
// of CTAs (one per SM), 64 columns halve the CTAs and the shared-memory traffic
// per column, which wins (measured: -20% to -26% on multi-wave shapes).
bool scan_wide(int64_t N, int HV, int V, int sms) { return V % 64 == 0 && N * HV * (V / 32) > sms; }
// 128 columns per CTA once 64-column CTAs would not fit one wave of SMs: a round
// then shares its operand tiles over twice the columns.
bool scan_wider(int64_t N, int HV, int V, int sms) { return V % 128 == 0 && N * HV * (V / 64) > sms; }

template <int KK, int VV>
cudaError_t launch_scan_any(const ChunkArgs &a, cudaStream_t st, int sms) {
    if constexpr (VV % 128 == 0)
        if (scan_wider(a.N, a.HV, a.V, sms)) return launch_scan<KK, 128>(a, st);
    if constexpr (VV % 64 == 0)
        if (scan_wide(a.N, a.HV, a.V, sms)) return launch_scan<KK, 64>(a, st);
    return launch_scan<KK, 32>(a, st);
}

// The library's own stream for a pipelined launch's later preps (lowest
// priority), the event that forks it from the caller's stream and one event per
// later part that joins it back, one set per device.
struct PipeStreams {
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr;
    cudaEvent_t join[kMaxPipeParts] = {};
};
std::mutex g_pipe_mu;

cudaError_t pipe_streams(PipeStreams **out) {
    static PipeStreams per_dev[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    PipeStreams &ps = per_dev[dev];
    if (!ps.side) {
        int least = 0, greatest = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&ps.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        for (int i = 0; i < kMaxPipeParts; ++i)
            if ((e = cudaEventCreateWithFlags(&ps.join[i], cudaEventDisableTiming)) != cudaSuccess)
                return e;
        if ((e = cudaStreamCreateWithPriority(&ps.side, cudaStreamNonBlocking, least)) != cudaSuccess)
            return e;
    }
    *out = &ps;
    return cudaSuccess;
}

// Pipelined: the prep of part 0 on every SM, then on the caller's stream the
// scans of parts 0, 1, ... in order, each from the state the one before left in
// e0 (the last one to ht).  The preps of parts 1, 2, ... run one after another
// on the side stream, on the SMs the scans leave free, from the moment part 0's
// prep ends; part i's scan also waits on the event recorded after its prep.
// Part 0's scan follows its prep in stream order, so its CTAs are placed as soon
// as that prep ends, ahead of the side stream's prep, which waits on an event.
// No kernel waits for another: the streams and events order whole launches.
template <int KK, int VV>
cudaError_t launch_pipelined(const ChunkArgs &a, cudaStream_t st, int sms) {
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    PipeStreams *ps = nullptr;
    cudaError_t e = pipe_streams(&ps);
    if (e != cudaSuccess) return e;
    const PipePlan &pl = a.pipe;
    if (pl.parts < 2 || pl.parts > kMaxPipeParts) return cudaErrorInvalidValue;
    const int64_t scan_ctas = (int64_t)a.N * a.HV * (a.V / (scan_wide(a.N, a.HV, a.V, sms) ? 64 : 32));
    auto part = [&](int i, bool prep) {
        ChunkArgs x = a;
        if (prep) {
            x.prep_c0 = pl.cut[i];
            x.prep_c1 = pl.cut[i + 1];
        } else {
            x.scan_c0 = pl.cut[i];
            x.scan_c1 = pl.cut[i + 1];
        }
        return x;
    };
    if ((e = launch_prep<KK>(part(0, true), st)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ps->fork, st)) != cudaSuccess) return e;
    if ((e = launch_scan_any<KK, VV>(part(0, false), st, sms)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ps->side, ps->fork, 0)) != cudaSuccess) return e;
    for (int i = 1; i < pl.parts; ++i) {
        if ((e = launch_prep<KK>(part(i, true), ps->side, 2 * (sms - scan_ctas))) != cudaSuccess)
            return e;
        if ((e = cudaEventRecord(ps->join[i], ps->side)) != cudaSuccess) return e;
    }
    for (int i = 1; i < pl.parts; ++i) {
        if ((e = cudaStreamWaitEvent(st, ps->join[i], 0)) != cudaSuccess) return e;
        if ((e = launch_scan_any<KK, VV>(part(i, false), st, sms)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int KK, int VV>
cudaError_t launch_kv(const ChunkArgs &a, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    int sms = 0;
    if ((e = sm_count(&sms)) != cudaSuccess) return e;
    if (a.pipe.parts > 0) return launch_pipelined<KK, VV>(a, st, sms);
    if (a.slots > 0 && (e = launch_prep<KK>(a, st)) != cudaSuccess) return e;
    if (!a.split) return launch_scan_any<KK, VV>(a, st, sms);
    if ((e = launch_scan<KK, 64>(a, st)) != cudaSuccess) return e;
    if constexpr (VV % 64 == 0) return launch_fix<KK, VV>(a, st);
    return cudaErrorInvalidValue;
}

template <int KK>
cudaError_t launch_k(const ChunkArgs &a, cudaStream_t st) {
    switch (a.V) {
        case 32: return launch_kv<KK, 32>(a, st);
        case 64: return launch_kv<KK, 64>(a, st);
        case 96: return launch_kv<KK, 96>(a, st);
        case 128: return launch_kv<KK, 128>(a, st);
        case 160: return launch_kv<KK, 160>(a, st);
        case 192: return launch_kv<KK, 192>(a, st);
        case 224: return launch_kv<KK, 224>(a, st);
        case 256: return launch_kv<KK, 256>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool chunk_tc_supported(int K, int V) {
    return K >= 8 && K <= 128 && K % 8 == 0 && V >= 32 && V <= 256 && V % 32 == 0;
}

size_t chunk_tc_unit_bytes(int K, int V, bool bwd) {
    return tc_layout(K <= 64 ? 64 : 128, V, bwd).stride;
}

namespace {
PipePlan pipe_plan_search(int B, int HV, int K, int V, int T, int sms) {
    // Cost model in scan rounds.  At two prep CTAs per SM a wave of prep units
    // takes about 19 scan rounds (14.3 us against 0.78 us at K = V = 128, measured
    // on the whole GPU).  Serial: every unit, then 1 + nc rounds.  Pipelined: part
    // 0's units on every SM; part i's scan starts when part i - 1's scan has ended
    // and the side stream has prepped parts 1..i (on the SMs the scans leave
    // free), and takes 1 + its chunks rounds.  Each middle part (with more than
    // two parts) is the largest whose prep, started when the previous one ends,
    // is done by the time the previous part's scan is; the last part takes the
    // rest.  Every first cut and part count is tried.  At the training shape the
    // model picks chunk 76, the best of a measured sweep (181 us; 189 us at the
    // earlier cost of 23 rounds a wave, which picked chunk 91).
    constexpr int64_t kUnit = 19;
    PipePlan best_plan;
    if (!chunk_tc_supported(K, V) || B <= 0 || HV <= 0 || T <= 0 || sms <= 0) return best_plan;
    const int64_t nc = (T + kBT - 1) / kBT;
    const int64_t scan_ctas = (int64_t)B * HV * (V / (scan_wide(B, HV, V, sms) ? 64 : 32));
    if (2 * scan_ctas > sms || nc < 16) return best_plan;
    const int64_t free_ctas = 2 * (sms - scan_ctas), all_ctas = 2 * (int64_t)sms;
    const int64_t hb = (int64_t)B * HV;
    auto waves = [](int64_t units, int64_t ctas) { return (units + ctas - 1) / ctas; };
    int64_t best = waves(hb * nc, all_ctas) * kUnit + nc + 1;
    for (int parts = 2; parts <= kMaxPipeParts; ++parts) {
        for (int64_t m = 1; m + 1 <= nc; ++m) {
            PipePlan pl;
            pl.parts = parts;
            pl.cut[0] = 0;
            pl.cut[1] = (int)m;
            int64_t prep = waves(hb * m, all_ctas) * kUnit;  // side stream's clock
            int64_t scan_end = prep + m + 1;
            int64_t done = m;
            bool ok = true;
            for (int i = 1; i < parts; ++i) {
                int64_t n = nc - done;
                if (i + 1 < parts) {
                    // the largest part whose prep ends by scan_end (at least one chunk,
                    // and one chunk left for every later part)
                    const int64_t w = (scan_end - prep) / kUnit;
                    n = std::min(w * free_ctas / hb, nc - done - (parts - 1 - i));
                    if (n < 1) n = 1;
                }
                if (n < 1) { ok = false; break; }
                prep += waves(hb * n, free_ctas) * kUnit;
                scan_end = std::max(scan_end, prep) + n + 1;
                done += n;
                pl.cut[i + 1] = (int)done;
            }
            if (ok && done == nc && scan_end < best) {
                best = scan_end;
                best_plan = pl;
            }
        }
    }
    return best_plan;
}
}  // namespace

PipePlan chunk_tc_pipe_plan(int B, int HV, int K, int V, int T, int sms) {
    // The search costs O(nc) per part count: remembered for the last 16 shapes.
    struct Entry {
        int key[6];
        PipePlan plan;
    };
    static std::mutex mu;
    static Entry cache[16];
    static int used = 0, next = 0;
    const int key[6] = {B, HV, K, V, T, sms};
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (std::equal(key, key + 6, cache[i].key)) return cache[i].plan;
    Entry &e = cache[next];
    std::copy(key, key + 6, e.key);
    e.plan = pipe_plan_search(B, HV, K, V, T, sms);
    next = (next + 1) % 16;
    if (used < 16) ++used;
    return e.plan;
}

bool chunk_tc_split(int N, int HV, int K, int V, int T) {
    // Few long sequences: without a split the scan occupies under half of the
    // SMs for its whole sequential length; with it, every scan CTA still fits
    // one wave (at most 128 CTAs).
    return V % 64 == 0 && (int64_t)N * HV * (V / 32) <= 64 && T >= 1024 && (K == 64 || K == 128);
}

// K up to 64 runs in the 64-channel kernels, K up to 128 in the 128-channel ones;
// the channels past K are zero throughout (loads fill zeros, state rows past K
// are neither read nor stored).
cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st) {
    if (a.K <= 64) return launch_k<64>(a, st);
    return launch_k<128>(a, st);
}

}  // namespace kda

// kda_chunk_layout.cuh -- what the tensor-core chunk kernels share: the byte
// layout of a workspace unit (one chunk of one value head), the unit index, the
// map from a chunk slot to its rows, and bf16 packing helpers.  Not part of the
// public ABI.
#pragma once

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kUB = 16;               // column block of u in the workspace
constexpr float kSafeRange = 100.f;   // max |g2| (log2) for the split grams: factors
                                      // 2^-100..2^100 stay normal bf16, and the masked
                                      // upper triangle's sums stay finite in fp32
constexpr uint64_t kWaitNs = 1000000000ull;

// Byte layout of one workspace unit (chunk c, value head).
struct TcLayout {
    uint32_t aw;      // [128][dk] tile: rows 0..63 W~_c = W_c Diag(2^G_{c-1}) (W_0 for a
                      // sequence's first chunk), rows 64..127 qg_c (the scan
                      // applies the attention scale to o)
    uint32_t kgt;     // [64][dk] tile: kg_c (rows = tokens), read by the scan as an
                      // MN-major operand, i.e. as kg_c^T
    uint32_t mt;      // [64][64] tile: M_c = W_c kg_{c-1}^T (unused for a first chunk)
    uint32_t aqk;     // [64][64] tile: Aqk_c (unscaled, like qg_c)
    uint32_t u;       // [dv / kUB][64][kUB] bf16 row-major blocks: u_c
    uint32_t dec;     // [128] fp32: 2^G_c (0 beyond dk)
    // The backward's extra tiles (0 in a forward layout):
    uint32_t wb;      // [64][dk] tile: W_c itself (untilded)
    uint32_t akk;     // [64][64] tile: Akk_c = (I + L_c)^-1, zero above the diagonal
    uint32_t stride;  // unit size, 256-byte multiple
};

__host__ __device__ inline TcLayout tc_layout(int K, int V, bool bwd = false) {
    TcLayout L;
    uint32_t off = 0;
    L.aw = off;  off += 128u * K * 2;
    L.kgt = off; off += 64u * K * 2;
    L.mt = off;  off += 64u * 64 * 2;
    L.aqk = off; off += 64u * 64 * 2;
    L.u = off;   off += 64u * V * 2;
    L.dec = off; off += 128u * 4;
    L.wb = L.akk = 0;
    if (bwd) {
        L.wb = off;  off += 64u * K * 2;
        L.akk = off; off += 64u * 64 * 2;
    }
    L.stride = (uint32_t)align_up(off, 256);
    return L;
}

// Maps a chunk slot to its rows and its index within the sequence (and, when
// asked, the sequence and its chunk count).  Returns false for slots past the
// last chunk or when the offsets failed validation.
__device__ __forceinline__ bool locate_chunk(const ChunkArgs &p, int64_t gc, int &b, int &r0,
                                             int &nr, int &cl, int *seq = nullptr,
                                             int *seq_chunks = nullptr) {
    if (p.cu) {
        if (!p.ctrl->valid || gc >= p.ctrl->total_chunks) return false;
        const int n = upper_bound_minus_one(p.chunk_start, p.N + 1, (int)gc);
        cl = (int)gc - p.chunk_start[n];
        b = 0;
        r0 = p.cu[n] + kBT * cl;
        nr = min(kBT, p.cu[n + 1] - r0);
        if (seq) *seq = n;
        if (seq_chunks) *seq_chunks = p.chunk_start[n + 1] - p.chunk_start[n];
    } else {
        const int ntc = (p.T + kBT - 1) / kBT;
        b = (int)(gc / ntc);
        cl = (int)(gc % ntc);
        r0 = cl * kBT;
        nr = min(kBT, p.T - r0);
        if (seq) *seq = b;
        if (seq_chunks) *seq_chunks = ntc;
    }
    return nr > 0;
}

// Index of the workspace unit of chunk slot gc and value head hv.  Head-major: a
// head's consecutive chunks are adjacent, so the scan, which walks one head's
// chunks, stays within a few memory pages instead of stepping HV units per round.
__host__ __device__ __forceinline__ int64_t unit_index(const ChunkArgs &p, int64_t gc, int hv) {
    return (int64_t)hv * p.slots + gc;
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

}  // namespace
}  // namespace kda

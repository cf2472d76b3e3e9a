// tc_probe.cu -- a single-tile tcgen05 GEMM built from the library's own
// wrappers (kda_tc.cuh), used by tests/test_gpu_tc_probe.py to check the
// operand layouts, descriptors and TMEM read-back against a plain matmul.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_tc.cuh"

using namespace kda::tc;

// D[128][N] = A[128][Kd] * B[Kd][N]; mode bit 0: B MN-major, bit 1: A MN-major,
// bit 2: the K-major operands in the 128-byte swizzled layout (64-column blocks
// of rows x 128 bytes), bit 3: an MN-major B in the 128-byte swizzled layout
// (64-column blocks of Kd x 128 bytes).
__global__ void __launch_bounds__(128) tc_probe_kernel(const __nv_bfloat16 *A,
                                                       const __nv_bfloat16 *B, float *D, int N,
                                                       int Kd, int mode, int *err) {
    // no static shared memory: the dynamic region starts 1024-byte aligned, as the
    // swizzled layouts need (checked below)
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *sA = sm;
    unsigned char *sB = sm + 128 * Kd * 2;
    uint64_t &bar = *reinterpret_cast<uint64_t *>(sm + 190 * 1024);
    uint32_t &slot = *reinterpret_cast<uint32_t *>(sm + 190 * 1024 + 8);
    if (smem_addr(sm) & 1023u) {
        if (threadIdx.x == 0) atomicExch(err, 2);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool a_mn = mode & 2, b_mn = mode & 1, swk = mode & 4, swmn = mode & 8;
    if (warp == 0) {
        tmem_alloc(&slot, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    for (int idx = tid; idx < 128 * Kd; idx += 128) {
        const int m = idx / Kd, k = idx % Kd;
        const uint32_t off = a_mn ? tile_off(k, m, 128)
                                  : (swk ? sw128_off(m, k, 128 * 128) : tile_off(m, k, Kd));
        *reinterpret_cast<__nv_bfloat16 *>(sA + off) = A[idx];
    }
    for (int idx = tid; idx < Kd * N; idx += 128) {
        const int k = idx / N, n = idx % N;
        const uint32_t off = b_mn ? (swmn ? sw128_off(k, n, Kd * 128) : tile_off(k, n, N))
                                  : (swk ? sw128_off(n, k, N * 128) : tile_off(n, k, Kd));
        *reinterpret_cast<__nv_bfloat16 *>(sB + off) = B[idx];
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = slot;
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(128, N, a_mn, b_mn);
        if (swk || swmn) {
            // K step kk: K-major swizzled operands move 32 bytes inside an atom row
            // and a whole 64-column block every 4 steps; an MN-major swizzled B
            // moves 16 rows (two 8-row groups)
            for (int kk = 0; kk < Kd / 16; ++kk) {
                const uint32_t ksw = (kk & 3) * 32;
                const uint64_t a =
                    (swk && !a_mn) ? sdesc_sw128(smem_addr(sA) + (kk >> 2) * 128 * 128 + ksw, 16, 1024)
                                   : sdesc(smem_addr(sA) + kk * 2 * (a_mn ? 128 * 16 : 128),
                                           a_mn ? 128 * 16 : 128, a_mn ? 128 : Kd * 16);
                uint64_t b;
                if (b_mn && swmn)
                    b = sdesc_sw128(smem_addr(sB) + kk * 2048, Kd * 128, 1024);
                else if (!b_mn && swk)
                    b = sdesc_sw128(smem_addr(sB) + (kk >> 2) * N * 128 + ksw, 16, 1024);
                else
                    b = sdesc(smem_addr(sB) + kk * 2 * (b_mn ? N * 16 : 128), b_mn ? N * 16 : 128,
                              b_mn ? 128 : Kd * 16);
                mma_bf16(tmem, a, b, idesc, kk > 0);
            }
        } else {
            const uint32_t a_lbo = a_mn ? 128 * 16 : 128, a_sbo = a_mn ? 128 : Kd * 16;
            const uint32_t b_lbo = b_mn ? N * 16 : 128, b_sbo = b_mn ? 128 : Kd * 16;
            mma_bf16_k(tmem, smem_addr(sA), a_lbo, a_sbo, smem_addr(sB), b_lbo, b_sbo, idesc,
                       Kd / 16, 0);
        }
        mma_commit(&bar);
    }
    if (!mbar_wait(&bar, 0) && tid == 0) atomicExch(err, 1);
    tc_fence_after();
    for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
        tmem_ld16(tmem_at(tmem, warp * 32, c0), v);
#pragma unroll
        for (int j = 0; j < 16; ++j) D[(warp * 32 + lane) * N + c0 + j] = v[j];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

extern "C" int tc_probe(const void *A, const void *B, float *D, int N, int Kd, int mode, int *err,
                        cudaStream_t st) {
    if (N < 16 || N > 256 || N % 16 || Kd < 16 || Kd > 128 || Kd % 16) return -1;
    // Room for the tiles read with either descriptor interpretation.
    const int smem = 200 * 1024;
    cudaFuncSetAttribute(tc_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if ((mode & 8) && N % 64) return -1;  // swizzled MN-major B: whole 64-column blocks
    tc_probe_kernel<<<1, 128, smem, st>>>(static_cast<const __nv_bfloat16 *>(A),
                                          static_cast<const __nv_bfloat16 *>(B), D, N, Kd, mode,
                                          err);
    return (int)cudaGetLastError();
}

// TMEM read-back shapes: every warp stores lane * 1000 + column into its 32 lanes x
// 64 columns (32x32b stores), then reads them back with the 16-lane shape that
// hands the second half of the warp the same 16 lanes at a column offset
// (16x32bx2, offset 32): out[warp][thread][0..15].
__global__ void __launch_bounds__(128) tmem_ld16x2_kernel(float *out) {
    __shared__ uint32_t slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) {
        tmem_alloc(&slot, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = slot;
    const uint32_t row = tmem + ((uint32_t)(32 * warp) << 16);
    for (int c0 = 0; c0 < 64; c0 += 8) {
        uint32_t v[8];
        for (int j = 0; j < 8; ++j) v[j] = __float_as_uint((float)((32 * warp + lane) * 1000 + c0 + j));
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                         row + c0),
                     "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                     "r"(v[7])
                     : "memory");
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], 32;\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(row)
        : "memory");
    for (int j = 0; j < 16; ++j) out[(warp * 32 + lane) * 16 + j] = __uint_as_float(r[j]);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

extern "C" int tmem_ld16x2_probe(float *out, cudaStream_t st) {
    tmem_ld16x2_kernel<<<1, 128, 0, st>>>(out);
    return (int)cudaGetLastError();
}

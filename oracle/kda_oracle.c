/*
 * kda_oracle.c -- plain fp64 CPU reference for the KDA forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only tests/, the smoke check of __graft_entry__ and the
 * cpu_baseline leg of bench.py use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (the definition, written out token by token):
 *
 *   attention-gym PR #317 "Add fused recurrent_kda for decode and inference
 *   prefill", PR description: one recurrence per (sequence, head) over the
 *   tokens of that sequence, an fp32 (here fp64) state S of shape [K, V],
 *   `gate` the per-token log2 decay, queries scaled by 1/sqrt(K), packed
 *   sequences given by int32 offsets where repeated offsets are empty slots
 *   whose state passes through bitwise, and rows at or beyond the terminal
 *   offset outside the contract.
 *
 *   kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, preamble: all logs base 2,
 *   q/k of value head hv live at head h = hv / (HV/H), scale = K^-1/2.
 *
 *   The update of the gated delta rule with a per-channel diagonal decay:
 *       S_t = (I - beta_t k_t k_t^T) Diag(2^{g_t}) S_{t-1} + beta_t k_t v_t^T
 *       o_t = scale * S_t^T q_t
 *   is evaluated in the algebraically identical three-step form
 *       S      <- Diag(2^{g_t}) S                  (decay every row d)
 *       delta  <- beta_t (v_t - S^T k_t)           (delta-rule residual)
 *       S      <- S + k_t delta^T                  (rank-1 write)
 *   since (I - b k k^T) D S + b k v^T = D S + k (b (v - (D S)^T k))^T.
 *
 *   Optional L2 normalisation of q and k (kernel-fun 0.2.0.dev1 wheel,
 *   kda/autograd.py, ChunkKDAFunction.forward, use_qk_l2norm): each row is
 *   divided by sqrt(sum x^2 + eps), eps = 1e-6 (the pages do not print the
 *   value; this reading is recorded with the design notes).
 *
 * The gate cumsum (kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Stage 1 --
 * cumsum"): a chunk-local inclusive prefix sum per channel, chunks restarting
 * at every sequence start, times a caller-given multiplier.
 *
 * All arithmetic is double.  Inputs are passed as double arrays that the
 * caller produced by exact upcasts from the stored dtype (bf16 and fp32 are
 * exactly representable in double).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_ORACLE_L2NORM_EPS 1e-6

/* Return codes. */
enum { ORACLE_OK = 0, ORACLE_BAD_ARGS = 1, ORACLE_BAD_OFFSETS = 2, ORACLE_NOMEM = 3 };

int kda_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sequence n spans physical rows [*bos, *eos) of batch row *b. */
static void slot_bounds(const int32_t *cu, int T, int n, int *b, long *bos, long *eos) {
    if (cu) {
        *b = 0;
        *bos = cu[n];
        *eos = cu[n + 1];
    } else {
        *b = n;
        *bos = 0;
        *eos = T;
    }
}

static int check_offsets(const int32_t *cu, int N, int T) {
    if (!cu) return ORACLE_OK;
    if (cu[0] != 0) return ORACLE_BAD_OFFSETS;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return ORACLE_BAD_OFFSETS;
    if (cu[N] > T) return ORACLE_BAD_OFFSETS;
    return ORACLE_OK;
}

/*
 * kda_oracle_recurrent
 *   q, k  : [B, T, H, K]      v, o : [B, T, HV, V]
 *   g     : [B, T, HV, K]     (per-token log2 decay, multiplied by g_scale)
 *   beta  : [B, T, HV]
 *   h0    : [N, HV, K, V] or NULL (zeros)        ht : [N, HV, K, V] or NULL
 *   cu    : [N + 1] offsets or NULL (then N == B and every row is a sequence)
 *   o rows outside every sequence are left untouched.
 */
int kda_oracle_recurrent(const double *q, const double *k, const double *v, const double *g,
                         const double *beta, const double *h0, const int32_t *cu, int B, int T,
                         int H, int HV, int K, int V, int N, double scale, double g_scale,
                         int l2norm, double *o, double *ht) {
    if (B <= 0 || T < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || N < 0) return ORACLE_BAD_ARGS;
    if (HV % H != 0) return ORACLE_BAD_ARGS;
    if (cu ? (B != 1) : (N != B)) return ORACLE_BAD_ARGS;
    if (check_offsets(cu, N, T) != ORACLE_OK) return ORACLE_BAD_OFFSETS;
    const int group = HV / H;
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int n = 0; n < N; ++n) {
        for (int hv = 0; hv < HV; ++hv) {
            double *S = (double *)malloc(sizeof(double) * (size_t)K * V);
            double *qt = (double *)malloc(sizeof(double) * (size_t)K);
            double *kt = (double *)malloc(sizeof(double) * (size_t)K);
            double *delta = (double *)malloc(sizeof(double) * (size_t)V);
            if (!S || !qt || !kt || !delta) {
#pragma omp atomic write
                failed = 1;
                free(S); free(qt); free(kt); free(delta);
                continue;
            }
            const int h = hv / group;
            int b;
            long bos, eos;
            slot_bounds(cu, T, n, &b, &bos, &eos);
            const size_t state_off = ((size_t)n * HV + hv) * (size_t)K * V;

            if (h0)
                memcpy(S, h0 + state_off, sizeof(double) * (size_t)K * V);
            else
                for (size_t i = 0; i < (size_t)K * V; ++i) S[i] = 0.0;

            for (long t = bos; t < eos; ++t) {
                const size_t row = (size_t)b * T + (size_t)t; /* token index in [B*T] */
                const double *qsrc = q + (row * H + h) * (size_t)K;
                const double *ksrc = k + (row * H + h) * (size_t)K;
                const double *vt = v + (row * HV + hv) * (size_t)V;
                const double *gt = g + (row * HV + hv) * (size_t)K;
                const double bt = beta[row * HV + hv];
                double *ot = o + (row * HV + hv) * (size_t)V;

                double qn = 1.0, kn = 1.0;
                if (l2norm) {
                    double sq = 0.0, sk = 0.0;
                    for (int d = 0; d < K; ++d) {
                        sq += qsrc[d] * qsrc[d];
                        sk += ksrc[d] * ksrc[d];
                    }
                    qn = 1.0 / sqrt(sq + KDA_ORACLE_L2NORM_EPS);
                    kn = 1.0 / sqrt(sk + KDA_ORACLE_L2NORM_EPS);
                }
                for (int d = 0; d < K; ++d) {
                    qt[d] = qsrc[d] * qn;
                    kt[d] = ksrc[d] * kn;
                }

                /* S <- Diag(2^{g_t}) S */
                for (int d = 0; d < K; ++d) {
                    const double decay = exp2(g_scale * gt[d]);
                    double *Srow = S + (size_t)d * V;
                    for (int j = 0; j < V; ++j) Srow[j] *= decay;
                }
                /* delta <- beta_t (v_t - S^T k_t) */
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int d = 0; d < K; ++d) acc += S[(size_t)d * V + j] * kt[d];
                    delta[j] = bt * (vt[j] - acc);
                }
                /* S <- S + k_t delta^T */
                for (int d = 0; d < K; ++d) {
                    double *Srow = S + (size_t)d * V;
                    for (int j = 0; j < V; ++j) Srow[j] += kt[d] * delta[j];
                }
                /* o_t = scale * S^T q_t */
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int d = 0; d < K; ++d) acc += S[(size_t)d * V + j] * qt[d];
                    ot[j] = scale * acc;
                }
            }

            if (ht) {
                if (eos == bos && h0)
                    memcpy(ht + state_off, h0 + state_off, sizeof(double) * (size_t)K * V);
                else
                    memcpy(ht + state_off, S, sizeof(double) * (size_t)K * V);
            }
            free(S); free(qt); free(kt); free(delta);
        }
    }
    return failed ? ORACLE_NOMEM : ORACLE_OK;
}

/*
 * kda_oracle_gate_cumsum
 *   g, out : [B, T, HV, K].  For every sequence [bos, eos) and every row t in
 *   it, out[t] = g_scale * sum_{s = c(t)}^{t} g[s], where c(t) is the start of
 *   t's chunk: bos + chunk * floor((t - bos) / chunk).  Rows outside every
 *   sequence are left untouched.
 */
int kda_oracle_gate_cumsum(const double *g, const int32_t *cu, int B, int T, int HV, int K, int N,
                           int chunk, double g_scale, double *out) {
    if (B <= 0 || T < 0 || HV <= 0 || K <= 0 || N < 0 || chunk <= 0) return ORACLE_BAD_ARGS;
    if (cu ? (B != 1) : (N != B)) return ORACLE_BAD_ARGS;
    if (check_offsets(cu, N, T) != ORACLE_OK) return ORACLE_BAD_OFFSETS;

#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int n = 0; n < N; ++n) {
        for (int hv = 0; hv < HV; ++hv) {
            int b;
            long bos, eos;
            slot_bounds(cu, T, n, &b, &bos, &eos);
            for (long t = bos; t < eos; ++t) {
                const long start = bos + chunk * ((t - bos) / chunk);
                for (int d = 0; d < K; ++d) {
                    double acc = 0.0;
                    for (long s = start; s <= t; ++s)
                        acc += g[(((size_t)b * T + (size_t)s) * HV + hv) * (size_t)K + d];
                    out[(((size_t)b * T + (size_t)t) * HV + hv) * (size_t)K + d] = g_scale * acc;
                }
            }
        }
    }
    return ORACLE_OK;
}

/*
 * kda.h -- C ABI of the GB300 (sm_103a) library for KDA: the forward passes and
 * the recurrence's backward.
 *
 * KDA (Kimi Delta Attention) is a gated delta rule with a per-channel diagonal
 * decay.  Per (sequence n, value head hv), with q/k taken from head
 * h = hv / (HV / H), an fp32 state S of shape [K, V] evolves as
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(2^{g_t}) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t,            scale = K^{-1/2} unless given,
 *
 * with g_t <= 0 a base-2 log decay per channel (kernel-fun 0.2.0.dev1 sdist,
 * ALGORITHM.md, preamble; attention-gym PR #317 "Add fused recurrent_kda for
 * decode and inference prefill", PR description).
 *
 * Operations:
 *   kda_gate_cumsum    chunk-local gate cumsum (ALGORITHM.md, Stage 1)
 *   kda_chunk_fwd      chunked forward, BT = 64 (ALGORITHM.md, Stages 1-4)
 *   kda_recurrent_fwd  token-by-token forward for decode (PR #317)
 * each also as an *_act variant that applies the gate and beta activations to
 * raw inputs inside the op (kda_activation below), and
 *   kda_recurrent_bwd  the gradients of the recurrence (ALGORITHM.md, Backward),
 *                      also as kda_recurrent_bwd_act (gradients of the raw inputs)
 *   kda_chunk_bwd      the same gradients in the chunked form on the tensor cores
 *                      (ALGORITHM.md, Backward, the seven launches), also as
 *                      kda_chunk_bwd_act, and after kda_chunk_fwd_save (a forward
 *                      that keeps the backward's recomputed state) without the
 *                      recompute
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every tensor pointer is a DEVICE pointer owned by the caller, on
 * the current CUDA device.  The library allocates no memory and keeps no
 * global state beyond a per-process cache of device attributes and, once a
 * pipelined kda_chunk_fwd call has run on a device, one stream and two events
 * there (KDA_FLAG_SERIAL).  All work is enqueued on `stream` (NULL = the legacy
 * default stream); calls return without synchronising, except
 * kda_read_device_status.
 *
 * Layouts (all C-contiguous, row-major):
 *   q, k        [B, T, H, K]     dtype `shape->dtype`
 *   v, o        [B, T, HV, V]    dtype `shape->dtype`  (o has q's dtype)
 *   g, g_cum    [B, T, HV, K]    fp32 (the gate is per VALUE head)
 *   beta        [B, T, HV]       dtype `shape->dtype`
 *   h0, ht      [N, HV, K, V]    fp32, K-major state, one entry per sequence
 *   cu_seqlens  [N + 1]          int32, device resident
 * With cu_seqlens == NULL the batch is dense: N = B and row b is one sequence
 * of T tokens.  With cu_seqlens != NULL the batch is packed: B must be 1, T is
 * the physical capacity, and sequence n occupies rows [cu[n], cu[n+1]).
 * Packed-sequence contract (attention-gym PR #317, PR description; review
 * comments on offset validation): offsets must satisfy cu[0] == 0,
 * cu[n] <= cu[n+1] and cu[N] <= T.  Repeated offsets are empty slots whose
 * final state is h0 copied bit for bit (+0.0 when h0 is NULL).  Rows at or
 * beyond cu[N] are outside the contract: never written, and their input values
 * (NaN included) never reach any output.
 *
 * Errors.  Arguments the host can check are checked before anything is
 * enqueued; a failing call returns KDA_ERR_INVALID_ARG or KDA_ERR_UNSUPPORTED,
 * enqueues nothing, and kda_last_error_message() says why.  Offsets live on
 * the device and are validated there on every call (graph replay included):
 * invalid offsets never trap and never cause an out-of-bounds access; the
 * work they govern is skipped and bit KDA_DEVICE_BAD_CU_SEQLENS is OR-ed into
 * *dev_status (when dev_status is not NULL).  Outputs are unspecified for a
 * call whose status word reports an error.  The status word is only written
 * by OR; clear it with kda_clear_device_status.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Binary-compatible with cudaStream_t. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,      /* malformed arguments (host-detected)         */
    KDA_ERR_UNSUPPORTED = 2,      /* well-formed but outside the supported set    */
    KDA_ERR_BAD_CU_SEQLENS = 3,   /* reported via the device status word          */
    KDA_ERR_CUDA = 4,             /* a CUDA runtime call or a launch failed        */
    KDA_ERR_TIMEOUT = 5           /* a bounded on-device wait gave up              */
} kda_status;

typedef enum {
    KDA_DTYPE_F32 = 0,            /* q, k, v, beta, o in fp32                     */
    KDA_DTYPE_BF16 = 1            /* q, k, v, beta, o in bf16                     */
} kda_dtype;

/* shape->flags */
#define KDA_FLAG_QK_L2NORM   (1u << 0)  /* L2-normalise q and k rows inside the op:
                                           x / sqrt(sum x^2 + 1e-6)  (kernel-fun
                                           0.2.0.dev1 wheel, kda/autograd.py,
                                           use_qk_l2norm)                          */
#define KDA_FLAG_G_IS_CUMSUM (1u << 1)  /* kda_chunk_fwd only: g already holds the
                                           chunk-local cumsum (kda_gate_cumsum
                                           output with chunk_size 64)             */
#define KDA_FLAG_SPLIT_SCAN  (1u << 2)  /* kda_chunk_fwd, bf16 tensor-core path: for
                                           few long sequences (num_seqs * HV * V / 32
                                           <= 64, T >= 1024, V % 64 == 0) run each
                                           sequence's inter-chunk scan as two
                                           segments at once and compose them after
                                           (h_end = P h_start + E: context parallel
                                           within one GPU).  Needs a larger
                                           workspace (size it with the same flags);
                                           ignored elsewhere.                      */
#define KDA_FLAG_SERIAL      (1u << 3)  /* kda_chunk_fwd: run every launch on the
                                           caller's stream, one after the other.
                                           Without it, a dense bf16 input whose
                                           scan leaves at least half of the SMs
                                           idle is pipelined: while the scan of
                                           each sequence's first chunks runs on
                                           the caller's stream, the prep of the
                                           remaining chunks runs on a library-
                                           owned low-priority stream (forked from
                                           and joined back to the caller's stream
                                           with events, so graph capture sees one
                                           fork and one join) on the other SMs.    */

#define KDA_FLAG_BWD_SAVED   (1u << 4)  /* kda_chunk_bwd: the workspace holds what
                                           kda_chunk_fwd_save stored for the same
                                           inputs, shape and options, so the
                                           forward is not run again (the saved
                                           per-chunk tiles and states are read as
                                           they are; h0 is not read).  Refused by
                                           kda_chunk_fwd_save, ignored by the
                                           other entry points.                     */

#define KDA_FLAG_TEST_WAIT_TIMEOUT (1u << 31)
                                        /* Test hook, kda_chunk_fwd on the bf16
                                           tensor-core path: the scan kernel's MMA
                                           issuer first waits on a barrier that
                                           nothing signals, with a 2 us limit.  The
                                           wait gives up, KDA_DEVICE_TIMEOUT is set,
                                           and the kernel takes the path of any
                                           wait that runs out: no further MMA is
                                           issued, the copies already in flight are
                                           drained (bounded), every warp finishes
                                           its rounds and the kernel returns.  The
                                           outputs of such a call are unspecified;
                                           the context stays usable.  Ignored by
                                           the other kernels.                      */

/* Bits of the device status word. */
#define KDA_DEVICE_BAD_CU_SEQLENS (1 << 0)
#define KDA_DEVICE_TIMEOUT        (1 << 1)
#define KDA_DEVICE_INTERNAL       (1 << 2)  /* a launch found an internal invariant broken
                                               (e.g. the alignment of its shared memory)
                                               and skipped its work; reported as
                                               KDA_ERR_CUDA                            */
#define KDA_DEVICE_GATE_RANGE     (1 << 3)  /* kda_chunk_bwd: a chunk's gate range
                                               max |g2| (log2, chunk-local cumsum of
                                               g_scale g) exceeds 100, or is not
                                               finite; that chunk's gradients were not
                                               computed.  Reported as
                                               KDA_ERR_UNSUPPORTED                     */

typedef struct {
    int32_t B, T, H, HV, K, V;  /* see Layouts; HV % H == 0                         */
    int32_t num_seqs;           /* N: B when dense, len(cu_seqlens) - 1 when packed  */
    kda_dtype dtype;            /* of q, k, v, beta and o                           */
    float scale;                /* readout scale; <= 0 selects K^{-1/2}             */
    float g_scale;              /* multiplier applied to g before use: 1 for base-2
                                   log gates, 1/ln 2 for natural-log gates          */
    uint32_t flags;             /* KDA_FLAG_*                                       */
} kda_shape;

/*
 * Input activations applied inside the op (the *_act entry points).  Defined in
 * kernel-fun 0.2.0.dev1 wheel, kda/chain.py, gate_cumsum, and kda/ops.py,
 * chunk_kda (use_gate_in_kernel, use_beta_sigmoid_in_kernel, allow_neg_eigval);
 * sdist ALGORITHM.md, "Stage 1" note on the fused gate activation.
 *   A_log       [HV] fp32 device pointer, or NULL.  When set, g holds the raw
 *               gate pre-activation and the op uses, in g's place, the
 *               natural-log decay
 *                   -exp(A_log[hv]) * softplus(g[t, hv, d] + dt_bias[hv, d])
 *               (times shape->g_scale as always: 1/ln 2 for this form).
 *               softplus(x) = ln(1 + e^x), evaluated as x itself above 20.
 *   dt_bias     [HV, K] fp32 device pointer, or NULL (no bias); needs A_log.
 *   beta_scale  0: beta is the gate as given.  > 0: beta holds logits and the
 *               op uses sigmoid(beta) * beta_scale (1, or 2 to allow negative
 *               eigenvalues), rounded to the input dtype as the pages cast it to
 *               q's dtype.
 * The pages' lower_bound option has no formula there and is not provided.
 * A NULL kda_activation, or one with A_log == NULL and beta_scale == 0, is the
 * plain op.  The activation cannot be combined with KDA_FLAG_G_IS_CUMSUM.
 */
typedef struct {
    const float *A_log;
    const float *dt_bias;
    float beta_scale;
} kda_activation;

/*
 * kda_gate_cumsum -- chunk-local inclusive cumsum of the gate.
 * Defined in kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Stage 1 -- cumsum":
 *     g_cum[t, hv, d] = g_scale * sum_{s = c(t)}^{t} g[s, hv, d]
 * where c(t) is the first row of t's chunk, chunks of `chunk_size` rows being
 * counted from the first row of t's own sequence.  chunk_size == 1 is the
 * identity (times g_scale), as with attention-gym's bounded_gate_cumsum with
 * chunk_size=1 (PR #317, PR description).
 *   g, g_cum   [B, T, HV, K] fp32; must not alias; rows outside every sequence
 *              of g_cum are not written.
 *   chunk_size 1 <= chunk_size <= 64.
 *   Only B, T, H, HV, K, num_seqs and g_scale of *shape are used (H >= 1).
 */
kda_status kda_gate_cumsum(const float *g, float *g_cum, const int32_t *cu_seqlens,
                           const kda_shape *shape, int32_t chunk_size, int32_t *dev_status,
                           kda_stream_t stream);
/* kda_gate_cumsum with the gate activation of *act applied to g first (its
 * beta_scale is ignored). */
kda_status kda_gate_cumsum_act(const float *g, float *g_cum, const int32_t *cu_seqlens,
                               const kda_shape *shape, const kda_activation *act,
                               int32_t chunk_size, int32_t *dev_status, kda_stream_t stream);

/*
 * kda_chunk_fwd -- the chunked forward with chunks of BT = 64 rows.
 * Defined in kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Forward" (Stage 1
 * cumsum, Stage 2 intra/WY, Stage 3+4 scan + o); arguments and return contract
 * of kernel-fun 0.2.0.dev1 wheel, kda/ops.py, chunk_kda (o in q's dtype, ht
 * only when asked for, a NULL initial state meaning zeros).  Reaches the
 * result of the token recurrence above up to rounding.
 *   q, k, v, g, beta   inputs (Layouts).  g is the per-token log decay unless
 *                      KDA_FLAG_G_IS_CUMSUM is set.
 *   h0                 [N, HV, K, V] fp32 or NULL (zeros).
 *   o                  [B, T, HV, V] output, dtype of q.
 *   ht                 [N, HV, K, V] fp32 final state, or NULL (not stored).
 *                      May alias h0.
 *   workspace          device scratch of at least kda_chunk_workspace_size()
 *                      bytes, 256-byte aligned; its contents on entry do not
 *                      matter and on return are unspecified.  Calls that share
 *                      one workspace must be ordered on the GPU.
 *   stream             the call's work follows earlier work on `stream` and
 *                      later work on it sees the results.  Unless
 *                      KDA_FLAG_SERIAL is set, a dense bf16 call may run some
 *                      launches on a library stream forked from `stream` and
 *                      joined back to it with events (see KDA_FLAG_SERIAL);
 *                      such calls take a host-side lock while they enqueue.
 * Supported: K in {64, 128} with 1 <= V <= 256 (K, V multiples of 16 for bf16);
 * for bf16 also any K that is a multiple of 8 up to 128 when V is a multiple of
 * 32 up to 256 (the tensor-core kernels run such K padded with zero channels).
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                         const void *beta, const float *h0, const int32_t *cu_seqlens,
                         const kda_shape *shape, void *o, float *ht, void *workspace,
                         size_t workspace_bytes, int32_t *dev_status, kda_stream_t stream);
/* kda_chunk_fwd on raw g / beta with the activations of *act (see above). */
kda_status kda_chunk_fwd_act(const void *q, const void *k, const void *v, const float *g,
                             const void *beta, const float *h0, const int32_t *cu_seqlens,
                             const kda_shape *shape, const kda_activation *act, void *o,
                             float *ht, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, kda_stream_t stream);

/* Bytes of workspace kda_chunk_fwd needs for *shape (0 on invalid shapes).  For
 * shapes that may be pipelined it depends on the current device's SM count:
 * size the workspace with the device that will run the call current. */
size_t kda_chunk_workspace_size(const kda_shape *shape);
/* The same number under the name the boundary was first specified with. */
size_t kda_workspace_size(const kda_shape *shape);

/*
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd for callers that cannot allocate
 * device memory at call time (a runtime that owns a fixed, pre-planned memory
 * budget, a plugin host that forbids allocations outside its pool, or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device
 * synchronisation).  The pages have no counterpart to it: it is a property of
 * this library's interface, not of the method.
 *   Arguments, layouts, results and errors are those of kda_chunk_fwd, minus
 *   the workspace: the call uses a scratch array of KDA_NOALLOC_SCRATCH_BYTES
 *   built into the library, which every GPU that loads the library holds until
 *   the process exits.  Shapes whose kda_chunk_workspace_size exceeds it are
 *   rejected with KDA_ERR_UNSUPPORTED and a message; nothing is enqueued.
 *   The call allocates nothing and runs every launch on `stream`, one after
 *   the other (as with KDA_FLAG_SERIAL).  Its first call on a device looks up the
 *   array's device address (cudaGetSymbolAddress) and caches it.  With lazy
 *   module loading (the CUDA default) that lookup is what loads the array onto
 *   the device and reserves its 32 MiB, so it can fail for lack of device
 *   memory (KDA_ERR_CUDA with a message saying so) or wait on the device: make
 *   the first call on each device during set-up, before any stream capture.
 *   Every call on a device shares the one array, so calls that overlap on the
 *   GPU (different streams without ordering) race and give wrong results;
 *   serialise them.  The array keeps the last call's contents; nothing in it
 *   needs to start at zero.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (32u << 20)
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                                 const void *beta, const float *h0, const int32_t *cu_seqlens,
                                 const kda_shape *shape, void *o, float *ht, int32_t *dev_status,
                                 kda_stream_t stream);

/*
 * kda_recurrent_fwd -- token-by-token forward for decode and inference prefill.
 * Defined in attention-gym PR #317, PR description: one sequential scan over
 * the tokens of each (sequence, head, value block) with the [K, BV] fp32 state
 * held in registers, fp32 arithmetic whatever the input dtype, queries scaled
 * by 1/sqrt(K); work flattened onto grid x so that N * HV beyond 65535 works
 * (PR #317, review comment on grid Y).
 *   g         per-token log decay (KDA_FLAG_G_IS_CUMSUM is rejected).
 *   h0, ht    as for kda_chunk_fwd; ht == h0 (in-place decode) is allowed.
 * Supported: 1 <= K <= 256, 1 <= V (any size; value blocks of 128 columns).
 */
kda_status kda_recurrent_fwd(const void *q, const void *k, const void *v, const float *g,
                             const void *beta, const float *h0, const int32_t *cu_seqlens,
                             const kda_shape *shape, void *o, float *ht, int32_t *dev_status,
                             kda_stream_t stream);
/* kda_recurrent_fwd on raw g / beta with the activations of *act (see above). */
kda_status kda_recurrent_fwd_act(const void *q, const void *k, const void *v, const float *g,
                                 const void *beta, const float *h0, const int32_t *cu_seqlens,
                                 const kda_shape *shape, const kda_activation *act, void *o,
                                 float *ht, int32_t *dev_status, kda_stream_t stream);

/*
 * kda_recurrent_bwd -- gradients of the token recurrence: given do = dL/do and
 * dht = dL/dht, dq, dk, dv, dbeta, dg (with respect to the per-token gate g, the
 * same g kda_recurrent_fwd takes) and dh0.  The contract is kernel-fun
 * 0.2.0.dev1 sdist, ALGORITHM.md, "Backward" (kernel-fun wheel, kda/chain.py,
 * backward: dq, dk, dv, dbeta, dg, dh0; GVA gradients of q and k summed over the
 * value heads that share them); the result is computed for the recurrence the
 * chunked form reaches exactly, in fp32 whatever the input dtype.
 *   q, k, v, g, beta, h0, cu_seqlens, shape   as for kda_recurrent_fwd.
 *   dout               [B, T, HV, V], dtype of q.
 *   dht                [N, HV, K, V] fp32, or NULL (zero).
 *   dq, dk             [B, T, H, K] fp32 outputs; dv [B, T, HV, V]; dg [B, T, HV, K];
 *                      dbeta [B, T, HV]; dh0 [N, HV, K, V] or NULL (not stored).
 *                      Rows outside every sequence are zero.  dq, dk, dg and dbeta
 *                      are summed with atomic adds: their rounding order varies.
 *   workspace          kda_recurrent_bwd_workspace_size() bytes, 16-byte aligned:
 *                      the state at the start of every 8 tokens.
 *   flags              KDA_FLAG_QK_L2NORM: q, k are normalised inside the op (as in
 *                      the forward) and dq, dk are the gradients of the raw rows.
 * Supported: K <= 128, any V; not with KDA_FLAG_G_IS_CUMSUM.
 */
kda_status kda_recurrent_bwd(const void *q, const void *k, const void *v, const float *g,
                             const void *beta, const float *h0, const int32_t *cu_seqlens,
                             const kda_shape *shape, const void *dout, const float *dht,
                             float *dq, float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                             void *workspace, size_t workspace_bytes, int32_t *dev_status,
                             kda_stream_t stream);
/*
 * kda_recurrent_bwd on raw g / beta with the activations of *act (see
 * kda_activation): the forward is kda_recurrent_fwd_act's (or kda_chunk_fwd_act's)
 * and the gradients are those of its inputs.  The chain rule through the
 * activations (kernel-fun 0.2.0.dev1 wheel, kda/chain.py, gate_backward):
 *   dg       with respect to the raw gate g;
 *   dbeta    with respect to the raw beta logits when beta_scale > 0 (the
 *            rounding of the activated beta to the input dtype passes the
 *            gradient through);
 *   dA_log   [HV] fp32, required when act->A_log is set: sum over tokens and
 *            channels of dL/dg' * g', g' the activated gate (zeroed, then summed);
 *   ddt_bias [HV, K] fp32, required when act->dt_bias is set: the sum over tokens
 *            of dg (zeroed, then summed).
 * Both may be NULL when the corresponding input is not set; their rounding
 * order varies (atomic adds).
 */
kda_status kda_recurrent_bwd_act(const void *q, const void *k, const void *v, const float *g,
                                 const void *beta, const float *h0, const int32_t *cu_seqlens,
                                 const kda_shape *shape, const kda_activation *act,
                                 const void *dout, const float *dht, float *dq, float *dk,
                                 float *dv, float *dg, float *dbeta, float *dh0, float *dA_log,
                                 float *ddt_bias, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, kda_stream_t stream);
/* Bytes of workspace kda_recurrent_bwd needs for *shape (0 on invalid shapes). */
size_t kda_recurrent_bwd_workspace_size(const kda_shape *shape);

/*
 * kda_chunk_bwd -- the same gradients as kda_recurrent_bwd, computed in the chunked
 * form of kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Backward" (the seven launches:
 * recompute, re-scan, dAv, dhu, wy_dqkg, intra, dg cumsum; kernel-fun wheel,
 * kda/chain.py, backward) on the tensor cores: the forward's prep and scan run again
 * and store, per (chunk, value head), w, Akk, the state at the chunk's start and v';
 * a reverse scan forms dL/dv' and dL/dh per chunk; one kernel per (chunk, value
 * head) then forms dq, dk, dv, dbeta and dg.  Operands are bf16 (the inputs, the
 * checkpoints and the intermediate gradients), accumulation fp32.
 *   q, k, v, g, beta, h0, cu_seqlens, shape   as for kda_chunk_fwd.
 *   dout, dht, dq, dk, dv, dg, dbeta, dh0     as for kda_recurrent_bwd.  With
 *                      HV > H, dq and dk are summed over the value heads that share
 *                      a q/k head with atomic adds (their rounding order varies);
 *                      with HV == H every element is stored once and the result is
 *                      deterministic.  With cu_seqlens, rows outside every sequence
 *                      are zero.  A chunk refused for its gate range gets zero
 *                      gradients (and KDA_DEVICE_GATE_RANGE).
 *   workspace          kda_chunk_bwd_workspace_size() bytes, 256-byte aligned.
 *   flags              KDA_FLAG_QK_L2NORM (q, k normalised inside the op; dq, dk
 *                      are the raw rows' gradients), KDA_FLAG_SERIAL and
 *                      KDA_FLAG_BWD_SAVED (the workspace holds kda_chunk_fwd_save's
 *                      stores for these inputs: the recompute and re-scan are
 *                      skipped); a cumsummed gate takes kda_recurrent_bwd.
 * Supported: bf16, K = V = 128.  A chunk whose gate range is too wide raises
 * KDA_DEVICE_GATE_RANGE in *dev_status.  Tensors 16-byte aligned.
 */
kda_status kda_chunk_bwd(const void *q, const void *k, const void *v, const float *g,
                         const void *beta, const float *h0, const int32_t *cu_seqlens,
                         const kda_shape *shape, const void *dout, const float *dht, float *dq,
                         float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                         void *workspace, size_t workspace_bytes, int32_t *dev_status,
                         kda_stream_t stream);
/*
 * kda_chunk_bwd on raw g / beta with the activations of *act (see kda_activation), the
 * forward being kda_chunk_fwd_act's: the gradients of the raw inputs, dA_log and
 * ddt_bias as for kda_recurrent_bwd_act.  With KDA_FLAG_QK_L2NORM (either entry point)
 * the rows are normalised inside the op and dq, dk are the raw rows' gradients.  The
 * kernels form the gradients of the normalised rows and the activated gate and beta;
 * the chain rules follow in two elementwise passes (the ones kda_recurrent_bwd uses).
 */
kda_status kda_chunk_bwd_act(const void *q, const void *k, const void *v, const float *g,
                             const void *beta, const float *h0, const int32_t *cu_seqlens,
                             const kda_shape *shape, const kda_activation *act, const void *dout,
                             const float *dht, float *dq, float *dk, float *dv, float *dg,
                             float *dbeta, float *dh0, float *dA_log, float *ddt_bias,
                             void *workspace, size_t workspace_bytes, int32_t *dev_status,
                             kda_stream_t stream);
/*
 * kda_chunk_fwd_save -- the chunked forward of kda_chunk_fwd_act (act may be NULL:
 * kda_chunk_fwd), the same o and ht bit for bit, that also leaves in `workspace`
 * what kda_chunk_bwd re-derives in its first two stages (recompute and re-scan of
 * kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Backward"): per (chunk, value head)
 * the operand tiles, w, Akk, the state at the chunk's start and v', and every
 * sequence's final state.  A later kda_chunk_bwd (or _act) of the same inputs,
 * shape, options and workspace with KDA_FLAG_BWD_SAVED then starts at the reverse
 * scan: memory (kda_chunk_bwd_workspace_size bytes held from the forward to the
 * backward) for the forward's second run.
 *   arguments          as for kda_chunk_fwd_act; ht may be NULL.
 *   workspace          kda_chunk_bwd_workspace_size() bytes, 256-byte aligned,
 *                      owned by the caller and left untouched until the backward.
 *   flags              KDA_FLAG_QK_L2NORM and KDA_FLAG_SERIAL.
 * Supported: bf16, K = V = 128 (as kda_chunk_bwd).
 */
kda_status kda_chunk_fwd_save(const void *q, const void *k, const void *v, const float *g,
                              const void *beta, const float *h0, const int32_t *cu_seqlens,
                              const kda_shape *shape, const kda_activation *act, void *o,
                              float *ht, void *workspace, size_t workspace_bytes,
                              int32_t *dev_status, kda_stream_t stream);

/* Bytes of workspace kda_chunk_bwd needs for *shape (0 on invalid shapes).  As for
 * kda_chunk_workspace_size, a shape that may be packed (B == 1) is sized for packed
 * input, which covers a dense call of the same shape too. */
size_t kda_chunk_bwd_workspace_size(const kda_shape *shape);

/*
 * kda_read_device_status -- synchronise `stream`, copy the status word to
 * *host_bits (may be NULL) and map it to a status: KDA_OK when no bit is set,
 * KDA_ERR_BAD_CU_SEQLENS or KDA_ERR_TIMEOUT otherwise.  Does not clear it.
 */
kda_status kda_read_device_status(const int32_t *dev_status, int32_t *host_bits,
                                  kda_stream_t stream);

/* kda_clear_device_status -- enqueue a reset of the status word to 0. */
kda_status kda_clear_device_status(int32_t *dev_status, kda_stream_t stream);

/*
 * Stage timing for benchmarks (not needed for correct use).  While enabled,
 * every kernel the library enqueues is bracketed by two CUDA events recorded
 * on the caller's stream; do not enable it around stream capture.
 * kda_profile_report synchronises the recorded events and writes up to
 * max_entries rows: the kernel's name (NUL-separated into names, at most
 * names_len bytes), its summed duration in milliseconds and its launch count.
 * It returns the number of rows (or -1 on a CUDA error).  Reset clears the
 * totals.  Process-wide, guarded by a mutex.
 */
kda_status kda_profile_enable(int enable);
int kda_profile_report(char *names, size_t names_len, double *total_ms, int64_t *launches,
                       int max_entries);
void kda_profile_reset(void);

/*
 * Peak fp32 FMA throughput of the current device, measured: a kernel of 16
 * independent FMA chains per thread on 8 x 256 threads per SM, timed with CUDA
 * events on `stream` (best of three after a warm-up launch), in TFLOP/s (two
 * flops per FMA).  The roofline denominator for the fp32-bound kernels (the
 * recurrent prefill and backward).  Synchronises the stream.
 */
kda_status kda_measure_fp32_fma_peak(double *tflops, kda_stream_t stream);

/* Static text for a status code. */
const char *kda_status_string(kda_status status);

/* Reason for the most recent non-OK return on the calling host thread. */
const char *kda_last_error_message(void);

/* Library version, "major.minor.patch". */
const char *kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */

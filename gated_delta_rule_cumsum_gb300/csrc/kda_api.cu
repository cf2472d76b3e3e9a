// kda_api.cu -- the extern "C" entry points declared in include/kda.h:
// host-side argument checks, workspace carving and kernel launches.
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "kda_internal.cuh"

namespace {

thread_local std::string g_last_error;

kda_status fail(kda_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

kda_status cuda_fail(cudaError_t e, const char *where) {
    return fail(KDA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr uint32_t kKnownFlags = KDA_FLAG_QK_L2NORM | KDA_FLAG_G_IS_CUMSUM |
                                  KDA_FLAG_SPLIT_SCAN | KDA_FLAG_SERIAL | KDA_FLAG_BWD_SAVED |
                                  KDA_FLAG_TEST_WAIT_TIMEOUT;

// Checks shared by the three operations.  `need_h` also checks H and HV % H.
kda_status check_common(const char *op, const kda_shape *s, const int32_t *cu) {
    if (!s) return fail(KDA_ERR_INVALID_ARG, "%s: shape is NULL", op);
    if (s->B <= 0 || s->T < 0 || s->H <= 0 || s->HV <= 0 || s->K <= 0 || s->V <= 0)
        return fail(KDA_ERR_INVALID_ARG,
                    "%s: sizes must be positive (B=%d T=%d H=%d HV=%d K=%d V=%d)", op, s->B, s->T,
                    s->H, s->HV, s->K, s->V);
    if (s->HV % s->H != 0)
        return fail(KDA_ERR_INVALID_ARG, "%s: HV=%d must be divisible by H=%d", op, s->HV, s->H);
    if (s->HV > 65535) return fail(KDA_ERR_UNSUPPORTED, "%s: HV=%d > 65535", op, s->HV);
    if (cu) {
        if (s->B != 1)
            return fail(KDA_ERR_INVALID_ARG, "%s: packed sequences (cu_seqlens) need B == 1, got %d",
                        op, s->B);
        if (s->num_seqs < 0)
            return fail(KDA_ERR_INVALID_ARG, "%s: num_seqs=%d < 0", op, s->num_seqs);
    } else if (s->num_seqs != s->B) {
        return fail(KDA_ERR_INVALID_ARG, "%s: num_seqs=%d must equal B=%d without cu_seqlens", op,
                    s->num_seqs, s->B);
    }
    if (s->dtype != KDA_DTYPE_F32 && s->dtype != KDA_DTYPE_BF16)
        return fail(KDA_ERR_INVALID_ARG, "%s: unknown dtype %d", op, (int)s->dtype);
    if (s->flags & ~kKnownFlags)
        return fail(KDA_ERR_UNSUPPORTED, "%s: unknown flag bits 0x%x", op, s->flags & ~kKnownFlags);
    if (!std::isfinite(s->g_scale))
        return fail(KDA_ERR_INVALID_ARG, "%s: g_scale is not finite", op);
    // Element counts must fit comfortably in 64-bit index arithmetic and rows in int32.
    const double elems = (double)s->B * s->T * s->HV * (s->K > s->V ? s->K : s->V);
    if (elems > 4e18 || (double)s->B * s->T > INT_MAX)
        return fail(KDA_ERR_UNSUPPORTED, "%s: tensor too large", op);
    return KDA_OK;
}

float resolve_scale(const kda_shape *s) {
    return s->scale > 0.f ? s->scale : 1.0f / std::sqrt((float)s->K);
}

kda_status check_fwd_pointers(const char *op, const kda_shape *s, const void *q, const void *k,
                              const void *v, const float *g, const void *beta, const void *o,
                              const int32_t *cu) {
    const bool has_rows = (int64_t)s->B * s->T > 0;
    if (has_rows && (!q || !k || !v || !g || !beta || !o))
        return fail(KDA_ERR_INVALID_ARG, "%s: q, k, v, g, beta and o must be non-NULL", op);
    if (cu == nullptr && s->num_seqs != s->B)
        return fail(KDA_ERR_INVALID_ARG, "%s: num_seqs must equal B", op);
    return KDA_OK;
}

struct ChunkWs {
    size_t ctrl, chunk_start, units, total, unit_bytes;
    int64_t slots;
    bool split;
    size_t qc, e0, e1, pm, e0b;  // split launches (e0 also pipelined ones)
    kda::PipePlan pipe;          // parts > 0: a dense call is pipelined in these parts
};

// The tensor-core path serves bf16 inputs whose K and V it supports; fp32
// inputs (and bf16 shapes outside that set) take the fp32 SIMT path.
bool use_tc(const kda_shape *s) {
    return s->dtype == KDA_DTYPE_BF16 && kda::chunk_tc_supported(s->K, s->V);
}

// The current device's SM count (cached per device); false when no device answers.
bool device_sm_count(int *out) {
    static kda::DeviceOnce once;
    static int cache[64];
    int dev = 0;
    if (once.run(&dev, [](int d) {
            return cudaDeviceGetAttribute(&cache[d], cudaDevAttrMultiProcessorCount, d);
        }) != cudaSuccess)
        return false;
    *out = cache[dev];
    return true;
}

// `bwd`: the units of kda_chunk_bwd's re-run of the forward (tensor-core path,
// with the backward's extra tiles; never split).
ChunkWs chunk_ws_layout(const kda_shape *s, bool packed, bool bwd = false) {
    ChunkWs L;
    L.slots = kda::chunk_slots(*s, packed);
    L.unit_bytes = use_tc(s) ? kda::chunk_tc_unit_bytes(s->K, s->V, bwd)
                             : kda::chunk_simt_unit_bytes(s->K, s->V);
    L.ctrl = 0;
    L.chunk_start = 256;
    L.units = L.chunk_start + kda::align_up(sizeof(int32_t) * ((size_t)s->num_seqs + 1), 256);
    L.total = L.units + (size_t)L.slots * s->HV * L.unit_bytes;
    L.split = !bwd && (s->flags & KDA_FLAG_SPLIT_SCAN) && use_tc(s) &&
              kda::chunk_tc_split(s->num_seqs, s->HV, s->K, s->V, s->T);
    L.qc = L.e0 = L.e1 = L.pm = L.e0b = 0;
    L.pipe = kda::PipePlan{};
    if (!L.split && use_tc(s) && !(s->flags & KDA_FLAG_SERIAL)) {
        // Sized the same for dense and packed shapes (only dense calls pipeline;
        // the workspace size cannot tell a B = 1 dense call from a packed one).
        int sms = 0;
        if (device_sm_count(&sms)) L.pipe = kda::chunk_tc_pipe_plan(s->B, s->HV, s->K, s->V, s->T, sms);
        if (L.pipe.parts > 0) {
            L.e0 = kda::align_up(L.total, 256);
            L.total = L.e0 + (size_t)s->B * s->HV * s->K * s->V * 4;
        }
    }
    if (L.split) {
        const size_t nh = (size_t)s->num_seqs * s->HV;
        L.qc = kda::align_up(L.total, 256);
        L.e0 = kda::align_up(L.qc + (size_t)L.slots * s->HV * 64 * s->K * 2, 256);
        L.e1 = kda::align_up(L.e0 + nh * s->K * s->V * 4, 256);
        L.pm = kda::align_up(L.e1 + nh * s->K * s->V * 4, 256);
        L.e0b = kda::align_up(L.pm + nh * s->K * s->K * 4, 256);
        L.total = L.e0b + nh * s->K * s->V * 2;
    }
    return L;
}

// kda_chunk_bwd's workspace: the forward's (with the backward's unit tiles),
// then per unit the checkpoints h_c ([K][V] bf16) and v'_c ([64][V]), and the
// reverse scan's dL/dh_{c+1} ([K][V]) and dL/dv'_c ([64][V]); the final states
// ([N][HV][K][V] fp32), per unit [V/32][K] fp32 sums of h_{c+1} dh_{c+1}, and the
// state gradient where a pipelined call's two reverse-scan parts meet.
struct ChunkBwdWs {
    ChunkWs f;
    size_t ck_h, ck_vp, dhn, dvp, hend, dgs, dhm, total;
};
// The same for every flag a kda_chunk_fwd_save / kda_chunk_bwd pair may differ in
// (KDA_FLAG_SERIAL, KDA_FLAG_BWD_SAVED): the backward reads the forward's tiles where
// the forward put them.
ChunkBwdWs chunk_bwd_ws_layout(const kda_shape *s, bool packed) {
    ChunkBwdWs W;
    kda_shape sp = *s;
    sp.flags &= ~(uint32_t)(KDA_FLAG_SERIAL | KDA_FLAG_BWD_SAVED);
    W.f = chunk_ws_layout(&sp, packed, true);
    const size_t units = (size_t)W.f.slots * s->HV;
    const size_t hb = (size_t)s->K * s->V * 2, vb = (size_t)64 * s->V * 2;
    W.ck_h = kda::align_up(W.f.total, 256);
    W.ck_vp = W.ck_h + units * hb;
    W.dhn = W.ck_vp + units * vb;
    W.dvp = W.dhn + units * hb;
    W.hend = kda::align_up(W.dvp + units * vb, 256);
    W.dgs = kda::align_up(W.hend + (size_t)s->num_seqs * s->HV * s->K * s->V * 4, 256);
    W.dhm = kda::align_up(W.dgs + units * (size_t)(s->V / 32) * s->K * 4, 256);
    W.total = W.dhm + (size_t)s->num_seqs * s->HV * s->K * s->V * 4;
    return W;
}

// kda_activation -> the kernels' GateAct, with its argument checks.
kda_status resolve_act(const char *op, const kda_shape *s, const kda_activation *act,
                       kda::GateAct *out) {
    *out = kda::GateAct();
    if (!act) return KDA_OK;
    if (act->dt_bias && !act->A_log)
        return fail(KDA_ERR_INVALID_ARG, "%s: dt_bias needs A_log", op);
    if (!(act->beta_scale >= 0.f) || !std::isfinite(act->beta_scale))
        return fail(KDA_ERR_INVALID_ARG, "%s: beta_scale must be 0 or a positive finite scale", op);
    if (act->A_log && (s->flags & KDA_FLAG_G_IS_CUMSUM))
        return fail(KDA_ERR_INVALID_ARG, "%s: the gate activation needs the per-token gate, not "
                    "KDA_FLAG_G_IS_CUMSUM", op);
    out->A_log = act->A_log;
    out->dt_bias = act->dt_bias;
    out->beta_scale = act->beta_scale;
    return KDA_OK;
}

kda_status check_chunk_support(const char *op, const kda_shape *s) {
    if (use_tc(s)) return KDA_OK;
    if (s->K != 64 && s->K != 128)
        return fail(KDA_ERR_UNSUPPORTED,
                    "%s: K=%d (supported: 64, 128; for bf16 with V a multiple of 32 up to 256, "
                    "any multiple of 8 up to 128)", op, s->K);
    if (s->V > 256) return fail(KDA_ERR_UNSUPPORTED, "%s: V=%d > 256", op, s->V);
    return KDA_OK;
}

}  // namespace

namespace kda {
// Lets other translation units of the library report a reason through
// kda_last_error_message.
void set_last_error(const char *msg) { g_last_error = msg; }
}  // namespace kda

extern "C" {

const char *kda_version(void) { return "0.1.0"; }

const char *kda_status_string(kda_status st) {
    switch (st) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_BAD_CU_SEQLENS: return "KDA_ERR_BAD_CU_SEQLENS";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    }
    return "KDA_ERR_UNKNOWN";
}

const char *kda_last_error_message(void) { return g_last_error.c_str(); }

kda_status kda_gate_cumsum(const float *g, float *g_cum, const int32_t *cu_seqlens,
                           const kda_shape *shape, int32_t chunk_size, int32_t *dev_status,
                           kda_stream_t stream) {
    return kda_gate_cumsum_act(g, g_cum, cu_seqlens, shape, nullptr, chunk_size, dev_status,
                               stream);
}

kda_status kda_gate_cumsum_act(const float *g, float *g_cum, const int32_t *cu_seqlens,
                               const kda_shape *shape, const kda_activation *act,
                               int32_t chunk_size, int32_t *dev_status, kda_stream_t stream) {
    const char *op = "kda_gate_cumsum";
    kda_status st = check_common(op, shape, cu_seqlens);
    if (st != KDA_OK) return st;
    kda::GateAct ga;
    if ((st = resolve_act(op, shape, act, &ga)) != KDA_OK) return st;
    if (chunk_size < 1 || chunk_size > 64)
        return fail(KDA_ERR_UNSUPPORTED, "%s: chunk_size=%d (supported: 1..64)", op, chunk_size);
    if ((int64_t)shape->B * shape->T > 0) {
        if (!g || !g_cum) return fail(KDA_ERR_INVALID_ARG, "%s: g and g_cum must be non-NULL", op);
        if (g == g_cum) return fail(KDA_ERR_INVALID_ARG, "%s: g_cum must not alias g", op);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (cu_seqlens) {
        e = kda::launch_validate_offsets(cu_seqlens, shape->num_seqs, shape->T, dev_status, nullptr,
                                         nullptr, s);
        if (e != cudaSuccess) return cuda_fail(e, op);
    }
    e = kda::launch_gate_cumsum(g, g_cum, cu_seqlens, *shape, ga, chunk_size, s);
    if (e != cudaSuccess) return cuda_fail(e, op);
    g_last_error.clear();
    return KDA_OK;
}

kda_status kda_recurrent_fwd(const void *q, const void *k, const void *v, const float *g,
                             const void *beta, const float *h0, const int32_t *cu_seqlens,
                             const kda_shape *shape, void *o, float *ht, int32_t *dev_status,
                             kda_stream_t stream) {
    return kda_recurrent_fwd_act(q, k, v, g, beta, h0, cu_seqlens, shape, nullptr, o, ht,
                                 dev_status, stream);
}

kda_status kda_recurrent_fwd_act(const void *q, const void *k, const void *v, const float *g,
                                 const void *beta, const float *h0, const int32_t *cu_seqlens,
                                 const kda_shape *shape, const kda_activation *act, void *o,
                                 float *ht, int32_t *dev_status, kda_stream_t stream) {
    const char *op = "kda_recurrent_fwd";
    kda_status st = check_common(op, shape, cu_seqlens);
    if (st != KDA_OK) return st;
    kda::GateAct ga;
    if ((st = check_fwd_pointers(op, shape, q, k, v, g, beta, o, cu_seqlens)) != KDA_OK) return st;
    if (shape->flags & KDA_FLAG_G_IS_CUMSUM)
        return fail(KDA_ERR_UNSUPPORTED, "%s: g is the per-token gate; KDA_FLAG_G_IS_CUMSUM is "
                    "for kda_chunk_fwd", op);
    if ((st = resolve_act(op, shape, act, &ga)) != KDA_OK) return st;
    if (shape->K > 256) return fail(KDA_ERR_UNSUPPORTED, "%s: K=%d > 256", op, shape->K);
    const int64_t blocks = (int64_t)shape->num_seqs * shape->HV * ((shape->V + 127) / 128);
    if (blocks > INT_MAX) return fail(KDA_ERR_UNSUPPORTED, "%s: grid too large", op);
    kda::RecurrentArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.cu = cu_seqlens;
    a.o = o; a.ht = ht; a.status = dev_status;
    a.B = shape->B; a.T = shape->T; a.H = shape->H; a.HV = shape->HV; a.K = shape->K;
    a.V = shape->V; a.N = shape->num_seqs;
    a.scale = resolve_scale(shape);
    a.g_scale = shape->g_scale;
    a.l2norm = (shape->flags & KDA_FLAG_QK_L2NORM) ? 1 : 0;
    a.act = ga;
    cudaError_t e = kda::launch_recurrent(a, shape->dtype, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, op);
    g_last_error.clear();
    return KDA_OK;
}

size_t kda_recurrent_bwd_workspace_size(const kda_shape *shape) {
    if (!shape || shape->K <= 0 || shape->V <= 0 || shape->HV <= 0 || shape->B <= 0 ||
        shape->T < 0 || shape->num_seqs < 0)
        return 0;
    return kda::recurrent_bwd_ckpt_bytes(shape->B, shape->T, shape->num_seqs, shape->HV, shape->K,
                                         shape->V);
}

kda_status kda_recurrent_bwd(const void *q, const void *k, const void *v, const float *g,
                             const void *beta, const float *h0, const int32_t *cu_seqlens,
                             const kda_shape *shape, const void *dout, const float *dht, float *dq,
                             float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                             void *workspace, size_t workspace_bytes, int32_t *dev_status,
                             kda_stream_t stream) {
    return kda_recurrent_bwd_act(q, k, v, g, beta, h0, cu_seqlens, shape, nullptr, dout, dht, dq,
                                 dk, dv, dg, dbeta, dh0, nullptr, nullptr, workspace,
                                 workspace_bytes, dev_status, stream);
}

kda_status kda_recurrent_bwd_act(const void *q, const void *k, const void *v, const float *g,
                                 const void *beta, const float *h0, const int32_t *cu_seqlens,
                                 const kda_shape *shape, const kda_activation *act,
                                 const void *dout, const float *dht, float *dq, float *dk,
                                 float *dv, float *dg, float *dbeta, float *dh0, float *dA_log,
                                 float *ddt_bias, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, kda_stream_t stream) {
    const char *op = "kda_recurrent_bwd";
    kda_status st = check_common(op, shape, cu_seqlens);
    if (st != KDA_OK) return st;
    kda::GateAct ga;
    if ((st = resolve_act(op, shape, act, &ga)) != KDA_OK) return st;
    if ((ga.A_log && !dA_log) || (ga.dt_bias && !ddt_bias))
        return fail(KDA_ERR_INVALID_ARG, "%s: dA_log (and ddt_bias with dt_bias) must be non-NULL "
                    "with the gate activation", op);
    if ((st = check_fwd_pointers(op, shape, q, k, v, g, beta, dout, cu_seqlens)) != KDA_OK) return st;
    if (shape->flags & KDA_FLAG_G_IS_CUMSUM)
        return fail(KDA_ERR_UNSUPPORTED, "%s: g is the per-token gate; KDA_FLAG_G_IS_CUMSUM is "
                    "for kda_chunk_fwd", op);
    if (shape->K > 128) return fail(KDA_ERR_UNSUPPORTED, "%s: K=%d > 128", op, shape->K);
    const bool has_rows = (int64_t)shape->B * shape->T > 0;
    if (has_rows && (!dq || !dk || !dv || !dg || !dbeta))
        return fail(KDA_ERR_INVALID_ARG, "%s: dq, dk, dv, dg and dbeta must be non-NULL", op);
    const size_t need = kda_recurrent_bwd_workspace_size(shape);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(KDA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", op, need,
                    workspace_bytes);
    if ((uintptr_t)workspace % 16 != 0)
        return fail(KDA_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", op);
    const int64_t blocks = (int64_t)shape->num_seqs * shape->HV * ((shape->V + 31) / 32);
    if (blocks > INT_MAX) return fail(KDA_ERR_UNSUPPORTED, "%s: grid too large", op);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // dq, dk, dg, dbeta accumulate over value columns (and value heads); dv and rows
    // outside every sequence are zero unless written.
    const size_t rows = (size_t)shape->B * shape->T;
    cudaError_t e = cudaSuccess;
    if (rows > 0) {
        const size_t zero[5][2] = {{(size_t)dq, rows * shape->H * shape->K},
                                   {(size_t)dk, rows * shape->H * shape->K},
                                   {(size_t)dg, rows * shape->HV * shape->K},
                                   {(size_t)dbeta, rows * shape->HV},
                                   {(size_t)dv, rows * shape->HV * shape->V}};
        for (const auto &z : zero)
            if (e == cudaSuccess) e = cudaMemsetAsync(reinterpret_cast<void *>(z[0]), 0, z[1] * 4, s);
        if (e != cudaSuccess) return cuda_fail(e, op);
    }
    if (ga.A_log && e == cudaSuccess) e = cudaMemsetAsync(dA_log, 0, (size_t)shape->HV * 4, s);
    if (ga.dt_bias && e == cudaSuccess)
        e = cudaMemsetAsync(ddt_bias, 0, (size_t)shape->HV * shape->K * 4, s);
    if (e != cudaSuccess) return cuda_fail(e, op);
    kda::RecurrentBwdArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.cu = cu_seqlens;
    a.dout = dout; a.dht = dht;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
    a.ckpt = static_cast<float *>(workspace);
    a.status = dev_status;
    a.B = shape->B; a.T = shape->T; a.H = shape->H; a.HV = shape->HV; a.K = shape->K;
    a.V = shape->V; a.N = shape->num_seqs;
    a.scale = resolve_scale(shape);
    a.g_scale = shape->g_scale;
    a.l2norm = (shape->flags & KDA_FLAG_QK_L2NORM) ? 1 : 0;
    a.act = ga;
    a.dA_log = dA_log;
    a.ddt_bias = ddt_bias;
    e = kda::launch_recurrent_bwd(a, shape->dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, op);
    g_last_error.clear();
    return KDA_OK;
}

size_t kda_chunk_workspace_size(const kda_shape *shape) {
    if (!shape || shape->K <= 0 || shape->V <= 0 || shape->HV <= 0 || shape->B <= 0 ||
        shape->T < 0 || shape->num_seqs < 0)
        return 0;
    const bool packed = shape->num_seqs != shape->B || shape->B == 1;
    return chunk_ws_layout(shape, packed).total;
}

size_t kda_workspace_size(const kda_shape *shape) { return kda_chunk_workspace_size(shape); }

kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                         const void *beta, const float *h0, const int32_t *cu_seqlens,
                         const kda_shape *shape, void *o, float *ht, void *workspace,
                         size_t workspace_bytes, int32_t *dev_status, kda_stream_t stream) {
    return kda_chunk_fwd_act(q, k, v, g, beta, h0, cu_seqlens, shape, nullptr, o, ht, workspace,
                             workspace_bytes, dev_status, stream);
}

kda_status kda_chunk_fwd_act(const void *q, const void *k, const void *v, const float *g,
                             const void *beta, const float *h0, const int32_t *cu_seqlens,
                             const kda_shape *shape, const kda_activation *act, void *o,
                             float *ht, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, kda_stream_t stream) {
    const char *op = "kda_chunk_fwd";
    kda_status st = check_common(op, shape, cu_seqlens);
    if (st != KDA_OK) return st;
    kda::GateAct ga;
    if ((st = resolve_act(op, shape, act, &ga)) != KDA_OK) return st;
    if ((st = check_fwd_pointers(op, shape, q, k, v, g, beta, o, cu_seqlens)) != KDA_OK) return st;
    if ((st = check_chunk_support(op, shape)) != KDA_OK) return st;
    const bool packed = cu_seqlens != nullptr;
    const ChunkWs L = chunk_ws_layout(shape, packed);
    if (L.slots > INT_MAX) return fail(KDA_ERR_UNSUPPORTED, "%s: too many chunks", op);
    const size_t need = kda_chunk_workspace_size(shape);
    if (!workspace || workspace_bytes < need)
        return fail(KDA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", op, need,
                    workspace_bytes);
    if ((uintptr_t)workspace % 256 != 0)
        return fail(KDA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", op);

    char *ws = static_cast<char *>(workspace);
    kda::ChunkArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.cu = cu_seqlens;
    a.o = o; a.ht = ht; a.status = dev_status;
    a.B = shape->B; a.T = shape->T; a.H = shape->H; a.HV = shape->HV; a.K = shape->K;
    a.V = shape->V; a.N = shape->num_seqs;
    a.scale = resolve_scale(shape);
    a.g_scale = shape->g_scale;
    a.l2norm = (shape->flags & KDA_FLAG_QK_L2NORM) ? 1 : 0;
    a.g_is_cumsum = (shape->flags & KDA_FLAG_G_IS_CUMSUM) ? 1 : 0;
    a.test_timeout = (shape->flags & KDA_FLAG_TEST_WAIT_TIMEOUT) ? 1 : 0;
    a.act = ga;
    a.ctrl = reinterpret_cast<kda::ChunkCtrl *>(ws + L.ctrl);
    a.chunk_start = reinterpret_cast<int32_t *>(ws + L.chunk_start);
    a.units = ws + L.units;
    a.slots = L.slots;
    a.split = L.split ? 1 : 0;
    a.qc = L.split ? ws + L.qc : nullptr;
    a.e0 = L.split ? reinterpret_cast<float *>(ws + L.e0) : nullptr;
    a.e1 = L.split ? reinterpret_cast<float *>(ws + L.e1) : nullptr;
    a.pm = L.split ? reinterpret_cast<float *>(ws + L.pm) : nullptr;
    a.e0b = L.split ? ws + L.e0b : nullptr;
    a.pipe = packed ? kda::PipePlan{} : L.pipe;
    a.prep_c0 = a.prep_c1 = 0;
    a.scan_c0 = a.scan_c1 = 0;
    if (a.pipe.parts > 0) a.e0 = reinterpret_cast<float *>(ws + L.e0);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (packed) {
        e = kda::launch_validate_offsets(cu_seqlens, a.N, a.T, dev_status, a.ctrl, a.chunk_start, s);
        if (e != cudaSuccess) return cuda_fail(e, op);
    }
    if (use_tc(shape)) {
        const void *ptrs[] = {q, k, v, g, h0, ht, o};
        for (const void *ptr : ptrs)
            if ((uintptr_t)ptr % 16 != 0)
                return fail(KDA_ERR_INVALID_ARG, "%s: bf16 tensors, g, h0 and ht must be 16-byte "
                            "aligned", op);
        e = kda::launch_chunk_tc(a, s);
    } else {
        e = kda::launch_chunk_simt(a, shape->dtype, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, op);
    g_last_error.clear();
    return KDA_OK;
}

size_t kda_chunk_bwd_workspace_size(const kda_shape *shape) {
    if (!shape || shape->K <= 0 || shape->V <= 0 || shape->HV <= 0 || shape->B <= 0 ||
        shape->T < 0 || shape->num_seqs < 0)
        return 0;
    // sized for packed input when the shape may be packed: it covers a dense call too
    const bool packed = shape->num_seqs != shape->B || shape->B == 1;
    return chunk_bwd_ws_layout(shape, packed).total;
}

kda_status kda_chunk_bwd(const void *q, const void *k, const void *v, const float *g,
                         const void *beta, const float *h0, const int32_t *cu_seqlens,
                         const kda_shape *shape, const void *dout, const float *dht, float *dq,
                         float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                         void *workspace, size_t workspace_bytes, int32_t *dev_status,
                         kda_stream_t stream) {
    return kda_chunk_bwd_act(q, k, v, g, beta, h0, cu_seqlens, shape, nullptr, dout, dht, dq, dk,
                             dv, dg, dbeta, dh0, nullptr, nullptr, workspace, workspace_bytes,
                             dev_status, stream);
}

namespace {

// The checks and the forward's ChunkArgs (with the backward's stores) shared by
// kda_chunk_fwd_save and kda_chunk_bwd_act.
kda_status chunk_bwd_setup(const char *op, const void *q, const void *k, const void *v,
                           const float *g, const void *beta, const float *h0,
                           const int32_t *cu_seqlens, const kda_shape *shape,
                           const kda_activation *act, uint32_t flags_ok, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, kda::GateAct *ga,
                           ChunkBwdWs *W, kda::ChunkArgs *a) {
    kda_status st = check_common(op, shape, cu_seqlens);
    if (st != KDA_OK) return st;
    if ((st = resolve_act(op, shape, act, ga)) != KDA_OK) return st;
    if (shape->dtype != KDA_DTYPE_BF16 || !kda::chunk_bwd_tc_supported(shape->K, shape->V))
        return fail(KDA_ERR_UNSUPPORTED, "%s: bf16 inputs with K = V = 128 only (got dtype %d, "
                    "K=%d, V=%d); kda_recurrent_bwd takes the rest", op, (int)shape->dtype,
                    shape->K, shape->V);
    if (shape->flags & ~flags_ok)
        return fail(KDA_ERR_UNSUPPORTED, "%s: flags 0x%x (taken: 0x%x; a cumsummed gate goes "
                    "through kda_recurrent_bwd)", op, shape->flags, flags_ok);
    const bool has_rows = (int64_t)shape->B * shape->T > 0;
    if (has_rows && (!q || !k || !v || !g || !beta))
        return fail(KDA_ERR_INVALID_ARG, "%s: q, k, v, g and beta must be non-NULL", op);
    const bool packed = cu_seqlens != nullptr;
    *W = chunk_bwd_ws_layout(shape, packed);
    if (W->f.slots > INT_MAX) return fail(KDA_ERR_UNSUPPORTED, "%s: too many chunks", op);
    const size_t need = kda_chunk_bwd_workspace_size(shape);
    if (!workspace || workspace_bytes < need)
        return fail(KDA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", op, need,
                    workspace_bytes);
    if ((uintptr_t)workspace % 256 != 0)
        return fail(KDA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", op);
    const void *ptrs[] = {q, k, v, g, h0};
    for (const void *ptr : ptrs)
        if ((uintptr_t)ptr % 16 != 0)
            return fail(KDA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", op);

    char *ws = static_cast<char *>(workspace);
    a->q = q; a->k = k; a->v = v; a->g = g; a->beta = beta; a->h0 = h0; a->cu = cu_seqlens;
    a->o = nullptr; a->ht = nullptr; a->status = dev_status;
    a->B = shape->B; a->T = shape->T; a->H = shape->H; a->HV = shape->HV; a->K = shape->K;
    a->V = shape->V; a->N = shape->num_seqs;
    a->scale = resolve_scale(shape);
    a->g_scale = shape->g_scale;
    a->l2norm = (shape->flags & KDA_FLAG_QK_L2NORM) ? 1 : 0;
    a->g_is_cumsum = 0;
    a->test_timeout = 0;
    a->act = *ga;
    a->ctrl = reinterpret_cast<kda::ChunkCtrl *>(ws + W->f.ctrl);
    a->chunk_start = reinterpret_cast<int32_t *>(ws + W->f.chunk_start);
    a->units = ws + W->f.units;
    a->slots = W->f.slots;
    a->split = 0;
    a->qc = nullptr; a->e1 = nullptr; a->pm = nullptr; a->e0b = nullptr;
    a->pipe = (packed || (shape->flags & KDA_FLAG_SERIAL)) ? kda::PipePlan{} : W->f.pipe;
    a->e0 = a->pipe.parts > 0 ? reinterpret_cast<float *>(ws + W->f.e0) : nullptr;
    a->prep_c0 = a->prep_c1 = 0;
    a->scan_c0 = a->scan_c1 = 0;
    a->bwd = 1;
    a->ck_h = ws + W->ck_h;
    a->ck_vp = ws + W->ck_vp;
    return KDA_OK;
}

}  // namespace

kda_status kda_chunk_fwd_save(const void *q, const void *k, const void *v, const float *g,
                              const void *beta, const float *h0, const int32_t *cu_seqlens,
                              const kda_shape *shape, const kda_activation *act, void *o,
                              float *ht, void *workspace, size_t workspace_bytes,
                              int32_t *dev_status, kda_stream_t stream) {
    const char *op = "kda_chunk_fwd_save";
    kda::GateAct ga;
    ChunkBwdWs W;
    kda::ChunkArgs a;
    kda_status st = chunk_bwd_setup(op, q, k, v, g, beta, h0, cu_seqlens, shape, act,
                                    KDA_FLAG_SERIAL | KDA_FLAG_QK_L2NORM, workspace,
                                    workspace_bytes, dev_status, &ga, &W, &a);
    if (st != KDA_OK) return st;
    if ((st = check_fwd_pointers(op, shape, q, k, v, g, beta, o, cu_seqlens)) != KDA_OK) return st;
    if ((uintptr_t)o % 16 != 0 || (uintptr_t)ht % 16 != 0)
        return fail(KDA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", op);
    char *ws = static_cast<char *>(workspace);
    float *hend = reinterpret_cast<float *>(ws + W.hend);
    a.o = o;
    a.ht = hend;  // every sequence's final state, for the backward (and copied to ht)
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (cu_seqlens) {
        e = kda::launch_validate_offsets(cu_seqlens, a.N, a.T, dev_status, a.ctrl, a.chunk_start, s);
        if (e != cudaSuccess) return cuda_fail(e, op);
    }
    if ((e = kda::launch_chunk_tc(a, s)) != cudaSuccess) return cuda_fail(e, op);
    if (ht && (e = cudaMemcpyAsync(ht, hend, (size_t)shape->num_seqs * shape->HV * shape->K *
                                                 shape->V * sizeof(float),
                                   cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return cuda_fail(e, op);
    g_last_error.clear();
    return KDA_OK;
}

kda_status kda_chunk_bwd_act(const void *q, const void *k, const void *v, const float *g,
                             const void *beta, const float *h0, const int32_t *cu_seqlens,
                             const kda_shape *shape, const kda_activation *act, const void *dout,
                             const float *dht, float *dq, float *dk, float *dv, float *dg,
                             float *dbeta, float *dh0, float *dA_log, float *ddt_bias,
                             void *workspace, size_t workspace_bytes, int32_t *dev_status,
                             kda_stream_t stream) {
    const char *op = "kda_chunk_bwd";
    kda::GateAct ga;
    ChunkBwdWs W;
    kda::ChunkArgs a;
    kda_status st = chunk_bwd_setup(op, q, k, v, g, beta, h0, cu_seqlens, shape, act,
                                    KDA_FLAG_SERIAL | KDA_FLAG_QK_L2NORM | KDA_FLAG_BWD_SAVED,
                                    workspace, workspace_bytes, dev_status, &ga, &W, &a);
    if (st != KDA_OK) return st;
    if ((ga.A_log && !dA_log) || (ga.dt_bias && !ddt_bias))
        return fail(KDA_ERR_INVALID_ARG, "%s: dA_log (and ddt_bias with dt_bias) must be non-NULL "
                    "with the gate activation", op);
    const bool has_rows = (int64_t)shape->B * shape->T > 0;
    if (has_rows && (!dout || !dq || !dk || !dv || !dg || !dbeta))
        return fail(KDA_ERR_INVALID_ARG, "%s: dout and dq, dk, dv, dg, dbeta must be non-NULL", op);
    const void *ptrs[] = {dout, dht, dq, dk, dv, dg, dh0};
    for (const void *ptr : ptrs)
        if ((uintptr_t)ptr % 16 != 0)
            return fail(KDA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", op);
    const bool packed = cu_seqlens != nullptr;
    char *ws = static_cast<char *>(workspace);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (packed) {
        e = kda::launch_validate_offsets(cu_seqlens, a.N, a.T, dev_status, a.ctrl, a.chunk_start, s);
        if (e != cudaSuccess) return cuda_fail(e, op);
    }
    // dq, dk accumulate over the value heads that share a q/k head (else each chunk
    // stores its rows once); with packed sequences rows outside every sequence stay zero
    const size_t rows = (size_t)shape->B * shape->T;
    const bool qk_zero = packed || shape->HV != shape->H;
    const size_t zero[][2] = {{(size_t)dq, qk_zero ? rows * shape->H * shape->K * 4 : 0},
                              {(size_t)dk, qk_zero ? rows * shape->H * shape->K * 4 : 0},
                              {(size_t)dv, packed ? rows * shape->HV * shape->V * 4 : 0},
                              {(size_t)dg, packed ? rows * shape->HV * shape->K * 4 : 0},
                              {(size_t)dbeta, packed ? rows * shape->HV * 4 : 0}};
    for (const auto &z : zero)
        if (z[1] && (e = cudaMemsetAsync(reinterpret_cast<void *>(z[0]), 0, z[1], s)) != cudaSuccess)
            return cuda_fail(e, op);
    if (ga.A_log && (e = cudaMemsetAsync(dA_log, 0, (size_t)shape->HV * 4, s)) != cudaSuccess)
        return cuda_fail(e, op);
    if (ga.dt_bias &&
        (e = cudaMemsetAsync(ddt_bias, 0, (size_t)shape->HV * shape->K * 4, s)) != cudaSuccess)
        return cuda_fail(e, op);
    e = kda::launch_chunk_bwd_tc(a, dout, dht, dq, dk, dv, dg, dbeta, dh0, ws + W.dhn, ws + W.dvp,
                                 reinterpret_cast<float *>(ws + W.hend),
                                 reinterpret_cast<float *>(ws + W.dgs),
                                 reinterpret_cast<float *>(ws + W.dhm),
                                 (shape->flags & KDA_FLAG_SERIAL) != 0,
                                 (shape->flags & KDA_FLAG_BWD_SAVED) == 0, s);
    if (e != cudaSuccess) return cuda_fail(e, op);
    if (a.l2norm || ga.A_log || ga.beta_scale > 0.f) {
        // the kernels formed the gradients of the normalised rows and of the activated
        // gate and beta: the options' chain rules, as in kda_recurrent_bwd
        kda::RecurrentBwdArgs r{};
        r.q = q; r.k = k; r.v = v; r.g = g; r.beta = beta; r.h0 = h0; r.cu = cu_seqlens;
        r.dq = dq; r.dk = dk; r.dv = dv; r.dg = dg; r.dbeta = dbeta; r.dh0 = dh0;
        r.status = dev_status;
        r.B = shape->B; r.T = shape->T; r.H = shape->H; r.HV = shape->HV; r.K = shape->K;
        r.V = shape->V; r.N = shape->num_seqs;
        r.scale = a.scale;
        r.g_scale = a.g_scale;
        r.l2norm = a.l2norm;
        r.act = ga;
        r.dA_log = dA_log;
        r.ddt_bias = ddt_bias;
        if ((e = kda::launch_bwd_chain(r, KDA_DTYPE_BF16, s)) != cudaSuccess) return cuda_fail(e, op);
    }
    g_last_error.clear();
    return KDA_OK;
}

kda_status kda_read_device_status(const int32_t *dev_status, int32_t *host_bits,
                                  kda_stream_t stream) {
    if (!dev_status) return fail(KDA_ERR_INVALID_ARG, "kda_read_device_status: NULL status word");
    int32_t bits = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&bits, dev_status, sizeof(bits), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "kda_read_device_status");
    if (host_bits) *host_bits = bits;
    if (bits & KDA_DEVICE_BAD_CU_SEQLENS)
        return fail(KDA_ERR_BAD_CU_SEQLENS, "device reported invalid cu_seqlens");
    if (bits & KDA_DEVICE_TIMEOUT)
        return fail(KDA_ERR_TIMEOUT, "a bounded device-side wait timed out");
    if (bits & KDA_DEVICE_GATE_RANGE)
        return fail(KDA_ERR_UNSUPPORTED, "kda_chunk_bwd: a chunk's gate range exceeds what the "
                    "chunked backward takes (its gradients were not computed)");
    if (bits & KDA_DEVICE_INTERNAL)
        return fail(KDA_ERR_CUDA, "a kernel found an internal launch invariant broken");
    return KDA_OK;
}

kda_status kda_clear_device_status(int32_t *dev_status, kda_stream_t stream) {
    if (!dev_status) return fail(KDA_ERR_INVALID_ARG, "kda_clear_device_status: NULL status word");
    cudaError_t e = cudaMemsetAsync(dev_status, 0, sizeof(int32_t),
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_clear_device_status");
    return KDA_OK;
}

}  // extern "C"

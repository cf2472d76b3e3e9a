// kda_noalloc.cu -- kda_chunk_fwd_noalloc: the chunked forward for callers that
// cannot allocate device memory when they call it.
//
// Some callers are not allowed to allocate: runtimes that plan a fixed device
// memory budget up front and own every byte of it, plugin hosts that forbid
// allocations outside their own pool, and latency-critical loops where the
// implicit device synchronisation of cudaMalloc is not acceptable.  For them
// this entry point takes the same inputs and outputs as kda_chunk_fwd but
// brings its own scratch: a file-scope device array of fixed size, reserved in
// every GPU's memory that loads this library until the process exits.
//
// Its launches all run on the caller's stream (KDA_FLAG_SERIAL), so no stream or
// event is created either.
//
// The host cannot pass the array's name to a kernel (in host code it only
// names a host-side stand-in), so the array's device address is looked up with
// cudaGetSymbolAddress once per device, on that device's first call.  The
// computation itself is kda_chunk_fwd, unchanged, given that address as its
// workspace.
//
// With lazy module loading (the CUDA default since 12.2) this translation
// unit's device code, and with it the array, is loaded onto a device only when
// it is first used there: that first lookup is when the 32 MiB are reserved,
// and it can fail for lack of device memory or wait on the device.  So the
// first call on each device belongs in the caller's set-up, before any stream
// capture and before the caller's memory budget is fixed.
#include <cstdio>
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
void set_last_error(const char *msg);
}

namespace {

constexpr size_t kScratchBytes = (size_t)KDA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The shared scratch.  Nothing in it has to start at zero: every call writes
// each byte it later reads (the offsets pre-pass rewrites its control block,
// the prep kernel writes every operand tile before the scan reads it).
static __device__ __align__(256) unsigned char g_scratch[KDA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

kda_status set_fail(kda_status st, const char *msg) {
    kda::set_last_error(msg);
    return st;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                           const float *g, const void *beta, const float *h0,
                                           const int32_t *cu_seqlens, const kda_shape *shape,
                                           void *o, float *ht, int32_t *dev_status,
                                           kda_stream_t stream) {
    if (!shape) return set_fail(KDA_ERR_INVALID_ARG, "kda_chunk_fwd_noalloc: shape is NULL");
    // Every launch on the caller's stream: a pipelined call would create the
    // library's scan stream and events on first use.
    kda_shape serial = *shape;
    serial.flags |= KDA_FLAG_SERIAL;
    shape = &serial;
    const size_t need = kda_chunk_workspace_size(shape);
    if (need == 0) return set_fail(KDA_ERR_INVALID_ARG, "kda_chunk_fwd_noalloc: invalid shape");
    if (need > kScratchBytes) {
        char buf[256];
        snprintf(buf, sizeof(buf),
                 "kda_chunk_fwd_noalloc: this shape needs %zu bytes of scratch; the built-in "
                 "buffer holds %zu (use kda_chunk_fwd with a caller workspace)",
                 need, kScratchBytes);
        return set_fail(KDA_ERR_UNSUPPORTED, buf);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return set_fail(KDA_ERR_CUDA, "kda_chunk_fwd_noalloc: no usable current device");
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_addr[dev]) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_scratch);
            if (e != cudaSuccess || ptr == nullptr) {
                char buf[320];
                if (e == cudaErrorMemoryAllocation)
                    snprintf(buf, sizeof(buf),
                             "kda_chunk_fwd_noalloc: the device has no room for the library's "
                             "%zu-byte scratch array (reserved when this device's first call "
                             "loads it; make that call during set-up)",
                             kScratchBytes);
                else
                    snprintf(buf, sizeof(buf),
                             "kda_chunk_fwd_noalloc: cudaGetSymbolAddress failed: %s",
                             cudaGetErrorString(e));
                return set_fail(KDA_ERR_CUDA, buf);
            }
            g_addr[dev] = ptr;
        }
        scratch = g_addr[dev];
    }
    return kda_chunk_fwd(q, k, v, g, beta, h0, cu_seqlens, shape, o, ht, scratch, kScratchBytes,
                         dev_status, stream);
}

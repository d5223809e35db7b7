// prefill_noalloc.cu -- gdn_prefill_noalloc: gdn_prefill with its scratch in a
// statically sized device array, for callers that cannot allocate device memory.
//
// The tensor-core prefill keeps one record per (chunk, value head) in scratch
// between its chunk-prep and state-scan kernels.  gdn_prefill takes that scratch
// from the caller; this entry point takes it from `g_prefill_scratch` below, so
// that nothing is allocated on any call.  The array is a module global of the
// library, created when this translation unit's module is loaded on a device and
// shared by every call on that device.
#include <stdio.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

// Scratch of the tensor-core prefill for calls through gdn_prefill_noalloc.
static __device__ __align__(256) unsigned char g_prefill_scratch[GDN_PREFILL_NOALLOC_SCRATCH_BYTES];

// Device address of g_prefill_scratch in the current device's context.  It is looked up
// on every call (a cheap runtime query), so that a context torn down and created again
// (cudaDeviceReset) never leaves a stale address behind.
gdn_status scratch_address(void **out) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress((void **)&ptr, g_prefill_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
        char msg[256];
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(prefill scratch): %s",
                 cudaGetErrorString(e));
        return report_error(GDN_ERR_CUDA, msg);
    }
    *out = ptr;
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_prefill_noalloc(const gdn_shape *shape, const void *q, const void *k,
                                          const void *v, const void *a, const void *b,
                                          const float *A_log, const float *dt_bias,
                                          const float *state_in, const int32_t *cu_seqlens,
                                          float scale, void *o, float *state_out, void *stream) {
    if (shape == nullptr) return gdn::report_error(GDN_ERR_INVALID_ARG, "shape is NULL");
    // Every scratch byte the kernels read is written earlier in the same call, so
    // nothing left by a previous call needs clearing.  The call runs the records-only
    // path (no time-parallel buffers, no internal stream), so the records are the need.
    const size_t need = gdn::prefill_records_bytes_for(shape, cu_seqlens != nullptr);
    if (need > (size_t)GDN_PREFILL_NOALLOC_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "gdn_prefill_noalloc: this shape needs %zu bytes of scratch, above the fixed %zu "
                 "(use gdn_prefill with a caller-provided workspace)",
                 need, (size_t)GDN_PREFILL_NOALLOC_SCRATCH_BYTES);
        return gdn::report_error(GDN_ERR_INVALID_ARG, msg);
    }
    void *scratch = nullptr;
    gdn_status st = gdn::scratch_address(&scratch);
    if (st != GDN_OK) return st;
    // No segment overlap: it would create an internal stream on first use.
    return gdn::prefill_impl(shape, q, k, v, a, b, A_log, dt_bias, state_in, cu_seqlens, scale, o,
                             state_out, scratch, (size_t)GDN_PREFILL_NOALLOC_SCRATCH_BYTES, false,
                             stream);
}

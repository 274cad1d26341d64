// static_ws.cu -- all-gather + GEMM for callers that cannot allocate device
// memory.
//
// Some callers cannot hand this library a workspace: a plugin behind an
// operator interface with no scratch argument, or code that must not call the
// device allocator while it runs (a caller whose allocator owns all device
// memory, or a latency-critical path that forbids allocation).  For them,
// kosmos_ag_gemm_noalloc keeps the ticket counters, readiness flags and
// status word in the file-scope array below instead of a caller workspace.
//
// The array is a __device__ symbol: in host code its name is only a host-side
// stand-in, never a device address.  Every call looks the device address up
// with cudaGetSymbolAddress (with the caller's device current) and passes it to
// the kernel like any workspace pointer.  The lookup is not cached: after a
// cudaDeviceReset, or in a new primary context, the module is loaded again and
// the array may live at another address.
#include <cuda_runtime.h>

#include "../../include/kosmos.h"

namespace {

// Held by every GPU that loads this library until the process exits.
__device__ __align__(256) unsigned char g_kosmos_static_ws[KOSMOS_STATIC_WS_BYTES];

// Device address of g_kosmos_static_ws in the current device's context.  The
// first lookup in a context loads the module (lazy loading), which is why the
// first call on a device should come before any stream capture.
kosmos_status static_ws_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_kosmos_static_ws);
    if (e != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return KOSMOS_ERR_CUDA;
    }
    *out = p;
    return KOSMOS_OK;
}

}  // namespace

extern "C" KOSMOS_API kosmos_status kosmos_ag_gemm_noalloc(const void *const *x_shards, const void *const *x_scales,
                                                           int P, int64_t m_per_shard, int64_t k, int64_t n,
                                                           const void *w, const void *w_scales, int dtype,
                                                           void *x_gathered, void *y, const kosmos_opts *opts,
                                                           void *stream) {
    kosmos_opts o;
    kosmos_default_opts(&o);
    if (opts) o = *opts;
    if (o.trace) return KOSMOS_ERR_UNSUPPORTED;  // the trace ring does not fit the static scratch
    o.tail_split = 0;                            // nor do the K-split partials
    const size_t need = kosmos_workspace_bytes(KOSMOS_OP_AG_GEMM, P, m_per_shard, n, k, dtype, &o);
    if (need == 0) return KOSMOS_ERR_INVALID_ARG;
    if (need > static_cast<size_t>(KOSMOS_STATIC_WS_BYTES)) return KOSMOS_ERR_WORKSPACE;
    void *ws = nullptr;
    const kosmos_status s = static_ws_address(&ws);
    if (s != KOSMOS_OK) return s;
    // The array keeps the previous call's counters, flags and status: clear the
    // part this call uses so it starts from zero.
    if (cudaMemsetAsync(ws, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return KOSMOS_ERR_CUDA;
    }
    return kosmos_ag_gemm(x_shards, x_scales, P, m_per_shard, k, n, w, w_scales, dtype, x_gathered, y, ws,
                          static_cast<size_t>(KOSMOS_STATIC_WS_BYTES), &o, stream);
}

extern "C" KOSMOS_API kosmos_status kosmos_noalloc_status_sync(void *stream, int64_t *failing_entry) {
    void *ws = nullptr;
    const kosmos_status s = static_ws_address(&ws);
    if (s != KOSMOS_OK) return s;
    return kosmos_status_sync(ws, stream, failing_entry);
}

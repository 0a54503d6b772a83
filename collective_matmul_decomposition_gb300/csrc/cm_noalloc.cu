// cm_noalloc.cu -- cm_ag_gemm for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and have no
// way to obtain more device memory: a plugin run by a host framework that
// owns every device allocation, or a latency-critical loop where cudaMalloc
// (which may synchronise the device) is not acceptable.  This entry point
// needs no workspace argument: the AllGather->GEMM scratch (status word,
// per-chunk flags, tile counters and the ring receive slots) lives in one
// file-scope device array of fixed size, CM_NOALLOC_SCRATCH_BYTES.  Every GPU
// that loads this library holds that array until the process exits.
//
// Properties the caller must know:
//  - The first call on a device looks up the array's device address (with
//    that device current) and caches it; make that first call outside any
//    stream capture.
//  - All calls share the one array, and it keeps the last call's contents.
//    The status word, flags and counters are cleared on the stream at the
//    start of every call; the receive slots need no clearing.  Two calls that
//    can overlap on the GPU (different streams, no ordering) race on it.
//  - A problem whose scratch exceeds the array is rejected with
//    CM_ERR_WORKSPACE before any device work.
//  - The array's status word records a device-side wait that timed out in
//    the last call; cm_ag_gemm_noalloc_check_status reads it (with the same
//    device current), as cm_check_status does for a caller's workspace.
//  - Nothing here calls cudaMalloc, cudaFree or an allocating library routine.
#include <cuda_runtime.h>

#include <mutex>

#include "cm.h"

namespace {

static __device__ __align__(256) unsigned char g_cm_noalloc_scratch[CM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
cm_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_cm_noalloc_scratch) != cudaSuccess || !p) return CM_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return CM_OK;
}

}  // namespace

extern "C" cm_status cm_ag_gemm_noalloc(cm_plan_t plan, const void *x, const void *w, cm_wlayout wlayout, void *y,
                                        cm_dtype y_dtype, int64_t m, int64_t K, int64_t n, cm_stream_t stream) {
    if (!plan) return CM_ERR_INVALID_ARG;
    const size_t need = cm_ag_gemm_workspace_size(plan, m, K);
    if (need == 0) return CM_ERR_SHAPE;
    if (need > size_t(CM_NOALLOC_SCRATCH_BYTES)) return CM_ERR_WORKSPACE;
    void *ws = nullptr;
    const cm_status st = scratch_address(&ws);
    if (st != CM_OK) return st;
    return cm_ag_gemm(plan, x, w, wlayout, y, y_dtype, m, K, n, ws, need, stream);
}

extern "C" cm_status cm_ag_gemm_noalloc_check_status(cm_stream_t stream, int32_t info[4]) {
    void *ws = nullptr;
    const cm_status st = scratch_address(&ws);
    if (st != CM_OK) return st;
    return cm_check_status(ws, stream, info);
}

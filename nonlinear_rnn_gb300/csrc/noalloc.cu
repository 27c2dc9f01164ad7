// Newton forward for callers that cannot allocate device memory.
//
// nrnn_newton_forward takes its look-back scratch from a caller-provided
// workspace.  Some callers have no way to obtain one: a plugin running inside
// a host framework that owns every device allocation and exposes no pool to
// it, or a latency-bounded loop that must not call cudaMalloc/cudaFree (which
// can synchronise the whole device) once it is running.  This entry point
// needs no workspace: its scratch is one file-scope device array of
// NRNN_NOALLOC_SCRATCH_BYTES that every GPU using the library holds until the
// process exits.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/nrnn.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[NRNN_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 128;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[MAX_DEVICES];   // device address of the array, per device

// Device address of the scratch array on the current device.  The host-side
// name of a __device__ array is not a device address, so it is looked up once
// per device (with that device current) and cached.
int noalloc_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return NRNN_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return NRNN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return NRNN_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return NRNN_OK;
}

}  // namespace

extern "C" int nrnn_newton_forward_noalloc(const void *preact, int dtype, const float *params,
                                           int64_t B, int64_t T, int64_t d_h,
                                           const int32_t *cu_seqlens, int64_t num_segments,
                                           int K, float residual_fail, void *H_out,
                                           float *residual_dev, float *residual_host,
                                           void *stream) {
    const size_t need = nrnn_newton_workspace_bytes(B, T, d_h, dtype, K, NRNN_ALGO_FUSED);
    if (need == 0) return NRNN_ERR_INVALID_ARG;
    if (need > NRNN_NOALLOC_SCRATCH_BYTES) return NRNN_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != NRNN_OK) return st;
    return nrnn_newton_forward(preact, dtype, params, B, T, d_h, cu_seqlens, num_segments, K,
                               residual_fail, NRNN_ALGO_FUSED, H_out, residual_dev,
                               residual_host, scratch, NRNN_NOALLOC_SCRATCH_BYTES, stream);
}

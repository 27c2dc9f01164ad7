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

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/nrnn.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[NRNN_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 128;

// Device address of the array per device, tagged with the unique id of the
// context it was looked up in (cuCtxGetId ids are never reused within a
// process): after cudaDeviceReset the primary context is created anew, the
// module is loaded again, and the id no longer matches, so the address is
// looked up again instead of pointing at memory the library no longer owns.
struct ScratchAddr {
    unsigned long long ctx_id;
    void *ptr;
};
std::mutex g_noalloc_mu;
ScratchAddr g_noalloc_addr[MAX_DEVICES];

using PfnCtxGetCurrent = CUresult (*)(CUcontext *);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long *);

// unique id of the calling thread's current context, 0 if there is none
unsigned long long current_ctx_id() {
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PfnCtxGetCurrent>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PfnCtxGetId>(p);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array on the current device.  The host-side
// name of a __device__ array is not a device address, so it is looked up with
// the device current (cudaGetSymbolAddress, which also creates the device's
// context if the caller has not yet) and kept for later calls in that context.
int noalloc_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return NRNN_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return NRNN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    const unsigned long long id = current_ctx_id();
    if (id == 0 || g_noalloc_addr[dev].ctx_id != id || g_noalloc_addr[dev].ptr == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return NRNN_ERR_CUDA;
        g_noalloc_addr[dev].ctx_id = current_ctx_id();
        g_noalloc_addr[dev].ptr = p;
    }
    *out = g_noalloc_addr[dev].ptr;
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

// Segment-aligned chunks of a cu_seqlens pack for the Newton kernels.
//
// The segments of a pack are independent sequences (pararnn-torch
// shapes_layout, "cu_seqlens": the recurrence restarts at every segment
// head).  Cutting the pack's time axis into 64-step chunks chains every chunk
// to the one before it across segment boundaries, so a pack of a few long
// segments behaves like one very long row: few look-back chains, each with
// many chunks in flight at once, and every chunk waits for a predecessor that
// started just before it.  Cutting each segment into its own chunks instead
// gives one chain per segment; handing the chunks out level by level (chunk j
// of every segment before chunk j + 1 of any) spreads the chunks in flight
// over all segments, so that a chunk's predecessor has usually finished the
// iteration it waits for.  The last chunk of a segment may be short.  The
// backward scan runs each chain from the segment's end: its plan orders the
// chunks by how many chunks of the segment follow them.
#include "pack_plan.cuh"

namespace nrnn {

namespace {

constexpr int PT = 1024;   // threads of the stand-alone plan kernel

__global__ void __launch_bounds__(PT) k_pack_plan(const int32_t *__restrict__ cu, int S, int n_chunks,
                                                  bool reverse, int4 *__restrict__ plan) {
    extern __shared__ int sm[];
    build_pack_plan<PT>(cu, S, n_chunks, reverse, plan, sm);
}

}  // namespace

bool pack_plan_applies(int64_t B, int64_t T, int64_t S) {
    const int64_t n_chunks = (T + NEWTON_L - 1) / NEWTON_L;
    return B == 1 && S >= 2 && S <= PACK_PLAN_MAX_S && n_chunks <= PACK_PLAN_MAX_CHUNKS &&
           8 * S <= n_chunks;
}

size_t pack_plan_bytes(int64_t T, int64_t S) {
    const int64_t n_chunks = (T + NEWTON_L - 1) / NEWTON_L;
    return sizeof(int4) * static_cast<size_t>(1 + n_chunks + S);
}

cudaError_t launch_pack_plan(const int32_t *cu, int S, int n_chunks, int4 *plan, bool reverse,
                             cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = once_per_device(configured, [](int) {
        return cudaFuncSetAttribute(k_pack_plan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(pack_plan_smem(PACK_PLAN_MAX_S, PACK_PLAN_MAX_CHUNKS)));
    });
    if (e != cudaSuccess) return e;
    k_pack_plan<<<1, PT, pack_plan_smem(S, n_chunks), stream>>>(cu, S, n_chunks, reverse, plan);
    return cudaGetLastError();
}

}  // namespace nrnn

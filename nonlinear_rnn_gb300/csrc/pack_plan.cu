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
#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

namespace {

constexpr int PT = 1024;   // threads of the plan kernel

// Exclusive prefix sums of in[0, n) into out[0, n) by the whole CTA (in and
// out may be the same array); returns the total.  Each thread sums a
// contiguous range, the ranges' sums are scanned across the CTA, and each
// thread then writes its range.
__device__ int cta_exclusive_scan(const int *in, int *out, int n, int *s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + PT - 1) / PT;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += in[i];
    int x = sum;   // inclusive scan of the range sums within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL_MASK, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL_MASK, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    int run = x - sum + (warp > 0 ? s_warp[warp - 1] : 0);
    const int total = s_warp[PT / 32 - 1];
    for (int i = lo; i < hi; ++i) {
        const int v = in[i];
        out[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

// One CTA.  Shared memory: three arrays over chunk counts 0..n_chunks and
// three over the segments.
__global__ void __launch_bounds__(PT) k_pack_plan(const int32_t *__restrict__ cu, int S, int n_chunks,
                                                  bool reverse, int4 *__restrict__ plan) {
    extern __shared__ int sm[];
    __shared__ int s_warp[PT / 32];
    const int M = n_chunks + 1;
    int *cnt = sm;           // [M] segments with exactly c chunks; later the next free rank per c
    int *more = cnt + M;     // [M] segments with more than c chunks (active at level c)
    int *first = more + M;   // [M] plan item of the first chunk of level j
    int *nc = first + M;     // [S] chunks of segment s
    int *base = nc + S;      // [S] chunks of the segments before s
    int *rank = base + S;    // [S] place of s among the segments, most chunks first
    const int tid = threadIdx.x;
    for (int i = tid; i < M; i += PT) cnt[i] = 0;
    __syncthreads();
    for (int s = tid; s < S; s += PT) {
        const int len = max(0, __ldg(cu + s + 1) - __ldg(cu + s));
        const int c = min(n_chunks, (len + NEWTON_L - 1) / NEWTON_L);
        nc[s] = c;
        atomicAdd(&cnt[c], 1);
    }
    __syncthreads();
    cta_exclusive_scan(cnt, more, M, s_warp);   // segments with fewer than c chunks
    for (int i = tid; i < M; i += PT) more[i] = S - more[i] - cnt[i];
    __syncthreads();
    const int total = cta_exclusive_scan(more, first, M, s_warp);
    cta_exclusive_scan(nc, base, S, s_warp);
    for (int i = tid; i < M; i += PT) cnt[i] = 0;
    __syncthreads();
    // segments with more chunks first; the order among equal lengths does not
    // matter (every chunk's predecessor sits one level earlier)
    for (int s = tid; s < S; s += PT) rank[s] = more[nc[s]] + atomicAdd(&cnt[nc[s]], 1);
    __syncthreads();
    for (int s = tid; s < S; s += PT) {
        const int c = nc[s], r0 = __ldg(cu + s), r1 = __ldg(cu + s + 1), b = base[s], rk = rank[s];
        for (int j = 0; j < c; ++j)   // level: j, or the chunks after j (reverse)
            plan[1 + first[reverse ? c - 1 - j : j] + rk] = make_int4(r0 + j * NEWTON_L, r1, j, b + j);
    }
    if (tid == 0) plan[0] = make_int4(total, 0, 0, 0);
}

size_t plan_smem(int S, int n_chunks) {
    return sizeof(int) * (3 * static_cast<size_t>(n_chunks + 1) + 3 * static_cast<size_t>(S));
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
                                    static_cast<int>(plan_smem(PACK_PLAN_MAX_S, PACK_PLAN_MAX_CHUNKS)));
    });
    if (e != cudaSuccess) return e;
    k_pack_plan<<<1, PT, plan_smem(S, n_chunks), stream>>>(cu, S, n_chunks, reverse, plan);
    return cudaGetLastError();
}

}  // namespace nrnn

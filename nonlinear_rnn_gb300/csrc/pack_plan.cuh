// Segment-aligned chunks of a cu_seqlens pack: the plan one CTA builds (see
// pack_plan.cu for why, nrnn_internal.h for the layout of the plan).
#pragma once

#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

// Shared memory the plan takes: three int arrays over chunk counts
// 0..n_chunks and three over the segments.
__host__ __device__ inline size_t pack_plan_smem(int S, int n_chunks) {
    return sizeof(int) * (3 * static_cast<size_t>(n_chunks + 1) + 3 * static_cast<size_t>(S));
}

// Exclusive prefix sums of in[0, n) into out[0, n) by the whole CTA of NT
// threads (in and out may be the same array); returns the total.  Each
// thread sums a contiguous range, the ranges' sums are scanned across the
// CTA, and each thread then writes its range.
template <int NT>
__device__ int cta_exclusive_scan(const int *in, int *out, int n, int *s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + NT - 1) / NT;
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
        int w = lane < NT / 32 ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL_MASK, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NT / 32) s_warp[lane] = w;
    }
    __syncthreads();
    int run = x - sum + (warp > 0 ? s_warp[warp - 1] : 0);
    const int total = s_warp[NT / 32 - 1];
    for (int i = lo; i < hi; ++i) {
        const int v = in[i];
        out[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

// The plan of a pack of S segments (cu: device, S + 1 bounds) over n_chunks
// 64-step chunks of its time axis, built by one CTA of NT threads (all of
// them call this) in sm[0 .. pack_plan_smem(S, n_chunks)).  Chunks are
// ordered by level -- j, or with reverse the number of chunks of the segment
// after j -- and within one level by the segment's number of chunks, most
// first; the order among segments of equal chunk counts does not matter
// (every chunk's predecessor in its chain sits one level earlier).
template <int NT>
__device__ void build_pack_plan(const int32_t *__restrict__ cu, int S, int n_chunks, bool reverse,
                                int4 *__restrict__ plan, int *sm) {
    __shared__ int s_warp[32];
    const int M = n_chunks + 1;
    int *cnt = sm;           // [M] segments with exactly c chunks; later the next free rank per c
    int *more = cnt + M;     // [M] segments with more than c chunks (active at level c)
    int *first = more + M;   // [M] plan item of the first chunk of level j
    int *nc = first + M;     // [S] chunks of segment s
    int *base = nc + S;      // [S] chunks of the segments before s
    int *rank = base + S;    // [S] place of s among the segments, most chunks first
    const int tid = threadIdx.x;
    for (int i = tid; i < M; i += NT) cnt[i] = 0;
    __syncthreads();
    for (int s = tid; s < S; s += NT) {
        const int len = max(0, __ldg(cu + s + 1) - __ldg(cu + s));
        const int c = min(n_chunks, (len + NEWTON_L - 1) / NEWTON_L);
        nc[s] = c;
        atomicAdd(&cnt[c], 1);
    }
    __syncthreads();
    cta_exclusive_scan<NT>(cnt, more, M, s_warp);   // segments with fewer than c chunks
    for (int i = tid; i < M; i += NT) more[i] = S - more[i] - cnt[i];
    __syncthreads();
    const int total = cta_exclusive_scan<NT>(more, first, M, s_warp);
    cta_exclusive_scan<NT>(nc, base, S, s_warp);
    for (int i = tid; i < M; i += NT) cnt[i] = 0;
    __syncthreads();
    for (int s = tid; s < S; s += NT) rank[s] = more[nc[s]] + atomicAdd(&cnt[nc[s]], 1);
    __syncthreads();
    for (int s = tid; s < S; s += NT) {
        const int c = nc[s], r0 = __ldg(cu + s), r1 = __ldg(cu + s + 1), b = base[s], rk = rank[s];
        for (int j = 0; j < c; ++j)
            plan[1 + first[reverse ? c - 1 - j : j] + rk] = make_int4(r0 + j * NEWTON_L, r1, j, b + j);
    }
    if (tid == 0) plan[0] = make_int4(total, 0, 0, 0);
}

}  // namespace nrnn

// Picard sweep (fixed-point iteration of the recurrence), the warm start the
// pararnn pages suggest ahead of Newton (FAQs "How many Newton iterations
// should I use?": "try Picard warm-start").  Memory-bound: P and G_in in, G_out
// out, no dependency between time steps within a sweep.
#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

namespace {

constexpr int NW = NEWTON_NW;
constexpr int SEG = NEWTON_SEG;
constexpr int L = NEWTON_L;
constexpr int U = TILE_U;

// One Picard sweep G_out_t = f(G_in_{t-1}, P_t) for every t (G_in == null: the
// zero trajectory; shifted state 0 at t = 0 and at segment heads); the cell in
// the storage type's formulation.  A streaming kernel: each thread takes two
// adjacent units (one 4-byte bf16 pair or 8-byte fp32 pair per load, so a
// warp touches whole 128-byte lines) and one scalar step at a time.
template <typename TS> struct PairOf;
template <> struct PairOf<float> {
    using type = float2;
    __device__ static float2 f32(float2 v) { return v; }
    __device__ static float2 from(float a, float b) { return make_float2(a, b); }
};
template <> struct PairOf<__nv_bfloat16> {
    using type = __nv_bfloat162;
    __device__ static float2 f32(__nv_bfloat162 v) { return __bfloat1622float2(v); }
    __device__ static __nv_bfloat162 from(float a, float b) { return __floats2bfloat162_rn(a, b); }
};

template <typename TS>
__global__ void __launch_bounds__(NW * 32)
    k_picard(const TS *__restrict__ P, const float *__restrict__ params,
             const TS *__restrict__ G_in, TS *__restrict__ G_out, int T, int d_h,
             const int32_t *cu, int S) {
    using PT = PairOf<TS>;
    using Pair = typename PT::type;
    __shared__ uint32_t s_heads[L / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int u = (blockIdx.x * U + lane) * 2, t0 = blockIdx.y * L, b = blockIdx.z;
    if (tid < L / 32) s_heads[tid] = 0u;
    __syncthreads();
    if (tid == 0) mark_heads(cu, S, t0, L, s_heads);
    __syncthreads();
    if (u >= d_h) return;   // d_h is even: both units of the pair exist
    const UnitParams p0 = load_unit_params(params, d_h, u, true);
    const UnitParams p1 = load_unit_params(params, d_h, u + 1, true);
    const int r0 = warp * SEG;
    const size_t row0 = static_cast<size_t>(b) * T;
    float2 hprev = make_float2(0.f, 0.f);
    if (G_in != nullptr && t0 + r0 > 0)
        hprev = PT::f32(*reinterpret_cast<const Pair *>(G_in + (row0 + t0 + r0 - 1) * d_h + u));
    // the rows are independent given G_in: each batch of PF rows is loaded
    // before any of it is computed, so that PF rows of loads are in flight
    constexpr int PF = 4;
    const int nrows = min(SEG, T - (t0 + r0));
    for (int i0 = 0; i0 < nrows; i0 += PF) {
        Pair lz[PF], lr[PF], lc[PF], lg[PF];
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            const int t = t0 + r0 + min(i0 + j, nrows - 1);   // in range; duplicates unused
            const TS *p = P + (row0 + t) * 3 * d_h + u;
            lz[j] = *reinterpret_cast<const Pair *>(p);
            lr[j] = *reinterpret_cast<const Pair *>(p + d_h);
            lc[j] = *reinterpret_cast<const Pair *>(p + 2 * d_h);
            if (G_in != nullptr) lg[j] = *reinterpret_cast<const Pair *>(G_in + (row0 + t) * d_h + u);
        }
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            const int r = r0 + i0 + j, t = t0 + r;
            if (i0 + j < nrows) {
                const float2 pz = PT::f32(lz[j]), pr = PT::f32(lr[j]), pc = PT::f32(lc[j]);
                const bool head = head_bit(s_heads, r);
                const float f0 = cell_f_storage<TS>(head ? 0.f : hprev.x, pz.x, pr.x, pc.x, p0);
                const float f1 = cell_f_storage<TS>(head ? 0.f : hprev.y, pz.y, pr.y, pc.y, p1);
                *reinterpret_cast<Pair *>(G_out + (row0 + t) * d_h + u) = PT::from(f0, f1);
                hprev = (G_in != nullptr) ? PT::f32(lg[j]) : make_float2(0.f, 0.f);
            }
        }
    }
}

}  // namespace

cudaError_t launch_picard(int dtype, const void *P, const float *params, const void *G_in,
                          void *G_out, int B, int T, int d_h, const int32_t *cu, int S,
                          cudaStream_t stream) {
    const dim3 grid((d_h + 2 * U - 1) / (2 * U), (T + L - 1) / L, B);   // 64 units per CTA
    if (dtype == 1)
        k_picard<__nv_bfloat16><<<grid, NW * 32, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(P), params, static_cast<const __nv_bfloat16 *>(G_in),
            static_cast<__nv_bfloat16 *>(G_out), T, d_h, cu, S);
    else
        k_picard<float><<<grid, NW * 32, 0, stream>>>(static_cast<const float *>(P), params,
                                                  static_cast<const float *>(G_in),
                                                  static_cast<float *>(G_out), T, d_h, cu, S);
    return cudaGetLastError();
}

}  // namespace nrnn

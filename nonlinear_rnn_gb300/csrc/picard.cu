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
// the storage type's formulation.  A streaming kernel: each thread takes the
// NU = 8 / sizeof(TS) adjacent units of one 8-byte load (2 fp32 or 4 bf16),
// so a warp touches whole 128-byte lines, and one step at a time.
template <typename TS> constexpr int picard_nu() { return 8 / static_cast<int>(sizeof(TS)); }

template <typename TS>
__device__ __forceinline__ void unpack8(uint2 w, float (&o)[picard_nu<TS>()]) {
    if constexpr (sizeof(TS) == 2) {
        o[0] = __uint_as_float(w.x << 16);
        o[1] = __uint_as_float(w.x & 0xffff0000u);
        o[2] = __uint_as_float(w.y << 16);
        o[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
        o[0] = __uint_as_float(w.x);
        o[1] = __uint_as_float(w.y);
    }
}

template <typename TS>
__device__ __forceinline__ uint2 pack8(const float (&v)[picard_nu<TS>()]) {
    if constexpr (sizeof(TS) == 2) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
        return make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
    } else {
        return make_uint2(__float_as_uint(v[0]), __float_as_uint(v[1]));
    }
}

template <typename TS>
__global__ void __launch_bounds__(NW * 32)
    k_picard(const TS *__restrict__ P, const float *__restrict__ params,
             const TS *__restrict__ G_in, TS *__restrict__ G_out, int T, int d_h,
             const int32_t *cu, int S) {
    constexpr int NU = picard_nu<TS>();
    __shared__ uint32_t s_heads[L / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int u = (blockIdx.x * U + lane) * NU, t0 = blockIdx.y * L, b = blockIdx.z;
    if (tid < L / 32) s_heads[tid] = 0u;
    __syncthreads();
    if (tid == 0) mark_heads(cu, S, t0, L, s_heads);
    __syncthreads();
    if (u >= d_h) return;   // d_h is a multiple of 8: all NU units exist
    UnitParams prm[NU];
#pragma unroll
    for (int e = 0; e < NU; ++e) prm[e] = load_unit_params(params, d_h, u + e, true);
    const int r0 = warp * SEG;
    const size_t row0 = static_cast<size_t>(b) * T;
    float hprev[NU];
#pragma unroll
    for (int e = 0; e < NU; ++e) hprev[e] = 0.f;
    if (G_in != nullptr && t0 + r0 > 0)
        unpack8<TS>(*reinterpret_cast<const uint2 *>(G_in + (row0 + t0 + r0 - 1) * d_h + u), hprev);
    // the rows are independent given G_in: each batch of PF rows is loaded
    // before any of it is computed, so that PF rows of loads are in flight
    constexpr int PF = 4;
    const int nrows = min(SEG, T - (t0 + r0));
    for (int i0 = 0; i0 < nrows; i0 += PF) {
        uint2 lz[PF], lr[PF], lc[PF], lg[PF];
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            const int t = t0 + r0 + min(i0 + j, nrows - 1);   // in range; duplicates unused
            const TS *p = P + (row0 + t) * 3 * d_h + u;
            lz[j] = *reinterpret_cast<const uint2 *>(p);
            lr[j] = *reinterpret_cast<const uint2 *>(p + d_h);
            lc[j] = *reinterpret_cast<const uint2 *>(p + 2 * d_h);
            if (G_in != nullptr) lg[j] = *reinterpret_cast<const uint2 *>(G_in + (row0 + t) * d_h + u);
        }
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            const int r = r0 + i0 + j, t = t0 + r;
            if (i0 + j < nrows) {
                float pz[NU], pr[NU], pc[NU], f[NU];
                unpack8<TS>(lz[j], pz);
                unpack8<TS>(lr[j], pr);
                unpack8<TS>(lc[j], pc);
                const bool head = head_bit(s_heads, r);
#pragma unroll
                for (int e = 0; e < NU; ++e)
                    f[e] = cell_f_storage<TS>(head ? 0.f : hprev[e], pz[e], pr[e], pc[e], prm[e]);
                *reinterpret_cast<uint2 *>(G_out + (row0 + t) * d_h + u) = pack8<TS>(f);
                if (G_in != nullptr) {
                    unpack8<TS>(lg[j], hprev);
                } else {
#pragma unroll
                    for (int e = 0; e < NU; ++e) hprev[e] = 0.f;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_picard(int dtype, const void *P, const float *params, const void *G_in,
                          void *G_out, int B, int T, int d_h, const int32_t *cu, int S,
                          cudaStream_t stream) {
    const int units = U * (dtype == 1 ? picard_nu<__nv_bfloat16>() : picard_nu<float>());   // per CTA
    const dim3 grid((d_h + units - 1) / units, (T + L - 1) / L, B);
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

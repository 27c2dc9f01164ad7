// Sequential forward on the GPU: h_t = f(h_{t-1}, P_t) from h = 0, one thread
// per (row or segment, hidden unit) (pararnn-torch FAQs, "train() vs eval()":
// eval() runs the sequential step; numerics contract: sequential_apply is the
// reference trajectory).  Lanes of a warp hold consecutive units, so each
// step's three gate loads are coalesced; the next group of steps is loaded
// while the current group is computed.
#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

namespace {

constexpr int SEQ_THREADS = 128;
constexpr int SEQ_D = 8;   // steps per register group

template <typename TS>
__global__ void __launch_bounds__(SEQ_THREADS)
    k_sequential(const TS *__restrict__ P, const float *__restrict__ params, int T, int d_h,
                 const int32_t *__restrict__ cu, TS *__restrict__ H) {
    const int u = blockIdx.x * SEQ_THREADS + threadIdx.x;
    const int row = blockIdx.y;
    if (u >= d_h) return;
    int b = row, s0 = 0, s1 = T;
    if (cu != nullptr) {
        b = 0;
        s0 = min(max(__ldg(cu + row), 0), T);
        s1 = min(max(__ldg(cu + row + 1), s0), T);
    }
    const UnitParams prm = load_unit_params(params, d_h, u, true);
    const size_t stride = static_cast<size_t>(3) * d_h;
    const TS *p = P + (static_cast<size_t>(b) * T + s0) * stride + u;
    TS *h_out = H + (static_cast<size_t>(b) * T + s0) * d_h + u;
    const int n = s1 - s0;

    float cz[SEQ_D], cr[SEQ_D], cc[SEQ_D];
    float nz[SEQ_D], nr[SEQ_D], nc[SEQ_D];
#pragma unroll
    for (int i = 0; i < SEQ_D; ++i) {
        const bool ok = i < n;
        cz[i] = ok ? to_f32(p[i * stride]) : 0.f;
        cr[i] = ok ? to_f32(p[i * stride + d_h]) : 0.f;
        cc[i] = ok ? to_f32(p[i * stride + 2 * d_h]) : 0.f;
    }
    float h = 0.f;
    for (int g = 0; g < n; g += SEQ_D) {
#pragma unroll
        for (int i = 0; i < SEQ_D; ++i) {
            const int t = g + SEQ_D + i;
            const bool ok = t < n;
            nz[i] = ok ? to_f32(p[t * stride]) : 0.f;
            nr[i] = ok ? to_f32(p[t * stride + d_h]) : 0.f;
            nc[i] = ok ? to_f32(p[t * stride + 2 * d_h]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < SEQ_D; ++i) {
            if (g + i < n) {
                h = cell_f(h, cz[i], cr[i], cc[i], prm);
                h_out[static_cast<size_t>(g + i) * d_h] = from_f32<TS>(h);
            }
        }
#pragma unroll
        for (int i = 0; i < SEQ_D; ++i) {
            cz[i] = nz[i];
            cr[i] = nr[i];
            cc[i] = nc[i];
        }
    }
}

}  // namespace

cudaError_t launch_sequential(int dtype, const void *P, const float *params, int B, int T,
                              int d_h, const int32_t *cu, int S, void *H, cudaStream_t stream) {
    const int rows = cu != nullptr ? S : B;
    if (rows == 0 || T == 0) return cudaSuccess;
    const dim3 grid((d_h + SEQ_THREADS - 1) / SEQ_THREADS, rows);
    if (dtype == 1)
        k_sequential<__nv_bfloat16><<<grid, SEQ_THREADS, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(P), params, T, d_h, cu,
            static_cast<__nv_bfloat16 *>(H));
    else
        k_sequential<float><<<grid, SEQ_THREADS, 0, stream>>>(static_cast<const float *>(P),
                                                              params, T, d_h, cu,
                                                              static_cast<float *>(H));
    return cudaGetLastError();
}

}  // namespace nrnn

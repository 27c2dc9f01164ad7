// Decode: one T = 1 step of the diagonal-mix GRU per slot, with the recurrent
// state carried between calls in a fixed (slots, d_h) buffer (pararnn-torch
// FAQs, "How do I pass recurrent state between decode steps?": a carry of
// size (slots, d_h), prefill then decode_wx + decode_step(..., out=) per token).
//
// k_decode_step: h_out = f(h_in, P) elementwise from given preactivations.
// k_decode_step_x: the same step with the input projection fused in: warp w of
// a CTA takes slot s = 4 blockIdx.y + w and unit j = blockIdx.x; its lanes
// split d_in for the three dot products x_s . W_x[g d_h + j] (fp32
// accumulation, shuffle reduction), and lane 0 applies the cell.
#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

namespace {

template <typename TS>
__global__ void __launch_bounds__(256)
    k_decode_step(const TS *__restrict__ P, const float *__restrict__ params,
                  const TS *__restrict__ h_in, TS *__restrict__ h_out, int slots, int d_h) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(slots) * d_h) return;
    const int s = static_cast<int>(i / d_h), j = static_cast<int>(i - static_cast<int64_t>(s) * d_h);
    const UnitParams prm = load_unit_params(params, d_h, j, true);
    const TS *p = P + static_cast<int64_t>(s) * 3 * d_h + j;
    const float h = (h_in != nullptr) ? to_f32(h_in[i]) : 0.f;
    h_out[i] = from_f32<TS>(cell_f(h, to_f32(p[0]), to_f32(p[d_h]), to_f32(p[2 * d_h]), prm));
}

constexpr int DEC_WARPS = 4;

template <typename TS>
__global__ void __launch_bounds__(DEC_WARPS * 32)
    k_decode_step_x(const TS *__restrict__ x, const TS *__restrict__ W, const float *__restrict__ params,
                    const TS *__restrict__ h_in, TS *__restrict__ h_out, int slots, int d_in,
                    int d_h) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = blockIdx.x;
    const int s = blockIdx.y * DEC_WARPS + warp;
    if (s >= slots) return;
    const TS *xs = x + static_cast<int64_t>(s) * d_in;
    const TS *wz = W + static_cast<int64_t>(j) * d_in;
    const TS *wr = W + static_cast<int64_t>(d_h + j) * d_in;
    const TS *wc = W + static_cast<int64_t>(2 * d_h + j) * d_in;
    float az = 0.f, ar = 0.f, ac = 0.f;
    for (int k = lane; k < d_in; k += 32) {
        const float xv = to_f32(xs[k]);
        az = fmaf(xv, to_f32(wz[k]), az);
        ar = fmaf(xv, to_f32(wr[k]), ar);
        ac = fmaf(xv, to_f32(wc[k]), ac);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        az += __shfl_xor_sync(FULL_MASK, az, o);
        ar += __shfl_xor_sync(FULL_MASK, ar, o);
        ac += __shfl_xor_sync(FULL_MASK, ac, o);
    }
    if (lane == 0) {
        // the preactivation is stored in TS before the cell reads it, as on the
        // projection path (decode_wx then decode_step)
        const float pz = round_to<TS>(az), pr = round_to<TS>(ar), pc = round_to<TS>(ac);
        const int64_t i = static_cast<int64_t>(s) * d_h + j;
        const float h = (h_in != nullptr) ? to_f32(h_in[i]) : 0.f;
        h_out[i] = from_f32<TS>(cell_f(h, pz, pr, pc, load_unit_params(params, d_h, j, true)));
    }
}

}  // namespace

cudaError_t launch_decode_step(int dtype, const void *P, const float *params, const void *h_in,
                               void *h_out, int slots, int d_h, cudaStream_t stream) {
    const int64_t n = static_cast<int64_t>(slots) * d_h;
    if (n == 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
    if (dtype == 1)
        k_decode_step<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(P), params, static_cast<const __nv_bfloat16 *>(h_in),
            static_cast<__nv_bfloat16 *>(h_out), slots, d_h);
    else
        k_decode_step<float><<<blocks, 256, 0, stream>>>(static_cast<const float *>(P), params,
                                                         static_cast<const float *>(h_in),
                                                         static_cast<float *>(h_out), slots, d_h);
    return cudaGetLastError();
}

cudaError_t launch_decode_step_x(int dtype, const void *x, const void *W, const float *params,
                                 const void *h_in, void *h_out, int slots, int d_in, int d_h,
                                 cudaStream_t stream) {
    if (slots == 0) return cudaSuccess;
    const dim3 grid(d_h, (slots + DEC_WARPS - 1) / DEC_WARPS);
    if (dtype == 1)
        k_decode_step_x<__nv_bfloat16><<<grid, DEC_WARPS * 32, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(W), params,
            static_cast<const __nv_bfloat16 *>(h_in), static_cast<__nv_bfloat16 *>(h_out), slots,
            d_in, d_h);
    else
        k_decode_step_x<float><<<grid, DEC_WARPS * 32, 0, stream>>>(
            static_cast<const float *>(x), static_cast<const float *>(W), params,
            static_cast<const float *>(h_in), static_cast<float *>(h_out), slots, d_in, d_h);
    return cudaGetLastError();
}

}  // namespace nrnn

// Input projection P = x W_x^T (rows x d_in times d_in x 3 d_h), fp32
// accumulation with fp32 operands (no TF32 rounding).  Register-blocked SIMT
// kernel: 128 x 128 output tile per CTA, 8 x 8 outputs per thread, k-slices
// of 16 staged in shared memory (transposed so that the inner loop reads
// consecutive addresses), next slice prefetched into registers while the
// current one is multiplied.  bf16 operands are widened on load and the
// result rounded to bf16.
#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

namespace {

constexpr int BM = 128, BN = 128, BK = 16, TM = 8, TN = 8, THREADS = 256;

template <typename TS>
__global__ void __launch_bounds__(THREADS)
    k_projection(const TS *__restrict__ X, const TS *__restrict__ W, int64_t rows, int K, int N,
                 TS *__restrict__ P) {
    __shared__ float As[2][BK][BM + 4];
    __shared__ float Bs[2][BK][BN + 4];
    const int tid = threadIdx.x;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int n0 = blockIdx.x * BN;
    // loader mapping: 256 threads x 8 elements = 128 rows x 16 k
    const int lr = tid >> 1, lk = (tid & 1) * 8;
    float ra[8], rb[8];
    auto load_regs = [&](int k0) {
        const int64_t gm = m0 + lr;
        const int gn = n0 + lr;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int kk = k0 + lk + i;
            ra[i] = (gm < rows && kk < K) ? to_f32(X[gm * K + kk]) : 0.f;
            rb[i] = (gn < N && kk < K) ? to_f32(W[static_cast<int64_t>(gn) * K + kk]) : 0.f;
        }
    };
    auto store_smem = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            As[buf][lk + i][lr] = ra[i];
            Bs[buf][lk + i][lr] = rb[i];
        }
    };
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    const int tr = (tid >> 4) * TM, tc = (tid & 15) * TN;
    load_regs(0);
    store_smem(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < K; k0 += BK) {
        const bool more = k0 + BK < K;
        if (more) load_regs(k0 + BK);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], bb[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = As[buf][kk][tr + i];
#pragma unroll
            for (int j = 0; j < TN; ++j) bb[j] = Bs[buf][kk][tc + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        if (more) {
            store_smem(buf ^ 1);
            __syncthreads();
            buf ^= 1;
        }
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t gm = m0 + tr + i;
        if (gm >= rows) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int gn = n0 + tc + j;
            if (gn < N) P[gm * N + gn] = from_f32<TS>(acc[i][j]);
        }
    }
}

}  // namespace

cudaError_t launch_projection(int dtype, const void *x, const void *W, int64_t rows, int d_in,
                              int n_out, void *P, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const dim3 grid((n_out + BN - 1) / BN, static_cast<unsigned>((rows + BM - 1) / BM));
    if (dtype == 1)
        k_projection<__nv_bfloat16><<<grid, THREADS, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(W), rows,
            d_in, n_out, static_cast<__nv_bfloat16 *>(P));
    else
        k_projection<float><<<grid, THREADS, 0, stream>>>(static_cast<const float *>(x),
                                                          static_cast<const float *>(W), rows,
                                                          d_in, n_out, static_cast<float *>(P));
    return cudaGetLastError();
}

}  // namespace nrnn

// Special-function (MUFU) throughput of the GPU the library runs on: the
// denominator of the fused Newton kernel's ALU roofline, whose work is three
// ex2 and two rcp per cell evaluation (fp32 storage) or three tanh (bf16).  One CTA of 1024 threads per SM (the
// dynamic shared memory request keeps a second CTA off the SM) runs eight
// independent chains of the instruction per thread and times itself with the
// SM cycle counter, so the rate comes out per SM clock, independent of the
// clock the GPU happens to run at.
#include <algorithm>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/nrnn.h"

namespace nrnn {

namespace {

constexpr int PROBE_THREADS = 1024;
constexpr int PROBE_CHAINS = 8;
constexpr int PROBE_ITERS = 4096;
constexpr size_t PROBE_SMEM = 160 * 1024;

// OP 0: x <- ex2(-x) (stays in [0.5, 1)); OP 1: x <- 0.5 rcp(x) + 0.75 (stays
// in [1, 1.25]; the fma keeps the compiler from pairing reciprocals away and
// runs on another pipe); OP 2: x <- tanh(x) + 0.5 (stays in [0.5, 1.5])
template <int OP>
__global__ void __launch_bounds__(PROBE_THREADS, 1)
    k_xu_probe(int iters, long long *cycles, float *sink) {
    float x[PROBE_CHAINS];
#pragma unroll
    for (int j = 0; j < PROBE_CHAINS; ++j) x[j] = 0.5f + 0.01f * j + 1e-6f * threadIdx.x;
    __syncthreads();
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < PROBE_CHAINS; ++j) {
            if (OP == 0) {
                asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x[j]) : "f"(-x[j]));
            } else if (OP == 2) {
                float y;
                asm volatile("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x[j]));
                x[j] = y + 0.5f;
            } else {
                float y;
                asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x[j]));
                x[j] = fmaf(y, 0.5f, 0.75f);
            }
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < PROBE_CHAINS; ++j) s += x[j];
    sink[blockIdx.x * PROBE_THREADS + threadIdx.x] = s;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int OP>
int run(int sms, long long *cycles_dev, float *sink, cudaStream_t stream, float *rate) {
    cudaError_t e = cudaFuncSetAttribute(k_xu_probe<OP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(PROBE_SMEM));
    if (e != cudaSuccess) return NRNN_ERR_CUDA;
    for (int rep = 0; rep < 2; ++rep)   // the first launch warms up
        k_xu_probe<OP><<<sms, PROBE_THREADS, PROBE_SMEM, stream>>>(PROBE_ITERS, cycles_dev, sink);
    if (cudaGetLastError() != cudaSuccess) return NRNN_ERR_CUDA;
    std::vector<long long> cyc(sms);
    e = cudaMemcpyAsync(cyc.data(), cycles_dev, sizeof(long long) * sms, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return NRNN_ERR_CUDA;
    std::sort(cyc.begin(), cyc.end());
    const double median = static_cast<double>(cyc[sms / 2]);
    if (median <= 0) return NRNN_ERR_CUDA;
    *rate = static_cast<float>(static_cast<double>(PROBE_THREADS) * PROBE_ITERS * PROBE_CHAINS / median);
    return NRNN_OK;
}

}  // namespace

}  // namespace nrnn

extern "C" int nrnn_probe_xu_rates(float *ex2_per_clk, float *rcp_per_clk, float *tanh_per_clk,
                                   void *stream_) {
    if (ex2_per_clk == nullptr || rcp_per_clk == nullptr || tanh_per_clk == nullptr)
        return NRNN_ERR_INVALID_ARG;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return NRNN_ERR_CUDA;
    long long *cycles = nullptr;
    float *sink = nullptr;
    if (cudaMalloc(&cycles, sizeof(long long) * sms) != cudaSuccess) return NRNN_ERR_CUDA;
    if (cudaMalloc(&sink, sizeof(float) * sms * nrnn::PROBE_THREADS) != cudaSuccess) {
        cudaFree(cycles);
        return NRNN_ERR_CUDA;
    }
    int st = nrnn::run<0>(sms, cycles, sink, stream, ex2_per_clk);
    if (st == NRNN_OK) st = nrnn::run<1>(sms, cycles, sink, stream, rcp_per_clk);
    if (st == NRNN_OK) st = nrnn::run<2>(sms, cycles, sink, stream, tanh_per_clk);
    cudaStreamSynchronize(stream);
    cudaFree(cycles);
    cudaFree(sink);
    return st;
}

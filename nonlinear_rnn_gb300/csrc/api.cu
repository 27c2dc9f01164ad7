// C ABI entry points (declared in include/nrnn.h): argument checks, workspace
// layout, TMA descriptors and the launch sequence of each call.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/nrnn.h"
#include "nrnn_internal.h"
#include "pack_plan.cuh"

using namespace nrnn;

namespace {

std::atomic<uint64_t> g_wait_ns{2000000000ull};
std::atomic<int64_t> g_withhold_tile{-1};
constexpr int MAX_K = 64;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t elem_size(int dtype) { return dtype == NRNN_BF16 ? 2 : 4; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ranges_overlap(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
    if (a == nullptr || b == nullptr || a_bytes == 0 || b_bytes == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + b_bytes && y < x + a_bytes;
}
bool overlaps(const void *a, const void *b, size_t bytes) { return ranges_overlap(a, bytes, b, bytes); }

// Workspace: [counters (K+1) u32 | error u32], then [slots K x n_tiles x 32
// u64], both cleared by one kernel per call, then (per-iteration, K > 1) one
// H buffer, then (a pack cut into segment-aligned chunks) the chunk plan.
// S > 0: the call carries a pack of S segments.
SyncLayout layout(int64_t B, int64_t T, int64_t d_h, int dtype, int K, bool fused, int64_t S = 0) {
    SyncLayout s{};
    const int64_t n_ut = (d_h + TILE_U - 1) / TILE_U;
    const int64_t n_chunks = (T + NEWTON_L - 1) / NEWTON_L;
    const int64_t kk = K > 0 ? K : 1;
    s.plan = S > 0 && pack_plan_applies(B, T, S);
    s.chain_stride = n_chunks + (s.plan ? S : 0);   // a segment adds at most one chunk
    s.n_tiles = B * n_ut * s.chain_stride;
    s.counters_off = 0;
    s.error_off = sizeof(uint32_t) * (kk + 1);
    s.slots_off = align_up(s.error_off + sizeof(uint32_t), 256);
    s.slots_bytes = sizeof(unsigned long long) * 32 * kk * s.n_tiles;
    s.zero_bytes = s.slots_off + s.slots_bytes;
    size_t end = s.zero_bytes;
    s.hbuf_off = align_up(end, 256);
    if (!fused && K > 1) end = s.hbuf_off + elem_size(dtype) * B * T * d_h;
    s.plan_off = align_up(end, 256);
    if (s.plan) end = s.plan_off + pack_plan_bytes(T, S);
    s.total = align_up(end, 256);
    return s;
}

// A pack's chunk plan, built by the first block of the clear kernel while the
// others clear.
struct PlanJob {
    const int32_t *cu;
    int S, n_chunks;
    bool reverse;
    int4 *plan;   // null: no plan
};

constexpr int CLEAR_THREADS = 256;

// The per-call clears of a forward or backward as one kernel instead of two
// memset nodes: the workspace's synchronisation area (counters, error word,
// look-back slots; bytes a multiple of 16) and a small output (the residual
// word, or the parameter gradients; bytes a multiple of 4); with a plan job
// block 0 builds the pack's chunk plan instead (no clearing in it).
__global__ void __launch_bounds__(CLEAR_THREADS)
    k_clear(uint4 *ws, size_t ws16, uint32_t *out, size_t out4, PlanJob job) {
    // the Newton kernel that follows may be scheduled now; it waits for this
    // grid's completion (griddepcontrol.wait) before it touches memory
    asm volatile("griddepcontrol.launch_dependents;");
    const bool planner = job.plan != nullptr;
    if (planner && blockIdx.x == 0) {
        extern __shared__ int sm[];
        build_pack_plan<CLEAR_THREADS>(job.cu, job.S, job.n_chunks, job.reverse, job.plan, sm);
        return;
    }
    const unsigned first = planner ? 1u : 0u, blocks = gridDim.x - first;
    const size_t stride = static_cast<size_t>(blocks) * blockDim.x;
    const size_t i0 = static_cast<size_t>(blockIdx.x - first) * blockDim.x + threadIdx.x;
    for (size_t i = i0; i < ws16; i += stride) ws[i] = make_uint4(0u, 0u, 0u, 0u);
    for (size_t i = i0; i < out4; i += stride) out[i] = 0u;
}

// Above this much shared memory for the plan, it is built by a kernel of its
// own before the clear kernel: every block of a launch reserves the same
// shared memory, and a large reservation would leave the clearing blocks one
// per SM.
constexpr size_t PLAN_IN_CLEAR_MAX_SMEM = 64 * 1024;

cudaError_t clear_for_call(void *ws, size_t ws_bytes, void *out, size_t out_bytes,
                           cudaStream_t stream, const PlanJob &job_in = PlanJob{}) {
    PlanJob job = job_in;
    if (job.plan != nullptr && pack_plan_smem(job.S, job.n_chunks) > PLAN_IN_CLEAR_MAX_SMEM) {
        cudaError_t e = launch_pack_plan(job.cu, job.S, job.n_chunks, job.plan, job.reverse, stream);
        if (e != cudaSuccess) return e;
        job.plan = nullptr;
    }
    const size_t ws16 = ws_bytes / 16, out4 = out_bytes / 4;
    const size_t n = ws16 > out4 ? ws16 : out4;
    const bool planner = job.plan != nullptr;
    if (n == 0 && !planner) return cudaSuccess;
    size_t blocks = (n + CLEAR_THREADS - 1) / CLEAR_THREADS;
    blocks = blocks < 1216 ? blocks : 1216;
    if (blocks == 0) blocks = 1;
    size_t smem = 0;
    if (planner) {
        static std::atomic<unsigned long long> configured{0};
        cudaError_t e = once_per_device(configured, [](int) {
            return cudaFuncSetAttribute(k_clear, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(pack_plan_smem(PACK_PLAN_MAX_S,
                                                                        PACK_PLAN_MAX_CHUNKS)));
        });
        if (e != cudaSuccess) return e;
        smem = pack_plan_smem(job.S, job.n_chunks);
        blocks += 1;   // block 0 plans
    }
    k_clear<<<static_cast<unsigned>(blocks), CLEAR_THREADS, smem, stream>>>(
        static_cast<uint4 *>(ws), ws16, static_cast<uint32_t *>(out), out4, job);
    return cudaGetLastError();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over a (B, T, width) row-major array with a (TILE_U x NEWTON_L x 1) box.
bool make_map(CUtensorMap *m, const void *base, int dtype, int64_t width, int64_t T, int64_t B) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const size_t es = elem_size(dtype);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(width * es),
                             static_cast<cuuint64_t>(width * es * T)};
    cuuint32_t box[3] = {TILE_U, NEWTON_L, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, dtype == NRNN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D map over a (B, T, 3 d_h) preactivation-shaped array seen as (d_h, gate,
// T, B), box (TILE_U x 1 x NEWTON_L x 1): one gate block of a tile, clipped at
// d_h so that a partial unit tile never reaches into the next gate's columns.
bool make_map_gates(CUtensorMap *m, const void *base, int dtype, int64_t d_h, int64_t T, int64_t B) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const size_t es = elem_size(dtype);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d_h), 3, static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d_h * es), static_cast<cuuint64_t>(3 * d_h * es),
                             static_cast<cuuint64_t>(3 * d_h * es * T)};
    cuuint32_t box[4] = {TILE_U, 1, NEWTON_L, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(m, dtype == NRNN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          4, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over a (outer, inner) row-major bf16 or fp32 array, box
// (box_inner x box_outer) with the given swizzle (box_inner * elem must not
// exceed the swizzle span).
bool make_map_2d(CUtensorMap *m, const void *base, int64_t inner, int64_t outer,
                 uint32_t box_inner, uint32_t box_outer, int dtype, CUtensorMapSwizzle swizzle) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const size_t es = elem_size(dtype);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner * es)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, dtype == NRNN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
// the same with the 128-byte swizzle (box_inner * elem must be 128 bytes)
bool make_map_2d_sw128(CUtensorMap *m, const void *base, int64_t inner, int64_t outer,
                       uint32_t box_inner, uint32_t box_outer, int dtype = NRNN_BF16) {
    return make_map_2d(m, base, inner, outer, box_inner, box_outer, dtype,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D bf16 map over x (B, T, d_in) row-major: dims (d_in, T, B), box
// (box_inner, rows, 1), 128-byte (box_inner 64) or 64-byte (box_inner 32) swizzle.
bool make_map_x_swizzled(CUtensorMap *m, const void *x, int64_t d_in, int64_t T, int64_t B,
                         uint32_t box_rows, uint32_t box_inner) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d_in), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d_in * 2),
                             static_cast<cuuint64_t>(d_in * 2 * T)};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(x), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          box_inner == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int check_common(const void *preact, int dtype, const float *params, int64_t B, int64_t T,
                 int64_t d_h, const int32_t *cu, int64_t S) {
    if (dtype != NRNN_F32 && dtype != NRNN_BF16) return NRNN_ERR_INVALID_ARG;
    if (B < 0 || T < 0 || d_h <= 0 || S < 0) return NRNN_ERR_INVALID_ARG;
    if (B * T > 0 && (preact == nullptr || params == nullptr)) return NRNN_ERR_INVALID_ARG;
    if (B > INT32_MAX || T > INT32_MAX || d_h > (1 << 24) || S > INT32_MAX - 1)
        return NRNN_ERR_UNSUPPORTED;
    if (d_h % 8 != 0) return NRNN_ERR_UNSUPPORTED;
    // tile indices and CTA tickets are 32-bit
    if (B * ((d_h + TILE_U - 1) / TILE_U) * ((T + NEWTON_L - 1) / NEWTON_L) > INT32_MAX)
        return NRNN_ERR_UNSUPPORTED;
    if (cu != nullptr && (B != 1 || S < 1)) return NRNN_ERR_CU_SEQLENS;
    if (preact != nullptr && !aligned16(preact)) return NRNN_ERR_INVALID_ARG;
    return NRNN_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? NRNN_OK : NRNN_ERR_CUDA; }

}  // namespace

namespace nrnn {
size_t newton_error_offset(int K) { return layout(0, 0, 8, NRNN_F32, K, true).error_off; }
}  // namespace nrnn

// Synchronous tail of the forward entry points: copies rho and the error word
// to the host, then applies the timeout and residual gates.  With no host
// pointer the call stays asynchronous and returns NRNN_OK.
static int gate_residual(const float *residual_dev, float *residual_host, const uint32_t *err,
                         float residual_fail, cudaStream_t stream) {
    if (residual_host == nullptr) return NRNN_OK;
    uint32_t err_host = 0;
    cudaError_t e =
        cudaMemcpyAsync(residual_host, residual_dev, sizeof(float), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&err_host, err, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return NRNN_ERR_CUDA;
    if (err_host != 0) return NRNN_ERR_TIMEOUT;
    const float rho = *residual_host;
    if (!std::isfinite(rho) || rho > residual_fail) return NRNN_ERR_DIVERGED;
    return NRNN_OK;
}

extern "C" {

const char *nrnn_status_string(int status) {
    switch (status) {
        case NRNN_OK: return "ok";
        case NRNN_ERR_INVALID_ARG: return "invalid argument";
        case NRNN_ERR_CU_SEQLENS: return "invalid cu_seqlens";
        case NRNN_ERR_UNSUPPORTED: return "unsupported configuration";
        case NRNN_ERR_CUDA: return "CUDA error";
        case NRNN_ERR_DIVERGED: return "Newton residual above residual_fail (diverged)";
        case NRNN_ERR_TIMEOUT: return "bounded device wait timed out";
        case NRNN_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int nrnn_version(void) { return 200; }   // 0.2.0: nrnn_input_projection takes a workspace

uint64_t nrnn_set_wait_limit_ns(uint64_t ns) { return g_wait_ns.exchange(ns); }

int nrnn_debug_lookback_form(int64_t B, int64_t T, int64_t d_h, int dtype, int algo) {
    if ((dtype != NRNN_F32 && dtype != NRNN_BF16) || B < 1 || T < 1 || d_h < 1 ||
        (algo != NRNN_ALGO_AUTO && algo != NRNN_ALGO_FUSED && algo != NRNN_ALGO_PER_ITER) ||
        B * ((d_h + TILE_U - 1) / TILE_U) * ((T + NEWTON_L - 1) / NEWTON_L) > INT32_MAX)
        return NRNN_ERR_INVALID_ARG;
    NewtonArgs a{};
    a.B = static_cast<int>(B);
    a.T = static_cast<int>(T);
    a.d_h = static_cast<int>(d_h);
    a.n_ut = static_cast<int>((d_h + TILE_U - 1) / TILE_U);
    a.n_chunks = static_cast<int>((T + NEWTON_L - 1) / NEWTON_L);
    return newton_lookback_form(dtype, algo != NRNN_ALGO_PER_ITER, a);
}

int nrnn_debug_pack_plan(const int32_t *cu_seqlens, int64_t num_segments, int64_t N, int reverse,
                         void *plan, void *stream) {
    if (cu_seqlens == nullptr || plan == nullptr || N < 1 || !pack_plan_applies(1, N, num_segments))
        return NRNN_ERR_INVALID_ARG;
    return launch_pack_plan(cu_seqlens, static_cast<int>(num_segments),
                            static_cast<int>((N + NEWTON_L - 1) / NEWTON_L), static_cast<int4 *>(plan),
                            reverse != 0, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? NRNN_OK
               : NRNN_ERR_CUDA;
}

int64_t nrnn_debug_withhold_publish(int64_t tile) {
    return g_withhold_tile.exchange(tile < 0 || tile > INT32_MAX ? -1 : tile);
}

int nrnn_validate_cu_seqlens(const int32_t *cu_host, int64_t num_segments, int64_t N) {
    if (cu_host == nullptr || num_segments < 0 || N < 0) return NRNN_ERR_INVALID_ARG;
    if (num_segments < 1) return NRNN_ERR_CU_SEQLENS;
    if (cu_host[0] != 0) return NRNN_ERR_CU_SEQLENS;
    for (int64_t i = 0; i < num_segments; ++i)
        if (cu_host[i + 1] < cu_host[i]) return NRNN_ERR_CU_SEQLENS;
    if (static_cast<int64_t>(cu_host[num_segments]) != N) return NRNN_ERR_CU_SEQLENS;
    return NRNN_OK;
}

size_t nrnn_newton_workspace_bytes(int64_t B, int64_t T, int64_t d_h, int dtype, int K,
                                   int algo) {
    if (B < 0 || T < 0 || d_h <= 0 || K < 0 || K > MAX_K) return 0;
    if (dtype != NRNN_F32 && dtype != NRNN_BF16) return 0;
    if (algo < NRNN_ALGO_AUTO || algo > NRNN_ALGO_FUSED) return 0;
    return layout(B, T, d_h, dtype, K, algo != NRNN_ALGO_PER_ITER).total;
}

size_t nrnn_newton_workspace_bytes_pack(int64_t N, int64_t d_h, int dtype, int K, int algo,
                                        int64_t num_segments) {
    if (num_segments < 1) return 0;
    if (nrnn_newton_workspace_bytes(1, N, d_h, dtype, K, algo) == 0) return 0;
    return layout(1, N, d_h, dtype, K, algo != NRNN_ALGO_PER_ITER, num_segments).total;
}

int nrnn_newton_forward(const void *preact, int dtype, const float *params, int64_t B,
                        int64_t T, int64_t d_h, const int32_t *cu_seqlens,
                        int64_t num_segments, int K, float residual_fail, int algo,
                        void *H_out, float *residual_dev, float *residual_host,
                        void *workspace, size_t ws_bytes, void *stream) {
    return nrnn_newton_forward_init(preact, dtype, params, B, T, d_h, cu_seqlens, num_segments,
                                    nullptr, K, residual_fail, algo, H_out, residual_dev,
                                    residual_host, workspace, ws_bytes, stream);
}

int nrnn_newton_forward_init(const void *preact, int dtype, const float *params, int64_t B,
                             int64_t T, int64_t d_h, const int32_t *cu_seqlens,
                             int64_t num_segments, const void *H_init, int K,
                             float residual_fail, int algo, void *H_out, float *residual_dev,
                             float *residual_host, void *workspace, size_t ws_bytes,
                             void *stream_) {
    int st = check_common(preact, dtype, params, B, T, d_h, cu_seqlens, num_segments);
    if (st != NRNN_OK) return st;
    if (H_init != nullptr &&
        (!aligned16(H_init) ||
         overlaps(H_init, H_out, elem_size(dtype) * static_cast<size_t>(B * T * d_h))))
        return NRNN_ERR_INVALID_ARG;
    if (K < 0 || K > MAX_K || residual_dev == nullptr) return NRNN_ERR_INVALID_ARG;
    if (algo < NRNN_ALGO_AUTO || algo > NRNN_ALGO_FUSED) return NRNN_ERR_INVALID_ARG;
    if (B * T > 0 && (H_out == nullptr || !aligned16(H_out))) return NRNN_ERR_INVALID_ARG;
    {
        const size_t hb = elem_size(dtype) * static_cast<size_t>(B * T * d_h);
        if (ranges_overlap(preact, 3 * hb, H_out, hb)) return NRNN_ERR_INVALID_ARG;
    }
    const bool fused = algo != NRNN_ALGO_PER_ITER;
    // a pack is cut into segment-aligned chunks when the workspace was sized
    // for it (nrnn_newton_workspace_bytes_pack), else into chunks of the time axis
    SyncLayout ly = layout(B, T, d_h, dtype, K, fused, cu_seqlens ? num_segments : 0);
    if (ly.plan && ws_bytes < ly.total) ly = layout(B, T, d_h, dtype, K, fused);
    if (workspace == nullptr || ws_bytes < ly.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return NRNN_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    uint32_t *res_bits = reinterpret_cast<uint32_t *>(residual_dev);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + ly.error_off);
    const int S = static_cast<int>(cu_seqlens ? num_segments : 0);

    // one kernel clears counters, error word, slots and rho (rho accumulates by
    // atomicMax into residual_dev) and builds the chunk plan of a
    // segment-aligned pack, which its dependents, the Newton launches, read
    PlanJob job{};
    if (ly.plan && K > 0 && B * T > 0)
        job = PlanJob{cu_seqlens, S, static_cast<int>((T + NEWTON_L - 1) / NEWTON_L), false,
                      reinterpret_cast<int4 *>(ws + ly.plan_off)};
    cudaError_t e = clear_for_call(ws, ly.zero_bytes, residual_dev, sizeof(float), stream, job);
    if (e != cudaSuccess) return NRNN_ERR_CUDA;

    if (B * T > 0) {
        if (K == 0) {
            const size_t hbytes = elem_size(dtype) * B * T * d_h;
            e = H_init ? cudaMemcpyAsync(H_out, H_init, hbytes, cudaMemcpyDeviceToDevice, stream)
                       : cudaMemsetAsync(H_out, 0, hbytes, stream);
            if (e == cudaSuccess)
                e = launch_residual(dtype, preact, params, H_init ? H_out : nullptr,
                                    static_cast<int>(B), static_cast<int>(T),
                                    static_cast<int>(d_h), cu_seqlens, S, res_bits, stream);
            if (e != cudaSuccess) return NRNN_ERR_CUDA;
        } else {
            CUtensorMap tmP;
            if (!make_map(&tmP, preact, dtype, 3 * d_h, T, B)) return NRNN_ERR_CUDA;
            NewtonArgs a{};
            a.params = params;
            a.cu = cu_seqlens;
            a.S = S;
            a.B = static_cast<int>(B);
            a.T = static_cast<int>(T);
            a.d_h = static_cast<int>(d_h);
            a.n_ut = static_cast<int>((d_h + TILE_U - 1) / TILE_U);
            a.n_chunks = static_cast<int>((T + NEWTON_L - 1) / NEWTON_L);
            a.slots = reinterpret_cast<unsigned long long *>(ws + ly.slots_off);
            a.residual_bits = res_bits;
            a.error = err;
            a.wait_ns = g_wait_ns.load();
            a.withhold_tile = static_cast<int>(g_withhold_tile.load());
            if (ly.plan) {   // the kernels read the plan, not the segment bounds
                a.plan = reinterpret_cast<const int4 *>(ws + ly.plan_off);
                a.chain_stride = static_cast<int>(ly.chain_stride);
            }
            uint32_t *counters = reinterpret_cast<uint32_t *>(ws + ly.counters_off);
            if (fused) {
                CUtensorMap tmH = tmP;
                if (H_init != nullptr && !make_map(&tmH, H_init, dtype, d_h, T, B))
                    return NRNN_ERR_CUDA;
                a.H_prev = H_init;
                a.H_next = H_out;
                a.k_first = 1;
                a.k_last = K;
                a.last = 1;
                a.ticket = counters;
                CUtensorMap tmO;
                if (!make_map(&tmO, H_out, dtype, d_h, T, B)) return NRNN_ERR_CUDA;
                e = launch_newton(dtype, true, tmP, tmH, tmO, a, ly.n_tiles, stream, ly.plan);
                if (e != cudaSuccess) return NRNN_ERR_CUDA;
            } else {
                void *hbuf = ws + ly.hbuf_off;
                const void *prev = H_init;
                for (int k = 1; k <= K; ++k) {
                    // iteration K lands in H_out; earlier ones alternate with hbuf
                    void *dst = ((K - k) % 2 == 0) ? H_out : hbuf;
                    CUtensorMap tmH = tmP, tmO;
                    if (prev != nullptr && !make_map(&tmH, prev, dtype, d_h, T, B))
                        return NRNN_ERR_CUDA;
                    if (!make_map(&tmO, dst, dtype, d_h, T, B)) return NRNN_ERR_CUDA;
                    a.H_prev = prev;
                    a.H_next = dst;
                    a.k_first = a.k_last = k;
                    a.last = (k == K) ? 1 : 0;
                    a.ticket = counters + k;
                    e = launch_newton(dtype, false, tmP, tmH, tmO, a, ly.n_tiles, stream, ly.plan);
                    if (e != cudaSuccess) return NRNN_ERR_CUDA;
                    prev = dst;
                }
            }
        }
    }
    return gate_residual(residual_dev, residual_host, err, residual_fail, stream);
}

int nrnn_newton_forward_x(const void *x, const void *W_x, int dtype, const float *params,
                          int64_t B, int64_t T, int64_t d_in, int64_t d_h,
                          const int32_t *cu_seqlens, int64_t num_segments, int K,
                          float residual_fail, void *H_out, float *residual_dev,
                          float *residual_host, void *workspace, size_t ws_bytes, void *stream_) {
    if (dtype == NRNN_F32) return NRNN_ERR_UNSUPPORTED;
    int st = check_common(x, dtype, params, B, T, d_h, cu_seqlens, num_segments);
    if (st != NRNN_OK) return st;
    if (K < 1 || K > MAX_K || residual_dev == nullptr || d_in <= 0) return NRNN_ERR_INVALID_ARG;
    if (d_in % 8 != 0 || d_in > INT32_MAX) return NRNN_ERR_UNSUPPORTED;
    if (B * T > 0 && (W_x == nullptr || H_out == nullptr || !aligned16(W_x) || !aligned16(H_out)))
        return NRNN_ERR_INVALID_ARG;
    const SyncLayout ly = layout(B, T, d_h, dtype, K, true);
    if (workspace == nullptr || ws_bytes < ly.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return NRNN_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + ly.error_off);
    cudaError_t e = clear_for_call(ws, ly.zero_bytes, residual_dev, sizeof(float), stream);
    if (e != cudaSuccess) return NRNN_ERR_CUDA;
    if (B * T > 0) {
        CUtensorMap tmX, tmW;
        // 32-wide K slices with the 64-byte swizzle (the kernel's stages)
        if (!make_map_x_swizzled(&tmX, x, d_in, T, B, NEWTON_L, 32) ||
            !make_map_2d(&tmW, W_x, d_in, 3 * d_h, 32, TILE_U, NRNN_BF16, CU_TENSOR_MAP_SWIZZLE_64B))
            return NRNN_ERR_CUDA;
        NewtonArgs a{};
        a.params = params;
        a.cu = cu_seqlens;
        a.S = static_cast<int>(cu_seqlens ? num_segments : 0);
        a.B = static_cast<int>(B);
        a.T = static_cast<int>(T);
        a.d_h = static_cast<int>(d_h);
        a.d_in = static_cast<int>(d_in);
        a.n_ut = static_cast<int>((d_h + TILE_U - 1) / TILE_U);
        a.n_chunks = static_cast<int>((T + NEWTON_L - 1) / NEWTON_L);
        a.slots = reinterpret_cast<unsigned long long *>(ws + ly.slots_off);
        a.residual_bits = reinterpret_cast<uint32_t *>(residual_dev);
        a.error = err;
        a.wait_ns = g_wait_ns.load();
        a.withhold_tile = static_cast<int>(g_withhold_tile.load());
        a.H_prev = nullptr;
        a.H_next = H_out;
        a.k_first = 1;
        a.k_last = K;
        a.last = 1;
        a.ticket = reinterpret_cast<uint32_t *>(ws + ly.counters_off);
        CUtensorMap tmO;
        if (!make_map(&tmO, H_out, dtype, d_h, T, B)) return NRNN_ERR_CUDA;
        if (launch_newton_x(tmX, tmW, tmO, a, ly.n_tiles, stream) != cudaSuccess) return NRNN_ERR_CUDA;
    }
    return gate_residual(residual_dev, residual_host, err, residual_fail, stream);
}

int nrnn_newton_backward(const void *preact, int dtype, const float *params, int64_t B,
                         int64_t T, int64_t d_h, const int32_t *cu_seqlens, int64_t num_segments,
                         const void *H, const void *gH, void *gP, float *gparams,
                         void *workspace, size_t ws_bytes, void *stream_) {
    int st = check_common(preact, dtype, params, B, T, d_h, cu_seqlens, num_segments);
    if (st != NRNN_OK) return st;
    if (gparams == nullptr) return NRNN_ERR_INVALID_ARG;
    if (B * T > 0 && (H == nullptr || gH == nullptr || gP == nullptr || !aligned16(H) ||
                      !aligned16(gH) || !aligned16(gP)))
        return NRNN_ERR_INVALID_ARG;
    // segment-aligned chunks of a pack when the workspace has room for them
    // (nrnn_newton_workspace_bytes_pack with K = 1)
    SyncLayout ly = layout(B, T, d_h, dtype, 1, true, cu_seqlens ? num_segments : 0);
    if (ly.plan && ws_bytes < ly.total) ly = layout(B, T, d_h, dtype, 1, true);
    if (workspace == nullptr || ws_bytes < ly.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return NRNN_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    if (B * T == 0)
        return cuda_status(cudaMemsetAsync(gparams, 0, sizeof(float) * 6 * d_h, stream));
    PlanJob job{};
    if (ly.plan)
        job = PlanJob{cu_seqlens, static_cast<int>(num_segments),
                      static_cast<int>((T + NEWTON_L - 1) / NEWTON_L), true,
                      reinterpret_cast<int4 *>(ws + ly.plan_off)};
    cudaError_t e = clear_for_call(ws, ly.zero_bytes, gparams, sizeof(float) * 6 * d_h, stream, job);
    if (e != cudaSuccess) return NRNN_ERR_CUDA;
    CUtensorMap tmP, tmH, tmG, tmGP;
    if (!make_map(&tmP, preact, dtype, 3 * d_h, T, B) || !make_map(&tmH, H, dtype, d_h, T, B) ||
        !make_map(&tmG, gH, dtype, d_h, T, B) || !make_map_gates(&tmGP, gP, dtype, d_h, T, B))
        return NRNN_ERR_CUDA;
    BackwardArgs a{};
    a.H = H;
    a.gH = gH;
    a.gparams = gparams;
    a.params = params;
    a.cu = cu_seqlens;
    a.S = static_cast<int>(cu_seqlens ? num_segments : 0);
    a.B = static_cast<int>(B);
    a.T = static_cast<int>(T);
    a.d_h = static_cast<int>(d_h);
    a.n_ut = static_cast<int>((d_h + TILE_U - 1) / TILE_U);
    a.n_chunks = static_cast<int>((T + NEWTON_L - 1) / NEWTON_L);
    if (ly.plan) {   // the kernel reads the plan, not the segment bounds
        a.plan = reinterpret_cast<const int4 *>(ws + ly.plan_off);
        a.n_chunks = static_cast<int>(ly.chain_stride);
    }
    a.slots = reinterpret_cast<unsigned long long *>(ws + ly.slots_off);
    a.ticket = reinterpret_cast<uint32_t *>(ws + ly.counters_off);
    a.error = reinterpret_cast<uint32_t *>(ws + ly.error_off);
    a.wait_ns = g_wait_ns.load();
    a.gP = gP;
    return cuda_status(launch_backward(dtype, tmP, tmH, tmG, tmGP, a, ly.n_tiles, stream, ly.plan));
}

int nrnn_picard(const void *preact, int dtype, const float *params, int64_t B, int64_t T,
                int64_t d_h, const int32_t *cu_seqlens, int64_t num_segments, int sweeps,
                void *H_out, void *H_tmp, void *stream_) {
    int st = check_common(preact, dtype, params, B, T, d_h, cu_seqlens, num_segments);
    if (st != NRNN_OK) return st;
    const size_t hbytes = elem_size(dtype) * static_cast<size_t>(B * T * d_h);
    if (sweeps < 0 || (B * T > 0 && H_out == nullptr)) return NRNN_ERR_INVALID_ARG;
    if (sweeps >= 2 && B * T > 0 && (H_tmp == nullptr || overlaps(H_tmp, H_out, hbytes)))
        return NRNN_ERR_INVALID_ARG;
    if (B * T > 0 && (!aligned16(H_out) || (sweeps >= 2 && !aligned16(H_tmp)) ||
                      ranges_overlap(preact, 3 * hbytes, H_out, hbytes) ||
                      (sweeps >= 2 && ranges_overlap(preact, 3 * hbytes, H_tmp, hbytes))))
        return NRNN_ERR_INVALID_ARG;
    if (B * T == 0) return NRNN_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (sweeps == 0) return cuda_status(cudaMemsetAsync(H_out, 0, hbytes, stream));
    const void *src = nullptr;
    for (int k = 1; k <= sweeps; ++k) {
        void *dst = ((sweeps - k) % 2 == 0) ? H_out : H_tmp;   // the last sweep lands in H_out
        cudaError_t e = launch_picard(dtype, preact, params, src, dst, static_cast<int>(B),
                                      static_cast<int>(T), static_cast<int>(d_h), cu_seqlens,
                                      static_cast<int>(cu_seqlens ? num_segments : 0), stream);
        if (e != cudaSuccess) return NRNN_ERR_CUDA;
        src = dst;
    }
    return NRNN_OK;
}

int nrnn_sequential_forward(const void *preact, int dtype, const float *params, int64_t B,
                            int64_t T, int64_t d_h, const int32_t *cu_seqlens,
                            int64_t num_segments, void *H_out, void *stream) {
    int st = check_common(preact, dtype, params, B, T, d_h, cu_seqlens, num_segments);
    if (st != NRNN_OK) return st;
    if (B * T > 0 && H_out == nullptr) return NRNN_ERR_INVALID_ARG;
    if (B * T == 0) return NRNN_OK;
    return cuda_status(launch_sequential(dtype, preact, params, static_cast<int>(B),
                                         static_cast<int>(T), static_cast<int>(d_h), cu_seqlens,
                                         static_cast<int>(cu_seqlens ? num_segments : 0), H_out,
                                         static_cast<cudaStream_t>(stream)));
}

int nrnn_decode_step(const void *preact, int dtype, const float *params, int64_t slots,
                     int64_t d_h, const void *h_in, void *h_out, void *stream) {
    if (dtype != NRNN_F32 && dtype != NRNN_BF16) return NRNN_ERR_INVALID_ARG;
    if (slots < 0 || d_h <= 0) return NRNN_ERR_INVALID_ARG;
    if (slots == 0) return NRNN_OK;
    if (preact == nullptr || params == nullptr || h_out == nullptr) return NRNN_ERR_INVALID_ARG;
    if (slots * d_h > INT32_MAX || d_h > INT32_MAX / 3) return NRNN_ERR_UNSUPPORTED;
    if (ranges_overlap(h_out, elem_size(dtype) * static_cast<size_t>(slots * d_h), preact,
                       elem_size(dtype) * static_cast<size_t>(slots * 3 * d_h)))
        return NRNN_ERR_INVALID_ARG;
    return cuda_status(launch_decode_step(dtype, preact, params, h_in, h_out,
                                          static_cast<int>(slots), static_cast<int>(d_h),
                                          static_cast<cudaStream_t>(stream)));
}

int nrnn_decode_step_x(const void *x, const void *W_x, int dtype, const float *params,
                       int64_t slots, int64_t d_in, int64_t d_h, const void *h_in, void *h_out,
                       void *stream) {
    if (dtype != NRNN_F32 && dtype != NRNN_BF16) return NRNN_ERR_INVALID_ARG;
    if (slots < 0 || d_in <= 0 || d_h <= 0) return NRNN_ERR_INVALID_ARG;
    if (slots == 0) return NRNN_OK;
    if (x == nullptr || W_x == nullptr || params == nullptr || h_out == nullptr)
        return NRNN_ERR_INVALID_ARG;
    if (slots > 8 * 65535 || d_h > INT32_MAX / 3 || d_in > INT32_MAX || d_in % 8 != 0)
        return NRNN_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(W_x)) return NRNN_ERR_INVALID_ARG;
    if (dtype == NRNN_BF16) {
        // the projection on the tensor cores, the step in the epilogue
        CUtensorMap tmX, tmW;
        const int64_t xg_tiles = (slots + 127) / 128 * ((d_h + 63) / 64);   // 32-bit tile indices
        if (slots >= DECODE_XG_MIN_SLOTS && d_in >= DECODE_XG_MIN_D_IN && d_h % 8 == 0 &&
            xg_tiles <= INT32_MAX && aligned16(params) && aligned16(h_out) &&
            (h_in == nullptr || aligned16(h_in))) {
            // more than one slot tile: M = 128 slots by 64 units (z, r, c rows) per
            // tile; a shorter K loop leaves the epilogue's cell work exposed
            if (!make_map_2d_sw128(&tmX, x, d_in, slots, 64, 128) ||
                !make_map_2d_sw128(&tmW, W_x, d_in, 3 * d_h, 64, 64))
                return NRNN_ERR_CUDA;
            return cuda_status(launch_decode_step_xg(tmX, tmW, params, h_in, h_out,
                                                     static_cast<int>(slots), static_cast<int>(d_in),
                                                     static_cast<int>(d_h),
                                                     static_cast<cudaStream_t>(stream)));
        }
        const int units = decode_xtc_units(static_cast<int>(slots), static_cast<int>(d_h));
        if (!make_map_2d_sw128(&tmX, x, d_in, slots, 64, 64) ||
            !make_map_2d_sw128(&tmW, W_x, d_in, 3 * d_h, 64, static_cast<uint32_t>(units)))
            return NRNN_ERR_CUDA;
        return cuda_status(launch_decode_step_xtc(tmX, tmW, params, h_in, h_out,
                                                  static_cast<int>(slots), static_cast<int>(d_in),
                                                  static_cast<int>(d_h),
                                                  static_cast<cudaStream_t>(stream)));
    }
    return cuda_status(launch_decode_step_x(dtype, x, W_x, params, h_in, h_out,
                                            static_cast<int>(slots), static_cast<int>(d_in),
                                            static_cast<int>(d_h),
                                            static_cast<cudaStream_t>(stream)));
}

int nrnn_residual(const void *preact, int dtype, const float *params, int64_t B, int64_t T,
                  int64_t d_h, const int32_t *cu_seqlens, int64_t num_segments, const void *G,
                  float *residual_dev, void *stream_) {
    int st = check_common(preact, dtype, params, B, T, d_h, cu_seqlens, num_segments);
    if (st != NRNN_OK) return st;
    if (residual_dev == nullptr || (B * T > 0 && G == nullptr)) return NRNN_ERR_INVALID_ARG;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (cudaMemsetAsync(residual_dev, 0, sizeof(float), stream) != cudaSuccess) return NRNN_ERR_CUDA;
    if (B * T == 0) return NRNN_OK;
    return cuda_status(launch_residual(dtype, preact, params, G, static_cast<int>(B),
                                       static_cast<int>(T), static_cast<int>(d_h), cu_seqlens,
                                       static_cast<int>(cu_seqlens ? num_segments : 0),
                                       reinterpret_cast<uint32_t *>(residual_dev), stream));
}

size_t nrnn_input_projection_workspace_bytes(int dtype, int64_t d_in, int64_t d_h) {
    if (dtype == NRNN_BF16 && d_in > 0 && d_h > 0) return 0;
    if (dtype != NRNN_F32 || d_in <= 0 || d_h <= 0 || d_in > INT32_MAX || 3 * d_h > INT32_MAX)
        return 0;
    // the low part of W_x, (3 d_h, d_in) fp32
    return sizeof(float) * static_cast<size_t>(3 * d_h) * static_cast<size_t>(d_in);
}

int nrnn_input_projection(const void *x, const void *W_x, int dtype, int64_t rows, int64_t d_in,
                          int64_t d_h, void *preact, void *workspace, size_t ws_bytes,
                          void *stream) {
    if (dtype != NRNN_F32 && dtype != NRNN_BF16) return NRNN_ERR_INVALID_ARG;
    if (rows < 0 || d_in <= 0 || d_h <= 0) return NRNN_ERR_INVALID_ARG;
    if (rows > 0 && (x == nullptr || W_x == nullptr || preact == nullptr)) return NRNN_ERR_INVALID_ARG;
    if (d_in % 8 != 0 || d_h % 8 != 0 || d_in > INT32_MAX || 3 * d_h > INT32_MAX ||
        rows > INT32_MAX)
        return NRNN_ERR_UNSUPPORTED;
    if (rows == 0) return NRNN_OK;
    const size_t need = nrnn_input_projection_workspace_bytes(dtype, d_in, d_h);
    if (need > 0 && (workspace == nullptr || ws_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return NRNN_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(W_x) || !aligned16(preact)) return NRNN_ERR_INVALID_ARG;
    CUtensorMap tmA, tmB, tmP;
    const int64_t n_out = 3 * d_h;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == NRNN_BF16) {
        if (!make_map_2d_sw128(&tmA, x, d_in, rows, PROJ_TC_BOX_K, PROJ_TC_BOX_M) ||
            !make_map_2d_sw128(&tmB, W_x, d_in, n_out, PROJ_TC_BOX_K, PROJ_TC_BOX_N) ||
            !make_map_2d(&tmP, preact, n_out, rows, PROJ_OUT_BOX, PROJ_OUT_BOX, NRNN_BF16,
                         CU_TENSOR_MAP_SWIZZLE_64B))
            return NRNN_ERR_CUDA;
        return cuda_status(launch_projection_tc(tmA, tmB, tmP, rows, static_cast<int>(d_in),
                                                static_cast<int>(n_out), st));
    }
    // split-TF32: the static operand W_x is split once per call (its low part
    // into the workspace); the kernel splits the x tiles as they arrive
    const int bn = projection_tf32x3_bn(static_cast<int>(n_out));
    CUtensorMap tmBlo;
    if (!make_map_2d_sw128(&tmA, x, d_in, rows, PROJ_T3_BOX_K, PROJ_T3_BOX_M, NRNN_F32) ||
        !make_map_2d_sw128(&tmB, W_x, d_in, n_out, PROJ_T3_BOX_K, bn, NRNN_F32) ||
        !make_map_2d_sw128(&tmBlo, workspace, d_in, n_out, PROJ_T3_BOX_K, bn, NRNN_F32) ||
        !make_map_2d(&tmP, preact, n_out, rows, PROJ_OUT_BOX, PROJ_OUT_BOX, NRNN_F32,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return NRNN_ERR_CUDA;
    cudaError_t e = launch_split_low(W_x, workspace, n_out * d_in, st);
    if (e != cudaSuccess) return NRNN_ERR_CUDA;
    return cuda_status(launch_projection_tf32x3(tmA, tmB, tmBlo, tmP, rows, static_cast<int>(d_in),
                                                static_cast<int>(n_out), st));
}

int nrnn_debug_head_mask(const int32_t *cu_seqlens, int64_t num_segments, int64_t N,
                         uint8_t *mask_dev, void *stream) {
    if (N < 0 || num_segments < 0 || (N > 0 && mask_dev == nullptr)) return NRNN_ERR_INVALID_ARG;
    if (N == 0) return NRNN_OK;
    if (num_segments > INT32_MAX - 1) return NRNN_ERR_UNSUPPORTED;
    return cuda_status(launch_head_mask(cu_seqlens, static_cast<int>(num_segments), N, mask_dev,
                                        static_cast<cudaStream_t>(stream)));
}

int nrnn_debug_bounded_wait(const uint32_t *flag_dev, uint64_t wait_ns, uint32_t *result_dev,
                            void *stream) {
    if (flag_dev == nullptr || result_dev == nullptr) return NRNN_ERR_INVALID_ARG;
    return cuda_status(
        launch_bounded_wait(flag_dev, wait_ns, result_dev, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// Newton forward on host buffers.  The problem is cut into blocks that need no
// data from one another -- groups of batch rows, or for a cu_seqlens pack
// groups of whole segments -- and each block goes host -> device, through
// nrnn_newton_forward, and device -> host on one of three staging slots.  The
// copies in and out run on two library streams, the kernels on the caller's
// stream, ordered by events, so the copies of one block overlap the kernels
// and the copies of its neighbours.  Results equal nrnn_newton_forward on the
// whole problem up to the look-back's composition order (a pack's blocks
// start their time chunks at their own first token).  The input of a block is
// either its preactivations (nrnn_newton_forward_host) or its rows of x, which
// nrnn_input_projection turns into preactivations on the device before the
// forward (nrnn_newton_forward_x_host: d_in instead of 3 d_h values per token
// cross the host link).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/nrnn.h"
#include "nrnn_internal.h"

namespace {

constexpr int NSLOT = 3;
constexpr size_t ALIGN = 256;

size_t align_up(size_t v) { return (v + ALIGN - 1) / ALIGN * ALIGN; }
size_t esize(int dtype) { return dtype == NRNN_BF16 ? 2 : 4; }

struct Block {
    int64_t b0, nb;     // rows [b0, b0 + nb)
    int64_t t0, nt;     // tokens [t0, t0 + nt) of those rows
    int64_t s0, ns;     // pack: segments [s0, s0 + ns), rebased bounds at cu_off
    int64_t cu_off;
};

struct Plan {
    std::vector<Block> blocks;
    size_t x_bytes = 0, p_bytes = 0, h_bytes = 0, ws_bytes = 0;   // per slot
    size_t slots_off[NSLOT] = {}, res_off = 0, err_off = 0, cu_off = 0, total = 0;
    size_t proj_off = 0, proj_bytes = 0;   // x input: the projection's workspace (one)
    int64_t cu_ints = 0;
};

// Splits the problem into blocks of about tokens_per_block tokens (0: about
// 16 blocks) and lays out the staging area: per slot [x rows (d_in > 0)] [P]
// [H] [forward workspace], then the projection's workspace, residuals, error
// words and rebased segment bounds.  Returns false on a bad shape.
bool make_plan(int64_t B, int64_t T, int64_t d_in, int64_t d_h, int dtype, int K,
               const int32_t *cu, int64_t S, int64_t tokens_per_block, Plan &pl) {
    const int64_t total = B * T;
    if (total == 0) return true;
    if (tokens_per_block <= 0) tokens_per_block = (total + 15) / 16;
    if (cu == nullptr) {
        const int64_t rows = std::max<int64_t>(1, std::min<int64_t>(B, tokens_per_block / std::max<int64_t>(T, 1)));
        for (int64_t b = 0; b < B; b += rows)
            pl.blocks.push_back({b, std::min(rows, B - b), 0, T, 0, 0, 0});
    } else {
        int64_t s = 0;
        while (s < S) {
            const int64_t s0 = s;
            int64_t tok = 0;
            do {
                tok += static_cast<int64_t>(cu[s + 1]) - cu[s];
                ++s;
            } while (s < S && tok < tokens_per_block);
            pl.blocks.push_back({0, 1, cu[s0], tok, s0, s - s0, pl.cu_ints});
            pl.cu_ints += (s - s0) + 1;
        }
    }
    const size_t es = esize(dtype);
    for (const Block &bk : pl.blocks) {
        const size_t n = static_cast<size_t>(bk.nb * bk.nt);
        if (d_in > 0) pl.x_bytes = std::max(pl.x_bytes, align_up(n * d_in * es));
        pl.p_bytes = std::max(pl.p_bytes, align_up(n * 3 * d_h * es));
        pl.h_bytes = std::max(pl.h_bytes, align_up(n * d_h * es));
        const size_t ws = cu == nullptr
                              ? nrnn_newton_workspace_bytes(bk.nb, bk.nt, d_h, dtype, K, NRNN_ALGO_FUSED)
                              : nrnn_newton_workspace_bytes_pack(bk.nt, d_h, dtype, K, NRNN_ALGO_FUSED,
                                                                 bk.ns);
        if (ws == 0 && bk.nb * bk.nt > 0) return false;
        pl.ws_bytes = std::max(pl.ws_bytes, align_up(ws));
    }
    size_t off = 0;
    for (int i = 0; i < NSLOT; ++i) {
        pl.slots_off[i] = off;
        off += pl.x_bytes + pl.p_bytes + pl.h_bytes + pl.ws_bytes;
    }
    if (d_in > 0) {
        pl.proj_off = off;
        pl.proj_bytes = align_up(nrnn_input_projection_workspace_bytes(dtype, d_in, d_h));
        off += pl.proj_bytes;
    }
    const size_t nblk = pl.blocks.size();
    pl.res_off = off;                                   // residuals, then error words:
    pl.err_off = off + sizeof(float) * nblk;            // one copy brings both home
    off = align_up(pl.err_off + sizeof(uint32_t) * nblk);
    pl.cu_off = off;
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(pl.cu_ints));
    pl.total = off;
    return true;
}

// Copy streams and slot events of the calling host thread on one device,
// created on first use and kept for the thread's lifetime.
struct Lanes {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t loaded[NSLOT], computed[NSLOT], drained[NSLOT];
};

Lanes *lanes_for_current_device() {
    thread_local std::vector<Lanes> per_dev;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    if (per_dev.size() <= static_cast<size_t>(dev)) per_dev.resize(dev + 1);
    Lanes &l = per_dev[dev];
    if (!l.ready) {
        if (cudaStreamCreateWithFlags(&l.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&l.out, cudaStreamNonBlocking) != cudaSuccess)
            return nullptr;
        for (int i = 0; i < NSLOT; ++i)
            if (cudaEventCreateWithFlags(&l.loaded[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&l.computed[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&l.drained[i], cudaEventDisableTiming) != cudaSuccess)
                return nullptr;
        l.ready = true;
    }
    return &l;
}

int validate(const void *preact_host, int dtype, const float *params, int64_t B, int64_t T,
             int64_t d_h, const int32_t *cu, int64_t S, int K, const void *H_host,
             const float *residual_host, int64_t d_in = 0, const void *W_x = nullptr) {
    if (dtype != NRNN_F32 && dtype != NRNN_BF16) return NRNN_ERR_INVALID_ARG;
    if (B < 0 || T < 0 || d_h <= 0 || K < 0 || residual_host == nullptr) return NRNN_ERR_INVALID_ARG;
    if (B > INT32_MAX || T > INT32_MAX || d_h > (1 << 24)) return NRNN_ERR_UNSUPPORTED;
    if (d_h % 8 != 0) return NRNN_ERR_UNSUPPORTED;
    if (B * T > 0 && (preact_host == nullptr || H_host == nullptr || params == nullptr))
        return NRNN_ERR_INVALID_ARG;
    if (d_in != 0) {
        if (d_in < 0) return NRNN_ERR_INVALID_ARG;
        if (d_in % 8 != 0 || d_in > INT32_MAX) return NRNN_ERR_UNSUPPORTED;
        if (B * T > 0 && (W_x == nullptr || (reinterpret_cast<uintptr_t>(W_x) & 15u) != 0))
            return NRNN_ERR_INVALID_ARG;
    }
    if (cu != nullptr) {
        if (B != 1) return NRNN_ERR_CU_SEQLENS;
        const int st = nrnn_validate_cu_seqlens(cu, S, T);
        if (st != NRNN_OK) return st;
    }
    return NRNN_OK;
}

size_t staging_bytes(int64_t B, int64_t T, int64_t d_in, int64_t d_h, int dtype, int K,
                     const int32_t *cu_seqlens_host, int64_t num_segments,
                     int64_t tokens_per_block) {
    if (dtype != NRNN_F32 && dtype != NRNN_BF16) return 0;
    if (B < 0 || T < 0 || d_h <= 0 || d_h % 8 != 0 || K < 0 || d_in < 0) return 0;
    if (cu_seqlens_host != nullptr &&
        (B != 1 || nrnn_validate_cu_seqlens(cu_seqlens_host, num_segments, T) != NRNN_OK))
        return 0;
    Plan pl;
    if (!make_plan(B, T, d_in, d_h, dtype, K, cu_seqlens_host, num_segments, tokens_per_block, pl))
        return 0;
    return std::max<size_t>(pl.total, ALIGN);
}

// The pipeline behind both entry points; in_host holds the blocks' inputs:
// x rows (d_in values per token, then projected with W_x) when d_in > 0,
// else preactivations (3 d_h values per token).
int forward_host(const void *in_host, int64_t d_in, const void *W_x, int dtype,
                 const float *params, int64_t B, int64_t T, int64_t d_h,
                 const int32_t *cu_seqlens_host, int64_t num_segments, int K,
                 float residual_fail, void *H_host, float *residual_host, void *staging,
                 size_t staging_bytes, int64_t tokens_per_block, void *stream_) {
    int st = validate(in_host, dtype, params, B, T, d_h, cu_seqlens_host, num_segments, K,
                      H_host, residual_host, d_in, W_x);
    if (st != NRNN_OK) return st;
    Plan pl;
    if (!make_plan(B, T, d_in, d_h, dtype, K, cu_seqlens_host, num_segments, tokens_per_block, pl))
        return NRNN_ERR_INVALID_ARG;
    if (B * T == 0) {
        *residual_host = 0.f;
        return NRNN_OK;
    }
    if (staging == nullptr || staging_bytes < pl.total ||
        (reinterpret_cast<uintptr_t>(staging) & (ALIGN - 1)) != 0)
        return NRNN_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    Lanes *ln = lanes_for_current_device();
    if (ln == nullptr) return NRNN_ERR_CUDA;

    unsigned char *base = static_cast<unsigned char *>(staging);
    float *res = reinterpret_cast<float *>(base + pl.res_off);
    uint32_t *err = reinterpret_cast<uint32_t *>(base + pl.err_off);
    int32_t *cu_dev = reinterpret_cast<int32_t *>(base + pl.cu_off);
    const size_t es = esize(dtype);
    const size_t err_word = nrnn::newton_error_offset(K);
    const size_t nblk = pl.blocks.size();

    cudaError_t e = cudaSuccess;
    if (cu_seqlens_host != nullptr) {
        // each block's segment bounds rebased to its first token
        std::vector<int32_t> rebased(static_cast<size_t>(pl.cu_ints));
        for (const Block &bk : pl.blocks)
            for (int64_t i = 0; i <= bk.ns; ++i)
                rebased[bk.cu_off + i] = cu_seqlens_host[bk.s0 + i] - static_cast<int32_t>(bk.t0);
        e = cudaMemcpyAsync(cu_dev, rebased.data(), sizeof(int32_t) * rebased.size(),
                            cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);   // `rebased` dies here
        if (e != cudaSuccess) return NRNN_ERR_CUDA;
    }

    // one block: everything on the caller's stream, no cross-stream events
    const bool single = nblk == 1;
    cudaStream_t s_in = single ? stream : ln->in, s_out = single ? stream : ln->out;
    int call_status = NRNN_OK;
    for (size_t i = 0; i < nblk && e == cudaSuccess && call_status == NRNN_OK; ++i) {
        const int s = static_cast<int>(i % NSLOT);
        const Block &bk = pl.blocks[i];
        unsigned char *X = base + pl.slots_off[s];
        unsigned char *P = X + pl.x_bytes;
        unsigned char *H = P + pl.p_bytes;
        unsigned char *ws = H + pl.h_bytes;
        // host offsets of the block: rows b0.. (full T) or tokens t0.. of row 0
        const size_t first = static_cast<size_t>(bk.b0 * T + bk.t0);
        const size_t n = static_cast<size_t>(bk.nb * bk.nt);
        const size_t in_row = static_cast<size_t>(d_in > 0 ? d_in : 3 * d_h) * es;   // per token
        const unsigned char *src = static_cast<const unsigned char *>(in_host) + first * in_row;
        unsigned char *dst = static_cast<unsigned char *>(H_host) + first * d_h * es;

        if (i >= NSLOT) e = cudaStreamWaitEvent(s_in, ln->computed[s], 0);   // input slot read
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(d_in > 0 ? X : P, src, n * in_row, cudaMemcpyHostToDevice, s_in);
        if (e == cudaSuccess && !single) e = cudaEventRecord(ln->loaded[s], s_in);
        if (e == cudaSuccess && !single) e = cudaStreamWaitEvent(stream, ln->loaded[s], 0);
        if (e == cudaSuccess && i >= NSLOT) e = cudaStreamWaitEvent(stream, ln->drained[s], 0);
        if (e != cudaSuccess) break;
        if (d_in > 0) {
            call_status = nrnn_input_projection(X, W_x, dtype, static_cast<int64_t>(n), d_in, d_h, P,
                                                base + pl.proj_off, pl.proj_bytes, stream_);
            if (call_status != NRNN_OK) break;
        }
        call_status = nrnn_newton_forward(P, dtype, params, bk.nb, bk.nt, d_h,
                                          cu_seqlens_host ? cu_dev + bk.cu_off : nullptr,
                                          cu_seqlens_host ? bk.ns : 0, K, residual_fail,
                                          NRNN_ALGO_FUSED, H, res + i, nullptr, ws, pl.ws_bytes,
                                          stream_);
        if (call_status != NRNN_OK) break;
        e = cudaMemcpyAsync(err + i, ws + err_word, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream);
        if (e == cudaSuccess && !single) e = cudaEventRecord(ln->computed[s], stream);
        if (e == cudaSuccess && !single) e = cudaStreamWaitEvent(s_out, ln->computed[s], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dst, H, n * d_h * es, cudaMemcpyDeviceToHost, s_out);
        if (e == cudaSuccess && !single) e = cudaEventRecord(ln->drained[s], s_out);
    }
    // join: the caller's stream waits for every slot's last copy out, then
    // brings the per-block residuals and error words home in one copy
    std::vector<uint32_t> tail(2 * nblk, 0u);   // nblk residual bit patterns, nblk error words
    if (!single)
        for (int s = 0; s < NSLOT && static_cast<size_t>(s) < nblk; ++s)
            if (cudaStreamWaitEvent(stream, ln->drained[s], 0) != cudaSuccess) e = cudaErrorUnknown;
    if (e == cudaSuccess && call_status == NRNN_OK)
        e = cudaMemcpyAsync(tail.data(), res, sizeof(uint32_t) * 2 * nblk, cudaMemcpyDeviceToHost, stream);
    const cudaError_t es1 = single ? cudaSuccess : cudaStreamSynchronize(ln->in);
    const cudaError_t es2 = single ? cudaSuccess : cudaStreamSynchronize(ln->out);
    const cudaError_t es3 = cudaStreamSynchronize(stream);
    if (call_status != NRNN_OK) return call_status;
    if (e != cudaSuccess || es1 != cudaSuccess || es2 != cudaSuccess || es3 != cudaSuccess)
        return NRNN_ERR_CUDA;
    float rho = 0.f;
    bool timeout = false;
    for (size_t i = 0; i < nblk; ++i) {
        timeout = timeout || tail[nblk + i] != 0u;
        float r;
        std::memcpy(&r, &tail[i], sizeof(float));
        rho = (r != r || r > rho) ? r : rho;   // NaN stays
        if (rho != rho) break;
    }
    if (rho != rho) rho = INFINITY;
    *residual_host = rho;
    if (timeout) return NRNN_ERR_TIMEOUT;
    if (!std::isfinite(rho) || rho > residual_fail) return NRNN_ERR_DIVERGED;
    return NRNN_OK;
}

}  // namespace

extern "C" {

size_t nrnn_newton_host_staging_bytes(int64_t B, int64_t T, int64_t d_h, int dtype, int K,
                                      const int32_t *cu_seqlens_host, int64_t num_segments,
                                      int64_t tokens_per_block) {
    return staging_bytes(B, T, 0, d_h, dtype, K, cu_seqlens_host, num_segments, tokens_per_block);
}

size_t nrnn_newton_x_host_staging_bytes(int64_t B, int64_t T, int64_t d_in, int64_t d_h, int dtype,
                                        int K, const int32_t *cu_seqlens_host,
                                        int64_t num_segments, int64_t tokens_per_block) {
    if (d_in <= 0 || d_in % 8 != 0) return 0;
    return staging_bytes(B, T, d_in, d_h, dtype, K, cu_seqlens_host, num_segments, tokens_per_block);
}

int nrnn_newton_forward_host(const void *preact_host, int dtype, const float *params, int64_t B,
                             int64_t T, int64_t d_h, const int32_t *cu_seqlens_host,
                             int64_t num_segments, int K, float residual_fail, void *H_host,
                             float *residual_host, void *staging, size_t staging_bytes,
                             int64_t tokens_per_block, void *stream) {
    return forward_host(preact_host, 0, nullptr, dtype, params, B, T, d_h, cu_seqlens_host,
                        num_segments, K, residual_fail, H_host, residual_host, staging,
                        staging_bytes, tokens_per_block, stream);
}

int nrnn_newton_forward_x_host(const void *x_host, const void *W_x, int dtype, const float *params,
                               int64_t B, int64_t T, int64_t d_in, int64_t d_h,
                               const int32_t *cu_seqlens_host, int64_t num_segments, int K,
                               float residual_fail, void *H_host, float *residual_host,
                               void *staging, size_t staging_bytes, int64_t tokens_per_block,
                               void *stream) {
    if (d_in <= 0) return NRNN_ERR_INVALID_ARG;
    return forward_host(x_host, d_in, W_x, dtype, params, B, T, d_h, cu_seqlens_host,
                        num_segments, K, residual_fail, H_host, residual_host, staging,
                        staging_bytes, tokens_per_block, stream);
}

}  // extern "C"

// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace nrnn {

// Runs configure(device) for the current device unless it already succeeded
// there (kernel attributes are per device).  Ordinals >= 64 configure on every
// call.
// Launch with programmatic stream serialization: the kernel may be scheduled
// while the kernel before it on the stream finishes (once that kernel's CTAs
// have all executed griddepcontrol.launch_dependents, or exited); it executes
// griddepcontrol.wait, which returns when that kernel has completed and its
// writes are visible, before touching memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

template <typename Fn>
inline cudaError_t once_per_device(std::atomic<unsigned long long> &done, Fn &&configure) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = configure(dev);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Tile of one Newton CTA: 32 hidden units (one per lane) x L time steps,
// L = NW warps x SEG steps per warp.
constexpr int TILE_U = 32;
constexpr int NEWTON_NW = 4;
constexpr int NEWTON_SEG = 16;
constexpr int NEWTON_L = NEWTON_NW * NEWTON_SEG;

struct NewtonArgs {
    const void *H_prev;           // (B, T, d_h) storage type: H^(k-1) (per-iteration) or the
                                  // initial iterate H^(0) (fused); null = zero
    void *H_next;                 // (B, T, d_h) storage type
    const float *params;          // (6, d_h)
    // the kernels that take a pack's segment-aligned chunks (k_pack_plan)
    // read the plan instead of the segment bounds; the layout of the struct
    // stays that of the other kernels (register allocation follows it)
    union {
        const int32_t *cu;        // null or (S + 1)
        const int4 *plan;         // segment-aligned chunks of the pack
    };
    int S;
    int B, T, d_h;
    int n_ut, n_chunks;           // unit tiles, time chunks
    int k_first, k_last;          // iterations this launch runs (1-based, inclusive)
    int last;                     // this launch ends with H^(K): compute the residual
    unsigned long long *slots;    // [K][n_tiles][32] packed (A, b); all-zero bits = not published
    uint32_t *ticket;             // this launch's CTA ticket counter
    uint32_t *residual_bits;      // float bits of rho (atomicMax), cleared by the caller
    uint32_t *error;              // error word (bit 0: look-back timeout, bit 1: TMA timeout)
    unsigned long long wait_ns;   // limit of every bounded wait
    int withhold_tile;            // debug: this tile never publishes its look-back slot (-1: none)
    union {
        int d_in;                 // fused projection only: input width
        int chain_stride;         // segment-aligned chunks: look-back slots per unit tile
                                  // and iteration
    };
};

struct BackwardArgs {
    const void *H;                // (B, T, d_h) trajectory the derivatives are taken at
    const void *gH;               // (B, T, d_h) dL/dH
    float *gparams;               // (6, d_h) dL/d(params), accumulated (zeroed by the caller)
    const float *params;
    union {
        const int32_t *cu;        // null or (S + 1)
        const int4 *plan;         // segment-aligned chunks of the pack, last chunks first
    };
    int S;
    int B, T, d_h;
    int n_ut, n_chunks;           // unit tiles; time chunks (segment-aligned: look-back
                                  // slots per unit tile)
    unsigned long long *slots;    // [n_tiles][32]
    uint32_t *ticket;
    uint32_t *error;
    unsigned long long wait_ns;
    void *gP;                     // (B, T, 3 d_h) dL/dP: a segment's short last chunk
                                  // stores its rows one by one
};

// tmP, tmH, tmG: load maps as for the Newton kernel (tile boxes of P, H, dL/dH);
// tmGP: 4-D store map over dL/dP as (d_h, 3, T, B) with a (32, 1, 64, 1) box.
// plan: a.plan holds a pack's segment-aligned chunks in reverse order (n_ctas
// an upper bound)
cudaError_t launch_backward(int dtype, const CUtensorMap &tmP, const CUtensorMap &tmH,
                            const CUtensorMap &tmG, const CUtensorMap &tmGP, const BackwardArgs &a,
                            int64_t n_ctas, cudaStream_t stream, bool plan = false);

// Workspace of one call: [counters | error] and [slots], cleared together at
// the start of every call (zero_bytes from the start), then (per-iteration
// variant, K > 1) one H buffer.
struct SyncLayout {
    size_t counters_off, error_off, zero_bytes;
    size_t slots_off, slots_bytes, hbuf_off, plan_off, total;
    int64_t n_tiles;        // CTAs of a Newton launch (an upper bound with a plan)
    int64_t chain_stride;   // look-back slots per (row, unit tile) and iteration
    bool plan;              // segment-aligned chunks of a pack
};

// Segment-aligned chunks of a cu_seqlens pack: chunk j of segment s covers
// rows [cu[s] + 64 j, min(cu[s] + 64 (j + 1), cu[s + 1])), so that every
// segment is a chain of its own and a pack of S segments has about S times
// as many independent chains as the time axis cut into 64-step chunks.
// plan[0].x = number of chunks; plan[1 + i] = {first row, end row of the
// segment, j, index of the chunk in segment order}; chunks in the order
// the tickets hand them out: by j, and within one j by the segment's
// number of chunks, most first (every chunk's predecessor comes earlier).
// reverse (the backward scan, whose chains run from a segment's end): by the
// number of chunks after j instead of j.  Used for packs
// of 2..PACK_PLAN_MAX_S segments, at most PACK_PLAN_MAX_CHUNKS 64-step
// chunks, and S <= n_chunks / 8 (so that at most 1/8 more chunks than the
// plain cut).
constexpr int PACK_PLAN_MAX_S = 4096;
constexpr int PACK_PLAN_MAX_CHUNKS = 8192;
bool pack_plan_applies(int64_t B, int64_t T, int64_t S);
size_t pack_plan_bytes(int64_t T, int64_t S);
cudaError_t launch_pack_plan(const int32_t *cu, int S, int n_chunks, int4 *plan, bool reverse,
                             cudaStream_t stream);

size_t newton_smem_bytes(int dtype, bool fused);

// byte offset of the error word in a Newton forward's workspace
size_t newton_error_offset(int K);

// Which look-back form launch_newton takes for these arguments (B, n_ut,
// plan are read): 0 plain, 1 early reads.
int newton_lookback_form(int dtype, bool fused, const NewtonArgs &a, bool plan = false);
// tmP over P (3 d_h, T, B), tmH over the H^(k-1) or H^(0) input, tmO over the
// H output, all with a TILE_U x NEWTON_L x 1 box
// plan: a.plan holds a pack's segment-aligned chunks (n_ctas an upper bound)
cudaError_t launch_newton(int dtype, bool fused, const CUtensorMap &tmP, const CUtensorMap &tmH,
                          const CUtensorMap &tmO, const NewtonArgs &a, int64_t n_ctas,
                          cudaStream_t stream, bool plan = false);

// fused algorithm with the input projection computed in-kernel (bf16): tmX over
// x (d_in, T, B) with a 64 x NEWTON_L x 1 box, tmW over W_x (d_in, 3 d_h) with
// a 64 x 32 box, both with the 128-byte swizzle; tmO over the H output
cudaError_t launch_newton_x(const CUtensorMap &tmX, const CUtensorMap &tmW, const CUtensorMap &tmO,
                            const NewtonArgs &a, int64_t n_ctas, cudaStream_t stream);

cudaError_t launch_residual(int dtype, const void *P, const float *params, const void *G,
                            int B, int T, int d_h, const int32_t *cu, int S,
                            uint32_t *residual_bits, cudaStream_t stream);

cudaError_t launch_picard(int dtype, const void *P, const float *params, const void *G_in,
                          void *G_out, int B, int T, int d_h, const int32_t *cu, int S,
                          cudaStream_t stream);

cudaError_t launch_decode_step(int dtype, const void *P, const float *params, const void *h_in,
                               void *h_out, int slots, int d_h, cudaStream_t stream);
cudaError_t launch_decode_step_x(int dtype, const void *x, const void *W, const float *params,
                                 const void *h_in, void *h_out, int slots, int d_in, int d_h,
                                 cudaStream_t stream);
// bf16 decode step with the projection on the tensor cores: tmX over x (d_in,
// slots) with a 64 x 64 box, tmW over W_x (d_in, 3 d_h) with a 64 x
// decode_xtc_units(slots, d_h) box, both with the 128-byte swizzle
int decode_xtc_units(int slots, int d_h);
cudaError_t launch_decode_step_xtc(const CUtensorMap &tmX, const CUtensorMap &tmW,
                                   const float *params, const void *h_in, void *h_out, int slots,
                                   int d_in, int d_h, cudaStream_t stream);
// the same in the GEMM orientation for more than one 64-slot tile: tmX over x
// (d_in, slots) with a 64 x 128 box, tmW over W_x (d_in, 3 d_h) with a 64 x 64
// box, both with the 128-byte swizzle; h_in (if given) and h_out 16-byte aligned
constexpr int DECODE_XG_MIN_SLOTS = 65;
constexpr int DECODE_XG_MIN_D_IN = 512;
cudaError_t launch_decode_step_xg(const CUtensorMap &tmX, const CUtensorMap &tmW,
                                  const float *params, const void *h_in, void *h_out, int slots,
                                  int d_in, int d_h, cudaStream_t stream);

cudaError_t launch_sequential(int dtype, const void *P, const float *params, int B, int T,
                              int d_h, const int32_t *cu, int S, void *H, cudaStream_t stream);

cudaError_t launch_head_mask(const int32_t *cu, int S, int64_t N, uint8_t *mask,
                             cudaStream_t stream);

cudaError_t launch_bounded_wait(const uint32_t *flag, uint64_t wait_ns, uint32_t *result,
                                cudaStream_t stream);

// bf16 tensor-core projection: tmA over x (d_in, rows) with a 64 x 128 box,
// tmB over W_x (d_in, n_out) with a 64 x 256 box, both bf16 with the 128-byte
// swizzle; tmP over P (n_out, rows) with a PROJ_OUT_BOX x PROJ_OUT_BOX box and
// the 64-byte swizzle.
constexpr int PROJ_TC_BOX_K = 64, PROJ_TC_BOX_M = 128, PROJ_TC_BOX_N = 256;
constexpr int PROJ_OUT_BOX = 32;
cudaError_t launch_projection_tc(const CUtensorMap &tmA, const CUtensorMap &tmB,
                                 const CUtensorMap &tmP, int64_t rows, int d_in, int n_out,
                                 cudaStream_t stream);

// fp32 split-TF32 tensor-core projection: tmA over x (d_in, rows) with a
// 32 x 128 box, tmB over W_x and tmBlo over its low part (both (d_in, n_out))
// with a 32 x projection_tf32x3_bn(n_out) box, all fp32 with the 128-byte
// swizzle; tmP over P (n_out, rows) with a PROJ_OUT_BOX x PROJ_OUT_BOX box and
// the 128-byte swizzle.
constexpr int PROJ_T3_BOX_K = 32, PROJ_T3_BOX_M = 128;
int projection_tf32x3_bn(int n_out);
cudaError_t launch_projection_tf32x3(const CUtensorMap &tmA, const CUtensorMap &tmB,
                                     const CUtensorMap &tmBlo, const CUtensorMap &tmP,
                                     int64_t rows, int d_in, int n_out, cudaStream_t stream);
// lo[i] = w[i] - (w[i] with its low 13 mantissa bits cleared), n fp32 values
cudaError_t launch_split_low(const void *w, void *lo, int64_t n, cudaStream_t stream);

}  // namespace nrnn

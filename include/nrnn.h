/*
 * nrnn.h -- C ABI of the GB300 parallel-Newton forward for a diagonal-mix GRU.
 *
 * The method (pararnn-torch pages: FAQs "Does parallel Newton match sequential
 * unroll?" and "What is critical Newton depth (K*)?", numerics contract
 * "Invariant", "Two thresholds" and "Four echelons / 1. Runtime",
 * shapes_layout "cu_seqlens"):
 *
 *   cell    z = sig(P_z + a_z h + b_z),  r = sig(P_r + a_r h + b_r),
 *           c = tanh(P_c + a_c (r h) + b_c),  f(h, P) = (1 - z) h + z c
 *           with P = W_x x the input projection, gate blocks [z | r | c];
 *   Newton  H^(0) = 0; for k = 1..K: at the shifted trajectory evaluate
 *           F_t = H_t - f(H_{t-1}, P_t) and J_t = df/dh(H_{t-1}, P_t), solve
 *           delta_t = J_t delta_{t-1} - F_t by a parallel scan over t, and set
 *           H <- H + delta.  At t = 0 and at every segment head of a ragged
 *           pack J = 0 and the shifted state is 0 (each segment starts from h=0);
 *   gate    rho = max |F(H^(K))| (NaN counts as +inf); rho > residual_fail is
 *           the divergence signal (NewtonDivergenceError on the pages).
 *
 * Conventions shared by every entry point
 *   - Every buffer is caller-owned.  No entry point of the computation
 *     allocates device memory.  Two exceptions, both outside it:
 *     nrnn_probe_xu_rates (a throughput measurement) allocates and frees a
 *     small buffer, and nrnn_newton_forward_host creates two streams and a
 *     few events per device on its first call and keeps them.
 *   - Device buffers are contiguous, row-major, 16-byte aligned.
 *   - dtype selects the storage type of preact, x, W_x and H: NRNN_F32 or
 *     NRNN_BF16 (bfloat16 storage; all arithmetic inside the kernels is fp32).
 *     Parameters are always fp32.
 *   - params: device, fp32, shape (6, d_h): rows a_z, a_r, a_c, b_z, b_r, b_c.
 *   - stream: a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream unless stated otherwise.  The Newton
 *     kernels are launched with programmatic stream serialization and signal
 *     their dependents early: a kernel the caller launches after them with
 *     that launch attribute must execute griddepcontrol.wait (as programmatic
 *     dependent launch requires) before it reads their outputs.  Ordinary
 *     launches, copies and events after a call are ordered as usual.
 *   - cu_seqlens (nullable): device int32 array of num_segments + 1 offsets
 *     for a ragged pack; then B must be 1 and T is the packed length N.  The
 *     offsets must satisfy cu[0] = 0, cu[i] <= cu[i+1], cu[S] = N; check
 *     them with nrnn_validate_cu_seqlens on a host copy before the call (the
 *     kernels only read them and stay in bounds for any values, but give
 *     meaningless results for invalid ones).  Empty segments are allowed.
 *   - Alignment: d_h must be a multiple of 8 (TMA tile rows are 16-byte
 *     aligned); other d_h return NRNN_ERR_UNSUPPORTED.
 *   - Return value: an nrnn_status (0 = success, negative = error).  Errors
 *     detected before any launch leave every output untouched.
 */
#ifndef NRNN_H
#define NRNN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NRNN_OK = 0,
    NRNN_ERR_INVALID_ARG = -1,  /* null pointer, negative size, bad dtype, misaligned */
    NRNN_ERR_CU_SEQLENS = -2,   /* cu_seqlens violates the rules above */
    NRNN_ERR_UNSUPPORTED = -3,  /* valid request the library does not handle (d_h % 8) */
    NRNN_ERR_CUDA = -4,         /* a CUDA runtime/driver call or a launch failed */
    NRNN_ERR_DIVERGED = -5,     /* rho > residual_fail, or rho is NaN/inf */
    NRNN_ERR_TIMEOUT = -6,      /* a bounded device wait gave up (result invalid) */
    NRNN_ERR_WORKSPACE = -7     /* workspace null or smaller than required */
} nrnn_status;

typedef enum { NRNN_F32 = 0, NRNN_BF16 = 1 } nrnn_dtype;

/* Newton implementation.  Both compute the same iteration in the same order
 * of operations per element; they differ in HBM traffic.
 *   NRNN_ALGO_PER_ITER: one fused cell+Jacobian+scan kernel per iteration;
 *                       H goes through HBM between iterations.
 *   NRNN_ALGO_FUSED:    one kernel runs all K iterations per T-chunk in
 *                       on-chip memory; P is read once and H written once.
 *   NRNN_ALGO_AUTO:     the library picks (currently NRNN_ALGO_FUSED).     */
typedef enum { NRNN_ALGO_AUTO = 0, NRNN_ALGO_PER_ITER = 1, NRNN_ALGO_FUSED = 2 } nrnn_algo;

/* Human-readable name of a status code (static storage, never NULL). */
const char *nrnn_status_string(int status);

/* ABI version: major * 10000 + minor * 100 + patch. */
int nrnn_version(void);

/*
 * Rules of cu_seqlens (shapes_layout page, "cu_seqlens": batch 1, length N,
 * S+1 offsets; validate_cu_seqlens): cu_host has num_segments + 1 >= 2
 * entries, cu[0] = 0, non-decreasing, cu[num_segments] = N.  Host pointer;
 * no CUDA call.  Returns NRNN_OK or NRNN_ERR_CU_SEQLENS (NRNN_ERR_INVALID_ARG
 * for a null pointer or negative sizes).
 */
int nrnn_validate_cu_seqlens(const int32_t *cu_host, int64_t num_segments, int64_t N);

/*
 * Workspace bytes nrnn_newton_forward needs for this shape, K and algo
 * (NRNN_ALGO_PER_ITER also holds one H buffer of B*T*d_h elements).
 * Returns 0 for invalid arguments.
 */
size_t nrnn_newton_workspace_bytes(int64_t B, int64_t T, int64_t d_h, int dtype, int K,
                                   int algo);

/*
 * Workspace bytes for a forward over a cu_seqlens pack (x of shape (1, N, d))
 * of num_segments segments (shapes_layout, "cu_seqlens").  With a workspace of
 * at least this size nrnn_newton_forward cuts each segment into chunks of its
 * own instead of cutting the pack's time axis, which keeps many more
 * look-back chains in flight (one per segment): for packs of 2 to 4096
 * segments, N <= 524288 and num_segments <= ceil(N / 64) / 8; other packs,
 * and a workspace sized by nrnn_newton_workspace_bytes, take the time-axis
 * chunks.  Results agree to rounding either way (the look-back composes in
 * another grouping).  Returns 0 for invalid arguments.
 */
size_t nrnn_newton_workspace_bytes_pack(int64_t N, int64_t d_h, int dtype, int K, int algo,
                                        int64_t num_segments);

/*
 * Parallel Newton forward (numerics contract, "Invariant"; FAQs "How many
 * Newton iterations should I use?": a fixed K).
 *
 *   preact        device, (B, T, 3 d_h) of dtype, gate blocks [z | r | c]
 *   params        device, fp32 (6, d_h)
 *   B, T, d_h     sizes; B, T >= 0, d_h > 0 and a multiple of 8
 *   cu_seqlens    device int32 (num_segments + 1) or NULL (rectangular batch)
 *   K             Newton iterations, 0 <= K <= 64 (K = 0: H = 0)
 *   residual_fail divergence threshold (the pages' default is 1.0)
 *   algo          nrnn_algo
 *   H_out         device, (B, T, d_h) of dtype: H^(K); 16-byte aligned, must
 *                 not overlap preact (NRNN_ERR_INVALID_ARG)
 *   residual_dev  device, 1 float: rho = max|F(H^(K))|, +inf if any F is NaN
 *   residual_host NULL: fully asynchronous, no gate, no timeout report.
 *                 Non-NULL: the call synchronises the stream, stores rho
 *                 there, and returns NRNN_ERR_TIMEOUT if a bounded device
 *                 wait gave up, else NRNN_ERR_DIVERGED if rho > residual_fail
 *                 or rho is not finite (H_out is written either way).
 *   workspace     device, ws_bytes >= nrnn_newton_workspace_bytes(...)
 *                 (a pack: nrnn_newton_workspace_bytes_pack(...) lets the
 *                 kernels cut each segment into chunks of its own);
 *                 256-byte aligned; its contents need no initialisation and
 *                 are scratch after the call.  Calls that share a
 *                 workspace must not overlap on the GPU.
 *   stream        cudaStream_t
 */
int nrnn_newton_forward(const void *preact, int dtype, const float *params, int64_t B,
                        int64_t T, int64_t d_h, const int32_t *cu_seqlens,
                        int64_t num_segments, int K, float residual_fail, int algo,
                        void *H_out, float *residual_dev, float *residual_host,
                        void *workspace, size_t ws_bytes, void *stream);

/*
 * Parallel Newton forward started from a given iterate H^(0) = H_init instead
 * of 0 (a warm start, e.g. from nrnn_picard; FAQs "How many Newton
 * iterations should I use?": "try Picard warm-start").  Arguments as
 * nrnn_newton_forward; H_init: device, (B, T, d_h) of dtype, 16-byte aligned,
 * must not overlap H_out (NRNN_ERR_INVALID_ARG), or NULL for H^(0) = 0.
 * With K = 0 the call returns H_out = H_init and rho = max|F(H_init)|.
 * The fused algorithm needs L*32*elem bytes more shared memory per CTA for
 * the initial tile; the workspace size does not change.
 */
int nrnn_newton_forward_init(const void *preact, int dtype, const float *params, int64_t B,
                             int64_t T, int64_t d_h, const int32_t *cu_seqlens,
                             int64_t num_segments, const void *H_init, int K,
                             float residual_fail, int algo, void *H_out, float *residual_dev,
                             float *residual_host, void *workspace, size_t ws_bytes,
                             void *stream);

/*
 * Newton forward with the input projection fused in (bf16 only): each CTA
 * computes its tile of P = x W_x^T on the tensor cores in on-chip memory and
 * runs the fused Newton iterations on it, so P never goes through HBM.  The
 * tile's fp32 accumulator is rounded to bf16 first, so the result equals
 * nrnn_input_projection followed by nrnn_newton_forward (NRNN_ALGO_FUSED)
 * up to the accumulation order of the projection.
 *   x      device, (B, T, d_in) bf16;  W_x device, (3 d_h, d_in) bf16
 *   d_in   multiple of 8;  K >= 1
 *   other arguments as nrnn_newton_forward; workspace size as for
 *   NRNN_ALGO_FUSED.  NRNN_F32 returns NRNN_ERR_UNSUPPORTED.
 */
int nrnn_newton_forward_x(const void *x, const void *W_x, int dtype, const float *params,
                          int64_t B, int64_t T, int64_t d_in, int64_t d_h,
                          const int32_t *cu_seqlens, int64_t num_segments, int K,
                          float residual_fail, void *H_out, float *residual_dev,
                          float *residual_host, void *workspace, size_t ws_bytes, void *stream);

/*
 * Backward (adjoint) pass for training (shapes_layout page: "train
 * forward+backward surface"; no equations on the pages, plainest reading):
 * with gH = dL/dH at the trajectory H (e.g. the Newton result),
 *   lambda_t = gH_t + J_{t+1} lambda_{t+1} (0 after the end; J = 0 at segment
 *   heads), dL/dP_{t,g} = lambda_t df/dP_g,
 *   dL/d(a_g, b_g) = sum over (b, t) of lambda_t df/d(a_g, b_g),
 * derivatives taken at (H_{t-1}, P_t) (H_{-1} = 0 at heads).  Solved by the
 * same chunked decoupled look-back scan as the forward, in reverse time.
 *   H, gH     device, (B, T, d_h) of dtype, 16-byte aligned
 *   gP        device, (B, T, 3 d_h) of dtype, 16-byte aligned (out; written by
 *             TMA stores of whole gate blocks)
 *   gparams   device, fp32 (6, d_h) (out; overwritten)
 *   workspace >= nrnn_newton_workspace_bytes(B, T, d_h, dtype, 1, NRNN_ALGO_FUSED); for a
 *              pack, one of nrnn_newton_workspace_bytes_pack(T, d_h, dtype, 1,
 *              NRNN_ALGO_FUSED, num_segments) bytes runs on segment-aligned
 *              chunks as the forward does (in reverse order)
 * Results are accumulated with atomics: within float rounding, not bitwise
 * reproducible.
 */
int nrnn_newton_backward(const void *preact, int dtype, const float *params, int64_t B,
                         int64_t T, int64_t d_h, const int32_t *cu_seqlens, int64_t num_segments,
                         const void *H, const void *gH, void *gP, float *gparams,
                         void *workspace, size_t ws_bytes, void *stream);

/*
 * Picard warm start (FAQs "How many Newton iterations should I use?":
 * "try Picard warm-start (picard_iters)"; read as fixed-point sweeps):
 * from G = 0, each sweep sets G_t = f(G_{t-1}, P_t) for all t at once from
 * the previous sweep (shifted state 0 at t = 0 and at segment heads).  Sweep
 * s makes steps 1..s exact.  One elementwise launch per sweep, no scan.  The
 * cell runs in the storage type's formulation (bf16: tanh.approx, as in the
 * Newton kernels).
 *   sweeps  >= 0 (0: H_out = 0)
 *   H_out   device, (B, T, d_h) of dtype, 16-byte aligned: the last sweep
 *   H_tmp   device scratch of the same size and alignment, needed when
 *           sweeps >= 2; must not overlap H_out
 * Neither may overlap preact (NRNN_ERR_INVALID_ARG).
 */
int nrnn_picard(const void *preact, int dtype, const float *params, int64_t B, int64_t T,
                int64_t d_h, const int32_t *cu_seqlens, int64_t num_segments, int sweeps,
                void *H_out, void *H_tmp, void *stream);

/*
 * Sequential forward on the GPU (sequential_apply on the pages: "eval()"
 * runs the sequential step): h_t = f(h_{t-1}, P_t) from h = 0 for each row,
 * or for each segment of a pack; one thread per (row or segment, unit).
 *   preact (B, T, 3 d_h) dtype -> H_out (B, T, d_h) dtype.  No workspace.
 */
int nrnn_sequential_forward(const void *preact, int dtype, const float *params, int64_t B,
                            int64_t T, int64_t d_h, const int32_t *cu_seqlens,
                            int64_t num_segments, void *H_out, void *stream);

/*
 * Residual of a given trajectory: rho = max |G_t - f(G_{t-1}, P_t)| over all
 * (b, t, j), with G_{-1} = 0 at t = 0 and at segment heads (the residual gate
 * of the numerics contract, "Two thresholds").  G (B, T, d_h) dtype.
 * residual_dev: device, 1 float (overwritten).
 */
int nrnn_residual(const void *preact, int dtype, const float *params, int64_t B, int64_t T,
                  int64_t d_h, const int32_t *cu_seqlens, int64_t num_segments,
                  const void *G, float *residual_dev, void *stream);

/*
 * Decode step (FAQs "How do I pass recurrent state between decode steps?":
 * a fixed-size carry (slots, d_h); decode_step(..., out=)): one T = 1 step
 * h_out = f(h_in, P) per slot.
 *   preact  device, (slots, 3 d_h) of dtype, gate blocks [z | r | c]
 *   h_in    device, (slots, d_h) of dtype, or NULL for the zero state
 *   h_out   device, (slots, d_h) of dtype; may be h_in (in place), must not
 *           overlap preact
 * No alignment or d_h restriction; with d_h a multiple of 4 (fp32) or 8
 * (bf16) and preact, params, h_in, h_out 16-byte aligned the step runs on
 * 16-byte vectors, else one element per thread (same results).
 */
int nrnn_decode_step(const void *preact, int dtype, const float *params, int64_t slots,
                     int64_t d_h, const void *h_in, void *h_out, void *stream);

/*
 * Decode step with the input projection fused in (FAQs: "decode_wx +
 * decode_step"): P_s = W_x x_s (fp32 accumulation on the CUDA cores, rounded
 * to dtype as the stored preactivation would be), then h_out = f(h_in, P).
 * bf16: the product on the tensor cores with the step in the epilogue; up to
 * 64 slots, 64 slots by 8 or 32 units per CTA, so W_x streams from HBM once
 * per 64 slots; above that, when d_in >= 512, d_h is a multiple of 8 and
 * params, h_in and h_out are 16-byte aligned, a GEMM of 128-slot by 64-unit
 * tiles on one persistent CTA per SM.  fp32: a batched matrix-vector product
 * on the CUDA cores (each W_x row read once per group of 8 slots).  For
 * hundreds of slots with fp32 or a short d_in, nrnn_input_projection into a
 * (slots, 3 d_h) buffer followed by nrnn_decode_step is faster (the Python
 * binding switches there above 64 slots).
 *   x       device, (slots, d_in) of dtype, 16-byte aligned
 *   W_x     device, (3 d_h, d_in) of dtype, 16-byte aligned
 *   h_in    device (slots, d_h) or NULL;  h_out device (slots, d_h), may be h_in
 *   slots <= 524280; d_in a multiple of 8 (else NRNN_ERR_UNSUPPORTED).
 */
int nrnn_decode_step_x(const void *x, const void *W_x, int dtype, const float *params,
                       int64_t slots, int64_t d_in, int64_t d_h, const void *h_in, void *h_out,
                       void *stream);

/*
 * Input projection P = x W_x^T (shapes_layout page: "W_x" reads x of layout
 * (B, T, d_in)); x (rows, d_in), W_x (3 d_h, d_in), preact (rows, 3 d_h), all
 * of dtype, fp32 accumulation.  NRNN_F32 keeps fp32 accuracy (no TF32
 * rounding of the operands: three TF32 products of a high/low split of each
 * operand); NRNN_BF16 uses the bf16 tensor-core path and rounds the fp32
 * accumulator to bf16.  d_in and d_h must be multiples of 8 and rows < 2^31
 * (else NRNN_ERR_UNSUPPORTED); x, W_x and preact 16-byte aligned (else
 * NRNN_ERR_INVALID_ARG).
 *   workspace  device, caller-owned, 256-byte aligned, at least
 *              nrnn_input_projection_workspace_bytes(dtype, d_in, d_h) bytes
 *              (NRNN_F32: the low part of W_x, written by this call; may be
 *              NULL when that size is 0); too small or misaligned returns
 *              NRNN_ERR_WORKSPACE
 */
size_t nrnn_input_projection_workspace_bytes(int dtype, int64_t d_in, int64_t d_h);
int nrnn_input_projection(const void *x, const void *W_x, int dtype, int64_t rows,
                          int64_t d_in, int64_t d_h, void *preact, void *workspace,
                          size_t ws_bytes, void *stream);

/*
 * Debug export of the segment-head mask the Newton kernels use
 * (shapes_layout page: "Segment heads use J=0 on the scan"): mask_dev[t] = 1
 * if t = 0 or t = cu[i] < cu[i+1] for some i, else 0, for t in [0, N).
 * Uses the same device routine as the Newton kernels.  mask_dev: device, N bytes.
 */
int nrnn_debug_head_mask(const int32_t *cu_seqlens, int64_t num_segments, int64_t N,
                         uint8_t *mask_dev, void *stream);

/*
 * Debug check of the bounded device wait used by the scan's look-back: one
 * thread waits for *flag_dev to become nonzero for at most wait_ns
 * nanoseconds.  *result_dev (device, 1 uint32) receives 1 if the flag was
 * seen, 2 if the wait gave up.  Never hangs: a flag nobody sets returns 2.
 */
int nrnn_debug_bounded_wait(const uint32_t *flag_dev, uint64_t wait_ns, uint32_t *result_dev,
                            void *stream);

/*
 * Newton forward on host buffers, with the host-device copies overlapped
 * with the computation (the pages run the forward on device tensors only;
 * this is the library's end-to-end entry point for data that lives on the
 * host).  The problem is cut into blocks that need nothing from one another
 * -- groups of batch rows, or for a pack groups of whole segments -- of about
 * tokens_per_block tokens each (0: about 16 blocks).  Each block is copied
 * in on a library stream, run through nrnn_newton_forward (fused algorithm)
 * on `stream`, and copied out on a second library stream, on one of three
 * slots of `staging`, so that one block's copies overlap another's kernels.
 * The library streams and their events are created on the calling host
 * thread's first call on a device and kept for that thread's lifetime.
 *   preact_host    host, (B, T, 3 d_h) of dtype; page-locked memory lets the
 *                  copies run asynchronously (pageable memory works, slower)
 *   params         device, (6, d_h) fp32, as for nrnn_newton_forward
 *   cu_seqlens_host host, (num_segments + 1) int32 or NULL; validated as by
 *                  nrnn_validate_cu_seqlens; B must be 1
 *   H_host         host, (B, T, d_h) of dtype: H^(K)
 *   residual_host  host, 1 float (required): rho = max over blocks of
 *                  max|F(H^(K))|, +inf if any F is NaN
 *   staging        device, staging_bytes >= nrnn_newton_host_staging_bytes(
 *                  same shape, cu_seqlens_host, tokens_per_block); 256-byte
 *                  aligned; scratch
 * Synchronous: returns once H_host and *residual_host hold the result.
 * Returns NRNN_OK, NRNN_ERR_TIMEOUT (a bounded device wait gave up),
 * NRNN_ERR_DIVERGED (rho > residual_fail or not finite; H_host written),
 * NRNN_ERR_WORKSPACE (staging too small or misaligned), NRNN_ERR_CU_SEQLENS,
 * NRNN_ERR_UNSUPPORTED, NRNN_ERR_INVALID_ARG or NRNN_ERR_CUDA.  Results equal
 * nrnn_newton_forward up to the composition order of the look-back (a pack's
 * blocks start their time chunks at their own first token).
 */
size_t nrnn_newton_host_staging_bytes(int64_t B, int64_t T, int64_t d_h, int dtype, int K,
                                      const int32_t *cu_seqlens_host, int64_t num_segments,
                                      int64_t tokens_per_block);
int nrnn_newton_forward_host(const void *preact_host, int dtype, const float *params, int64_t B,
                             int64_t T, int64_t d_h, const int32_t *cu_seqlens_host,
                             int64_t num_segments, int K, float residual_fail, void *H_host,
                             float *residual_host, void *staging, size_t staging_bytes,
                             int64_t tokens_per_block, void *stream);

/*
 * The same host-buffer forward from the input sequence x instead of its
 * preactivations: the cell's input weights W_x stay on the device, each
 * block's rows of x are copied in, projected by nrnn_input_projection into
 * the block's preactivations on `stream`, and run through the forward as
 * above.  d_in values per token cross the host link instead of 3 d_h.
 *   x_host     host, (B, T, d_in) of dtype (page-locked for asynchronous copies)
 *   W_x        device, (3 d_h, d_in) of dtype, 16-byte aligned
 *   d_in       > 0 and a multiple of 8 (else NRNN_ERR_INVALID_ARG /
 *              NRNN_ERR_UNSUPPORTED)
 *   staging    device, staging_bytes >= nrnn_newton_x_host_staging_bytes(same
 *              shape, cu_seqlens_host, tokens_per_block); 256-byte aligned;
 *              it also holds the projection's workspace
 * Other arguments, synchronisation and return codes as for
 * nrnn_newton_forward_host.  Results equal nrnn_input_projection followed by
 * nrnn_newton_forward up to the look-back's composition order.
 * nrnn_newton_x_host_staging_bytes returns 0 for an invalid shape.
 */
size_t nrnn_newton_x_host_staging_bytes(int64_t B, int64_t T, int64_t d_in, int64_t d_h, int dtype,
                                        int K, const int32_t *cu_seqlens_host,
                                        int64_t num_segments, int64_t tokens_per_block);
int nrnn_newton_forward_x_host(const void *x_host, const void *W_x, int dtype, const float *params,
                               int64_t B, int64_t T, int64_t d_in, int64_t d_h,
                               const int32_t *cu_seqlens_host, int64_t num_segments, int K,
                               float residual_fail, void *H_host, float *residual_host,
                               void *staging, size_t staging_bytes, int64_t tokens_per_block,
                               void *stream);

/*
 * Size of the device scratch array that nrnn_newton_forward_noalloc uses
 * (64 MiB on every GPU where the library is used, held until process exit).
 */
#define NRNN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * Newton forward that allocates nothing and takes no workspace.  The pages
 * describe no counterpart of this entry point; it exists for callers that
 * cannot allocate device memory -- e.g. a plugin inside a host framework that
 * owns all device allocations and offers it no pool, or a latency-bounded
 * loop that must not call cudaMalloc/cudaFree (they can synchronise the
 * device) -- and so cannot pass the workspace nrnn_newton_forward needs.
 *
 * Same arguments and results as nrnn_newton_forward with algo =
 * NRNN_ALGO_FUSED, minus the workspace: the look-back scratch lives in one
 * library-owned device array of NRNN_NOALLOC_SCRATCH_BYTES per GPU.
 *   - Requests whose workspace (nrnn_newton_workspace_bytes with
 *     NRNN_ALGO_FUSED) exceeds NRNN_NOALLOC_SCRATCH_BYTES return
 *     NRNN_ERR_WORKSPACE before any CUDA call.
 *   - The first call on a device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress) and keeps it for the
 *     device's context; make that first call before any stream capture on
 *     the device.  After cudaDeviceReset the next call looks the address up
 *     again (again: outside any stream capture).
 *   - Every call on a device shares the one array; each call re-initialises
 *     the parts that must start cleared.  Calls that overlap on the GPU
 *     (different streams, no ordering between them) race on it: serialise them.
 * Calls no cudaMalloc, cudaFree or allocating library routine.
 */
int nrnn_newton_forward_noalloc(const void *preact, int dtype, const float *params, int64_t B,
                                int64_t T, int64_t d_h, const int32_t *cu_seqlens,
                                int64_t num_segments, int K, float residual_fail, void *H_out,
                                float *residual_dev, float *residual_host, void *stream);

/*
 * Debug: from the next call on, the Newton tile with index `tile` (tile =
 * (b * ceil(d_h / 32) + unit_tile) * ceil(T / 64) + chunk; on the
 * segment-aligned chunks of a pack unit_tile * (ceil(T / 64) + num_segments)
 * + the chunk's index in segment order) never publishes its look-back slot,
 * so that the later chunks of its column wait for it until their bounded
 * wait gives up.  The call then still terminates and,
 * with residual_host non-NULL, returns NRNN_ERR_TIMEOUT (H_out is invalid).
 * tile < 0 switches it off (the default).  Process-wide; returns the
 * previous value.  For testing the failure path only.
 */
int64_t nrnn_debug_withhold_publish(int64_t tile);

/*
 * Debug: the look-back form nrnn_newton_forward's kernels take on the current
 * device for a problem of this shape (algo as for nrnn_newton_forward):
 *   0  plain: after the CTA barrier warp 0 reads up to 4 predecessor slots
 *      per round
 *   1  early: warp 0 reads the two nearest predecessor slots before the CTA
 *      barrier (at most 4 chunks of each column resident at once)
 * or NRNN_ERR_INVALID_ARG.  Host only; launches nothing.
 */
int nrnn_debug_lookback_form(int64_t B, int64_t T, int64_t d_h, int dtype, int algo);

/*
 * Debug: writes the segment-aligned chunk plan that nrnn_newton_forward
 * (reverse = 0) or nrnn_newton_backward (reverse != 0) uses for a pack (see
 * nrnn_newton_workspace_bytes_pack) into plan, device, at least
 * (2 + ceil(N / 64) + num_segments) x 4 int32, 16-byte aligned: plan[0] =
 * number of chunks n, then n entries {first row, end row of the segment,
 * chunk index j within the segment, index of the chunk in segment order}, in
 * the order the kernels take them (by j, or for reverse by the number of
 * chunks of the segment after j; within one level by the segment's number of
 * chunks, most first).  cu_seqlens: device, validated.  Returns
 * NRNN_ERR_INVALID_ARG for packs that take the time-axis chunks.
 */
int nrnn_debug_pack_plan(const int32_t *cu_seqlens, int64_t num_segments, int64_t N, int reverse,
                         void *plan, void *stream);

/*
 * Upper limit, in nanoseconds, of every bounded device wait that later calls
 * launch (default 2e9 = 2 s).  Process-wide; returns the previous value.
 */
uint64_t nrnn_set_wait_limit_ns(uint64_t ns);

/*
 * Measures the special-function unit throughput of the current device, the
 * denominator of the fused Newton kernel's ALU roofline (each cell evaluation
 * issues three ex2.approx and two rcp.approx for fp32 storage, three
 * tanh.approx for bf16 storage; the pages give no hardware figure for it, so
 * the library measures it).  No counterpart in the pages.  One CTA per SM runs
 * independent chains of each instruction and times itself with the SM cycle
 * counter.
 *   ex2_per_clk, rcp_per_clk, tanh_per_clk
 *                 host, 1 float each: median over SMs of results per SM
 *                 clock cycle
 *   stream        cudaStream_t to run on (NULL: legacy stream); the call
 *                 synchronises it
 * Allocates and frees a small device buffer; takes a few milliseconds.
 * Returns NRNN_OK, NRNN_ERR_INVALID_ARG (null output) or NRNN_ERR_CUDA.
 */
int nrnn_probe_xu_rates(float *ex2_per_clk, float *rcp_per_clk, float *tanh_per_clk,
                        void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NRNN_H */

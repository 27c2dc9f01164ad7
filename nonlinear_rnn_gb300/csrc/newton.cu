// Parallel Newton forward of the diagonal-mix GRU (sm_103a).
//
// One CTA owns a tile of 32 hidden units (one per lane) x L = 64 time steps
// of one batch row (4 warps; 8 CTAs fill an SM's registers); warp w owns rows
// [16 w, 16 w + 16), which each thread runs as two halves of 8 rows in the
// lanes of packed f32x2 arithmetic.  Per Newton iteration
//   1. each thread evaluates the cell at the shifted trajectory for its 16
//      steps, F_t = H_t - f(H_{t-1}, P_t) and J_t = df/dh (J = 0 and shifted
//      state 0 at segment heads; pararnn-torch shapes_layout, "cu_seqlens"),
//      and composes the affine maps delta -> J_t delta - F_t serially;
//   2. the warp aggregates meet in shared memory (one barrier): warp 0 hands
//      every warp its exclusive prefix, publishes the chunk aggregate and
//      completes it by a decoupled look-back over earlier chunks (one lane per
//      unit, 4 predecessors read per round);
//   3. after a second barrier every thread applies the carry:
//      delta_t = J_t delta_{t-1} - F_t, H <- H + delta.
// Each warp advances the shifted state at its first row itself
// (H^(k)_{r0-1} = H^(k-1)_{r0-1} + carry into the warp), so iterations need no
// other exchange.  The fused variant runs all K iterations on the tile kept
// in shared memory (P) and registers (H): P is read once and H written once.
// The per-iteration variant runs one iteration per launch, streaming H^(k-1)
// in and H^(k) out.  The launch that produces H^(K) evaluates F(H^(K)) once
// more for the residual gate max|F| (numerics contract, "Two thresholds").
//
// Tiles of P (three gate blocks) and of H^(k-1) are staged in shared memory
// by TMA (cp.async.bulk.tensor, completion on an mbarrier).  CTAs take tiles
// from an atomic ticket in chunk-major order (for a pack cut into
// segment-aligned chunks: level by level from the chunk plan), so every CTA
// whose result a CTA waits for has already started: the look-back cannot
// deadlock.  Every wait is bounded by the caller's limit and reports a
// timeout in the error word instead of hanging.
#include "nrnn_device.cuh"
#include "nrnn_internal.h"
#include "tcgen05.cuh"

namespace nrnn {

namespace {

constexpr int NW = NEWTON_NW;
constexpr int SEG = NEWTON_SEG;
constexpr int L = NEWTON_L;
constexpr int U = TILE_U;
// early look-back reads when at most this many chunks per column are resident
constexpr int EARLY_LOOKBACK_CHUNKS = 4;

// fused-projection prologue (XPROJ): bf16 operands, 32-wide K slices (64-byte
// rows, 64-byte swizzle), two stages in a ring that the P' tile aliases
constexpr int XP_BK = 32;
constexpr int XP_W_BOX_BYTES = 32 * XP_BK * 2;               // 32 W_x rows of one gate
// the A operand holds the 96 W_x rows of the tile's three gates; the MMA's
// M = 128 reads 32 rows more, which run on into the x tile that follows (their
// TMEM lanes 96..127 are never read), so a stage needs no room for them
constexpr int XP_A_BYTES = 3 * XP_W_BOX_BYTES;               // 96 W_x rows
constexpr int XP_X_BYTES = L * XP_BK * 2;                    // 64 x rows (time steps)
constexpr int XP_STAGE_BYTES = XP_A_BYTES + XP_X_BYTES;      // 10 KiB
// the ring: two stages, or the P' tile written over them, whichever is larger
// (24 KiB: 8 CTAs per SM, as registers allow)
constexpr int XP_RING_BYTES = 2 * XP_STAGE_BYTES > 3 * L * U * 4 ? 2 * XP_STAGE_BYTES : 3 * L * U * 4;
constexpr uint32_t XP_TMEM_COLS = L;                         // one fp32 column per time step
constexpr uint32_t XP_IDESC = idesc_kmajor<false>(128, L);
// Each thread's SEG rows are split into two halves of HALF rows that run side
// by side as the two lanes of f32x2 values: element j of a pair array holds
// rows (r0 + j, r0 + HALF + j).  The fused kernel keeps its pre-scaled tile in
// shared memory in the same order, [3][NW][HALF][U] float2, so that one 64-bit
// load per gate fetches both rows.
constexpr int HALF = SEG / 2;

// float2 index of rows (r0 + j, r0 + HALF + j) of gate g, lane `lane`, in the
// pair-ordered tile
__device__ __forceinline__ int pf2_index(int g, int warp, int j, int lane) {
    return (g * NW * HALF + warp * HALF + j) * U + lane;
}

// Affine pairs (J_t, g_t) of this warp's SEG rows at the shifted iterate,
// with g_t = f(h~_t) - J_t h~_t, so that the new iterate solves
// H^(k)_t = J_t H^(k)_{t-1} + g_t: the Newton step delta_t = J_t delta_{t-1} - F_t
// written for delta_t = H^(k)_t - H^(k-1)_t.  Composed per half into
// (A2, B2); the warp aggregate (A, Bv) composes the second half after the
// first; (A_lo, B_lo) is the first half's map, from which the second half's
// starting state follows.  On entry G holds H^(k-1), on return g_t.
// SCALED: Pv is the pair-ordered fp32 tile of pre-scaled arguments; otherwise
// raw [3][L][U] preactivations of type TS.  GENERAL handles segment heads
// (J = 0, shifted state 0) and rows past T (identity).  ZERO: the first
// iteration from H^(0) = 0, where every shifted state is 0 and g = f(0).
template <typename TS, bool SCALED, bool GENERAL, bool ZERO = false>
__device__ __forceinline__ void warp_pairs(const void *Pv, int warp, int lane,
                                           float2 (&G)[HALF], float hb, uint32_t hm, int nvalid,
                                           const typename CellOf<TS>::type::Params &prm,
                                           float2 (&J2)[HALF], float &A_lo, float &B_lo, float &A,
                                           float &Bv) {
    using Cell = typename CellOf<TS>::type;
    const int r0 = warp * SEG;
    float2 A2 = splat2(1.f), B2 = splat2(0.f);
    float2 prev = make_float2(hb, G[HALF - 1].x);   // H^(k-1) at rows r0 - 1, r0 + HALF - 1
#pragma unroll
    for (int j = 0; j < HALF; ++j) {
        float2 sz, sr, sc;
        if (SCALED) {
            const float2 *P = static_cast<const float2 *>(Pv);
            sz = P[pf2_index(0, warp, j, lane)];
            sr = P[pf2_index(1, warp, j, lane)];
            sc = P[pf2_index(2, warp, j, lane)];
        } else {
            const TS *P = static_cast<const TS *>(Pv);
            const int lo = (r0 + j) * U + lane, hi = lo + HALF * U;
            Cell::scale(make_float2(to_f32(P[lo]), to_f32(P[hi])),
                        make_float2(to_f32(P[L * U + lo]), to_f32(P[L * U + hi])),
                        make_float2(to_f32(P[2 * L * U + lo]), to_f32(P[2 * L * U + hi])), prm, sz,
                        sr, sc);
        }
        const bool head_lo = GENERAL && ((hm >> j) & 1u);
        const bool head_hi = GENERAL && ((hm >> (j + HALF)) & 1u);
        const float2 cur = G[j];
        float2 J, g;
        if (ZERO) {
            Cell::jg_zero(sz, sr, sc, prm, J, g);
        } else {
            float2 hs = prev;
            if (head_lo) hs.x = 0.f;
            if (head_hi) hs.y = 0.f;
            Cell::jg(hs, sz, sr, sc, prm, J, g);
        }
        if (GENERAL) {
            if (head_lo) J.x = 0.f;
            if (head_hi) J.y = 0.f;
            if (j >= nvalid) { J.x = 1.f; g.x = 0.f; }
            if (j + HALF >= nvalid) { J.y = 1.f; g.y = 0.f; }
        }
        prev = cur;
        J2[j] = J;
        G[j] = g;
        B2 = fma2(J, B2, g);
        A2 = mul2(A2, J);
    }
    A_lo = A2.x;
    B_lo = B2.x;
    A = A2.y * A2.x;
    Bv = fmaf(A2.y, B2.x, B2.y);
}

// max |F_t| = max |H_t - f(H_{t-1}, P_t)| over this thread's rows of the
// final iterate (values as stored).  prev holds the stored H at rows r0 - 1
// and r0 + HALF - 1.  NaN propagates.
template <typename TS, bool FUSED, bool GENERAL>
__device__ __forceinline__ float residual_rows(const float *Pf, const TS *Pt, int warp, int lane,
                                               const float2 (&G)[HALF], float2 prev, uint32_t hm,
                                               int nvalid,
                                               const typename CellOf<TS>::type::Params &prm) {
    using Cell = typename CellOf<TS>::type;
    const int r0 = warp * SEG;
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < HALF; ++j) {
        float2 sz, sr, sc;
        if (FUSED) {
            const float2 *P2 = reinterpret_cast<const float2 *>(Pf);
            sz = P2[pf2_index(0, warp, j, lane)];
            sr = P2[pf2_index(1, warp, j, lane)];
            sc = P2[pf2_index(2, warp, j, lane)];
        } else {
            const int lo = (r0 + j) * U + lane, hi = lo + HALF * U;
            Cell::scale(make_float2(to_f32(Pt[lo]), to_f32(Pt[hi])),
                        make_float2(to_f32(Pt[L * U + lo]), to_f32(Pt[L * U + hi])),
                        make_float2(to_f32(Pt[2 * L * U + lo]), to_f32(Pt[2 * L * U + hi])), prm,
                        sz, sr, sc);
        }
        // the per-iteration kernel keeps G rounded to the storage type already
        const float2 hq = FUSED ? round2_to<TS>(G[j]) : G[j];
        float2 hs = prev;
        if (GENERAL) {
            if ((hm >> j) & 1u) hs.x = 0.f;
            if ((hm >> (j + HALF)) & 1u) hs.y = 0.f;
        }
        const float2 F = fma2(Cell::f(hs, sz, sr, sc, prm), splat2(-1.0f), hq);
        float fx = fabsf(F.x), fy = fabsf(F.y);
        if (GENERAL) {
            if (j >= nvalid) fx = 0.f;
            if (j + HALF >= nvalid) fy = 0.f;
        }
        m = max_nan(m, max_nan(fx, fy));
        prev = hq;
    }
    return m;
}

// XPROJ (bf16, fused only): the tile's preactivations are not read from HBM
// but computed in the prologue from x and W_x on the tensor cores:
// D = W_tile x_tile^T with M = 128 TMEM lanes = (gate, unit) rows (3 x 32 used),
// N = 128 columns = time steps, K = d_in in 64-wide slices through a 2-stage
// TMA ring that aliases the P' tile; warps 0..2 then read their gate's lanes
// (tcgen05.ld: lane = unit, registers = time), round to bf16 as a stored
// preactivation would be, and write the pre-scaled arguments.
// CTAs per SM: 8 (64 registers); the bf16 per-iteration kernel runs 9 (56
// registers, a few spills in its prologue), which measured faster than 8
template <typename TS, bool FUSED>
constexpr int newton_min_blocks() { return (!FUSED && sizeof(TS) == 2) ? 9 : 8; }

// EARLY: warp 0 reads the nearest predecessors' look-back slots before the
// CTA barrier (see with_lookback_mode)
// PLAN: the chunks of a pack are segment-aligned, taken from a.plan.
// WARM: an iterate is given (fused: H^(0) instead of 0; per-iteration:
// H^(k-1), i.e. every launch but the first of a forward from 0).  A constant,
// so that the start from 0 compiles without the iterate's loads and the other
// launches without the zero-state cell.
template <typename TS, bool FUSED, bool XPROJ = false, bool EARLY = false, bool PLAN = false,
          bool WARM = false>
__global__ void __launch_bounds__(NW * 32, newton_min_blocks<TS, FUSED>())
    k_newton(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmH,
             const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmX,
             const __grid_constant__ CUtensorMap tmW, const NewtonArgs a) {
    extern __shared__ __align__(128) unsigned char dsmem_raw[];
    // the swizzled XPROJ stages want an aligned base (1024 bytes covers every swizzle)
    unsigned char *dsmem = XPROJ ? reinterpret_cast<unsigned char *>(
                                       (reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023))
                                 : dsmem_raw;
    // FUSED: [3][L][U] fp32 pre-scaled arguments (a bf16 tile lands by TMA in
    // the upper half and is widened in place), then, with an initial iterate,
    // its [L][U] tile.  Per-iteration: [3][L][U] raw preactivations of type TS,
    // then (bf16) the [L][U] tile of H^(k-1); fp32 reads H^(k-1) into registers.
    float *Pf = reinterpret_cast<float *>(dsmem);
    TS *Pt = FUSED ? reinterpret_cast<TS *>(dsmem + (sizeof(TS) == 2 ? 3 * L * U * 2 : 0))
                   : reinterpret_cast<TS *>(dsmem);
    TS *Hs = FUSED ? reinterpret_cast<TS *>(dsmem + 3 * L * U * sizeof(float))
                   : reinterpret_cast<TS *>(dsmem) + 3 * L * U;
    __shared__ float s_aggA[NW][32], s_aggB[NW][32];
    __shared__ float s_C[32];
    __shared__ uint32_t s_heads[L / 32];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ __align__(8) uint64_t s_xfull[2], s_xempty[2], s_xacc;   // XPROJ only
    __shared__ uint32_t s_tmem;                                         // XPROJ only
    // this CTA's ticket: chunk (position in its look-back chain), batch row,
    // unit tile, first row, end of the rows it may write, chain index of the
    // look-back slots
    __shared__ int s_tile[6];
    __shared__ uint32_t s_red[NW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr bool REG_H = !FUSED && sizeof(TS) == 4;   // H^(k-1) in registers, not a tile
    // launched as a dependent of the kernel before it on the stream (the
    // workspace clear, or the previous iteration); the next iteration's CTAs
    // may be scheduled as soon as all of this grid's have started.  Every
    // access to memory lies behind griddepcontrol.wait, except in iterations
    // 2..K of the per-iteration forward: these CTAs start only once the
    // previous iteration's have all started, so that the workspace clear
    // before iteration 1 has completed; they take their ticket (cleared
    // there) and load their tile of P (read-only) while the previous
    // iteration finishes, and wait only before they touch H^(k-1) and the
    // look-back slots
    const bool early_p = !FUSED && !XPROJ && a.k_first > 1;
    if (!early_p) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if (tid == 0) {
        // tickets run chunk-major: every chunk this tile's look-back waits for
        // belongs to a CTA that has already started
        const uint32_t ticket = atomicAdd(a.ticket, 1u);
        if constexpr (PLAN) {
            // segment-aligned chunks of a pack, level by level; the grid is
            // sized for an upper bound of their number
            const uint32_t item = ticket / a.n_ut;
            const int n_items = a.plan[0].x;
            const int4 e = a.plan[1 + item];
            s_tile[0] = e.z;
            s_tile[1] = 0;
            s_tile[2] = static_cast<int>(ticket - item * a.n_ut);
            s_tile[3] = item < static_cast<uint32_t>(n_items) ? e.x : -1;
            s_tile[4] = e.y;
            s_tile[5] = e.w;
        } else {
            const uint32_t per_chunk = static_cast<uint32_t>(a.B) * a.n_ut;
            const uint32_t cc = ticket / per_chunk, rem = ticket - cc * per_chunk;
            s_tile[0] = static_cast<int>(cc);
            s_tile[1] = static_cast<int>(rem / a.n_ut);
            s_tile[2] = static_cast<int>(rem % a.n_ut);
        }
    }
    if (tid < L / 32) s_heads[tid] = 0u;
    __syncthreads();
    if constexpr (PLAN) {
        if (s_tile[3] < 0) return;   // a ticket past the plan's last chunk
    }

    const int c = s_tile[0], b = s_tile[1], ut = s_tile[2];
    // t_end: rows at or past it are outside this tile's sequence (the end of
    // the row, or of the tile's segment in a segment-aligned pack)
    const int t0 = PLAN ? s_tile[3] : c * L, t_end = PLAN ? s_tile[4] : a.T;
    const int chain = PLAN ? s_tile[5] : c;
    const int u0 = ut * U;
    const bool load_h = WARM;   // H^(0) (fused) or H^(k-1) (per-iteration) given

    if (tid == 0) {
        if constexpr (XPROJ) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&s_xfull[i], 1);
                mbar_init(&s_xempty[i], 1);
            }
            mbar_init(&s_xacc, 1);
            fence_mbar_init();
        } else {
            mbar_init(&s_bar, 1);
            fence_mbar_init();
            // the fp32 per-iteration kernel reads H^(k-1) straight into registers
            const bool tile_h = !REG_H && load_h;
            const uint32_t bytes = (3u + (tile_h ? 1u : 0u)) * L * U * sizeof(TS);
            mbar_arrive_expect_tx(&s_bar, bytes);
#pragma unroll
            for (int g = 0; g < 3; ++g)
                tma_load_3d(Pt + g * L * U, &tmP, &s_bar, g * a.d_h + u0, t0, b);
            if (early_p) asm volatile("griddepcontrol.wait;" ::: "memory");
            if (tile_h) tma_load_3d(Hs, &tmH, &s_bar, u0, t0, b);
        }
        if constexpr (PLAN) {
            if (c == 0) s_heads[0] = 1u;   // a segment's first chunk starts at its head
        } else {
            mark_heads(a.cu, a.S, t0, L, s_heads);
        }
    }
    if (early_p && tid != 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (XPROJ) {
        if (warp == 2) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&s_tmem)),
                         "r"(XP_TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
    const int u = u0 + lane;
    const bool uok = u < a.d_h;
    using Cell = typename CellOf<TS>::type;
    const UnitParams up = load_unit_params(a.params, a.d_h, u, uok);
    const typename Cell::Params prm2 = Cell::make(up);
    const int r0 = warp * SEG;
    // shifted state at this warp's first row: H^(k-1) at row r0 - 1
    float hb = 0.f;
    if (load_h && warp == 0 && t0 > 0 && uok)
        hb = to_f32(reinterpret_cast<const TS *>(a.H_prev)[(static_cast<size_t>(b) * a.T + t0 - 1) *
                                                               a.d_h + u]);
    // fp32 per-iteration: H^(k-1) of this warp's rows goes straight into
    // registers (one 128-byte row per warp load), in flight together with the
    // P tile's TMA; rows past T and units past d_h read as 0.  Keeping it out
    // of shared memory leaves room for 8 CTAs per SM (bf16 tiles fit 8 with
    // it, and its 2-byte loads were slower than the TMA tile).
    float2 Hreg[HALF];
    if constexpr (REG_H) {
#pragma unroll
        for (int j = 0; j < HALF; ++j) Hreg[j] = splat2(0.f);
        if (load_h && uok) {
            const TS *Hp = reinterpret_cast<const TS *>(a.H_prev) +
                           (static_cast<size_t>(b) * a.T + t0) * a.d_h + u;
            const int rows = t_end - t0;   // rows of this chunk inside the sequence
#pragma unroll
            for (int j = 0; j < HALF; ++j) {
                if (r0 + j < rows) Hreg[j].x = to_f32(Hp[static_cast<size_t>(r0 + j) * a.d_h]);
                if (r0 + HALF + j < rows)
                    Hreg[j].y = to_f32(Hp[static_cast<size_t>(r0 + HALF + j) * a.d_h]);
            }
            if (warp > 0 && r0 - 1 < rows) hb = to_f32(Hp[static_cast<size_t>(r0 - 1) * a.d_h]);
        }
    }
    __syncthreads();   // barriers initialised, head bits visible
    if constexpr (XPROJ) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t tmem = s_tmem;
        const int kt_count = (a.d_in + XP_BK - 1) / XP_BK;
        if (warp == 0 && lane == 0) {
            // TMA producer: W_x rows of the three gates of this unit tile, x rows of this chunk
            for (int kt = 0; kt < kt_count; ++kt) {
                const int st = kt & 1;
                if (kt >= 2) mbar_wait_bounded(&s_xempty[st], ((kt >> 1) - 1) & 1, a.wait_ns, a.error);
                unsigned char *A = dsmem + st * XP_STAGE_BYTES;
                mbar_arrive_expect_tx(&s_xfull[st], 3 * XP_W_BOX_BYTES + XP_X_BYTES);
#pragma unroll
                for (int g = 0; g < 3; ++g)
                    tma_load_2d(A + g * XP_W_BOX_BYTES, &tmW, &s_xfull[st], kt * XP_BK, g * a.d_h + u0);
                tma_load_3d(A + XP_A_BYTES, &tmX, &s_xfull[st], kt * XP_BK, t0, b);
            }
        } else if (warp == 1 && lane == 0) {
            // MMA issuer
            for (int kt = 0; kt < kt_count; ++kt) {
                const int st = kt & 1;
                mbar_wait_bounded(&s_xfull[st], (kt >> 1) & 1, a.wait_ns, a.error);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t A = smem_u32(dsmem + st * XP_STAGE_BYTES);
#pragma unroll
                for (int kk = 0; kk < XP_BK / 16; ++kk)
                    mma<false, XP_IDESC>(tmem, sw64_desc(A + kk * 32),
                                         sw64_desc(A + XP_A_BYTES + kk * 32),
                                         (kt > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&s_xempty[st]);
            }
            mma_commit(&s_xacc);
        }
        __syncwarp();
        const bool ok = mbar_wait_bounded(&s_xacc, 0, a.wait_ns, a.error);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // P' overwrites the stages
        if (warp < 3) {
            // lane = unit of gate `warp`, registers = 32 time steps per load
            // (two warps' rows), written in pair order
            float mul, add;
            Cell::gate_affine(warp, up, mul, add);
            float2 *P2 = reinterpret_cast<float2 *>(Pf);
#pragma unroll 1
            for (int cc = 0; cc < L / 32; ++cc) {
                uint32_t v[32];
                tmem_ld_cols<32>(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    if ((i % SEG) >= HALF) continue;
                    const float lo = fmaf(round_to<__nv_bfloat16>(__uint_as_float(v[i])), mul, add);
                    const float hi =
                        fmaf(round_to<__nv_bfloat16>(__uint_as_float(v[i + HALF])), mul, add);
                    const float nan = __int_as_float(0x7fffffff);
                    P2[pf2_index(warp, cc * 2 + i / SEG, i % SEG, lane)] =
                        ok ? make_float2(lo, hi) : make_float2(nan, nan);
                }
            }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        if (warp == 2) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(XP_TMEM_COLS)
                         : "memory");
        }
    } else {
        mbar_wait_bounded(&s_bar, 0, a.wait_ns, a.error);
    }

    if (FUSED && !XPROJ) {
        // each warp pre-scales its own rows once, P' = scale (P + b) per gate,
        // into pair order; for fp32 the tile is rewritten in place inside the
        // warp's own rows, for bf16 the source tile overlaps other warps'
        // destinations
        float2 v[3][HALF];
        const TS *src = Pt + r0 * U + lane;
#pragma unroll
        for (int j = 0; j < HALF; ++j)
#pragma unroll
            for (int g = 0; g < 3; ++g)
                v[g][j] = make_float2(to_f32(src[g * L * U + j * U]), to_f32(src[g * L * U + (j + HALF) * U]));
        if (sizeof(TS) == 2) __syncthreads();
        else __syncwarp();
        float2 *P2 = reinterpret_cast<float2 *>(Pf);
#pragma unroll
        for (int j = 0; j < HALF; ++j) {
            float2 sz, sr, sc;
            Cell::scale(v[0][j], v[1][j], v[2][j], prm2, sz, sr, sc);
            P2[pf2_index(0, warp, j, lane)] = sz;
            P2[pf2_index(1, warp, j, lane)] = sr;
            P2[pf2_index(2, warp, j, lane)] = sc;
        }
        __syncwarp();
    }

    float2 G[HALF];   // H of this warp's rows (between iterations) / g_t (inside), in pairs
#pragma unroll
    for (int j = 0; j < HALF; ++j)
        G[j] = REG_H ? Hreg[j]
               : load_h ? make_float2(to_f32(Hs[(r0 + j) * U + lane]), to_f32(Hs[(r0 + HALF + j) * U + lane]))
                        : splat2(0.f);
    if (!REG_H && load_h && warp > 0) hb = to_f32(Hs[(r0 - 1) * U + lane]);
    const uint32_t hm = (s_heads[r0 >> 5] >> (r0 & 31)) & ((1u << SEG) - 1u);
    const int nvalid = min(SEG, t_end - (t0 + r0));
    const bool general = (hm != 0u) || (nvalid < SEG);
    const void *Pv = FUSED ? static_cast<const void *>(Pf) : static_cast<const void *>(Pt);

    const int stride = PLAN ? a.chain_stride : a.n_chunks;   // look-back slots per column
    const int n_tiles = a.B * a.n_ut * stride;
    const int tile = (b * a.n_ut + ut) * stride + chain;

    for (int k = a.k_first; k <= a.k_last; ++k) {
        float2 J2[HALF];
        float A_lo, B_lo, A, Bv;
        if ((!FUSED || k == 1) && !load_h) {   // from H^(0) = 0: every shifted state is 0
            if (general)
                warp_pairs<TS, FUSED, true, true>(Pv, warp, lane, G, hb, hm, nvalid, prm2, J2, A_lo, B_lo, A, Bv);
            else
                warp_pairs<TS, FUSED, false, true>(Pv, warp, lane, G, hb, hm, nvalid, prm2, J2, A_lo, B_lo, A, Bv);
        } else if (general) {
            warp_pairs<TS, FUSED, true>(Pv, warp, lane, G, hb, hm, nvalid, prm2, J2, A_lo, B_lo, A, Bv);
        } else {
            warp_pairs<TS, FUSED, false>(Pv, warp, lane, G, hb, hm, nvalid, prm2, J2, A_lo, B_lo, A, Bv);
        }
        // when few chunks of a column run at once, the nearest predecessors
        // have usually published by now: warp 0 reads their slots before the
        // barrier, so that the L2 round trip overlaps the other warps' rows
        unsigned long long *slot =
            a.slots + (static_cast<size_t>(k - 1) * n_tiles + tile) * 32 + lane;
        unsigned long long pre1 = SLOT_EMPTY, pre2 = SLOT_EMPTY;
        if (EARLY && warp == 0) {
            if (c > 0) pre1 = ld_relaxed_u64(slot - 32);
            if (c > 1) pre2 = ld_relaxed_u64(slot - 64);
        }
        s_aggA[warp][lane] = A;
        s_aggB[warp][lane] = Bv;
        __syncthreads();

        if (warp == 0) {
            // chunk aggregate; every warp's exclusive prefix replaces its aggregate
            float tA = 1.f, tB = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float wa = s_aggA[w][lane], wb = s_aggB[w][lane];
                s_aggA[w][lane] = tA;
                s_aggB[w][lane] = tB;
                tB = fmaf(wa, tB, wb);
                tA *= wa;
            }
            float C = 0.f;   // H^(k) at t0 - 1 (0 before the first step)
            const bool pub = tile != a.withhold_tile;
            if (c == 0) {
                if (pub) publish(slot, 0.f, tB);
            } else {
                if (pub) publish(slot, tA, tB);
                C = lookback_lane<EARLY ? 2 : 4>(slot, c, -1, a.n_chunks, a.wait_ns, a.error, pre1,
                                                  pre2);
                if (pub) publish(slot, 0.f, fmaf(tA, C, tB));
            }
            s_C[lane] = C;
        }
        __syncthreads();

        // H^(k) of this warp's rows from H^(k) at row r0 - 1 (first half) and at
        // row r0 + HALF - 1 (second half, through the first half's map)
        const float h = fmaf(s_aggA[warp][lane], s_C[lane], s_aggB[warp][lane]);
        hb = FUSED ? h : round_to<TS>(h);
        float2 h2 = make_float2(h, fmaf(A_lo, h, B_lo));
#pragma unroll
        for (int j = 0; j < HALF; ++j) {
            h2 = fma2(J2[j], h2, G[j]);
            G[j] = FUSED ? h2 : round2_to<TS>(h2);
        }
    }

    // residual max|F(H^(K))| at the values as stored (every fused launch; the
    // last per-iteration one).  The early fused forms take it as a constant
    // condition: their register allocation comes out faster that way (B16
    // T16384 bf16 1.016 -> 1.011 ms), the plain form's slower (B4 T131072
    // 0.147 -> 0.149 ms)
    if ((FUSED && EARLY) || a.last) {
        // each warp read only its own prefix slot in the apply step: reuse the
        // slots for the last row of each warp
        // (the per-iteration kernel's G and hb are rounded to the storage type already)
        s_aggA[warp][lane] = FUSED ? round_to<TS>(G[HALF - 1].y) : G[HALF - 1].y;
        __syncthreads();
        const float2 prev = make_float2((warp == 0) ? (FUSED ? round_to<TS>(hb) : hb) : s_aggA[warp - 1][lane],
                                        FUSED ? round_to<TS>(G[HALF - 1].x) : G[HALF - 1].x);
        float m = general ? residual_rows<TS, FUSED, true>(Pf, Pt, warp, lane, G, prev, hm, nvalid, prm2)
                          : residual_rows<TS, FUSED, false>(Pf, Pt, warp, lane, G, prev, hm, nvalid, prm2);
        if (!uok) m = 0.f;
        m = abs_residual(m);   // NaN counts as +inf
        const uint32_t v = __reduce_max_sync(FULL_MASK, __float_as_uint(m));
        if (lane == 0) s_red[warp] = v;
        __syncthreads();
        if (tid == 0) {
            uint32_t mx = 0u;
#pragma unroll
            for (int w = 0; w < NW; ++w) mx = max(mx, s_red[w]);
            atomicMax(a.residual_bits, mx);
        }
    }

    if constexpr (PLAN) {
        if (t_end - t0 < L) {
            // the last chunk of a segment in a segment-aligned pack: the rows
            // after it belong to the next segment, so the rows are stored one by one
            if (uok) {
                TS *Ho = static_cast<TS *>(a.H_next) + static_cast<size_t>(t0) * a.d_h + u;
                const int rows = t_end - t0;
#pragma unroll
                for (int j = 0; j < HALF; ++j) {
                    if (r0 + j < rows) Ho[static_cast<size_t>(r0 + j) * a.d_h] = from_f32<TS>(G[j].x);
                    if (r0 + HALF + j < rows)
                        Ho[static_cast<size_t>(r0 + HALF + j) * a.d_h] = from_f32<TS>(G[j].y);
                }
            }
            return;
        }
    }
    // H^(K) of the tile -> shared memory (the P tile's space: every read of it
    // lies behind the last barrier) -> one TMA store, which clips rows past T
    // and units past d_h
    TS *Hst = reinterpret_cast<TS *>(dsmem);   // [L][U]
#pragma unroll
    for (int j = 0; j < HALF; ++j) {
        Hst[(r0 + j) * U + lane] = from_f32<TS>(G[j].x);
        Hst[(r0 + HALF + j) * U + lane] = from_f32<TS>(G[j].y);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        tma_store_3d(&tmO, Hst, u0, t0, b);
        bulk_commit_and_wait_read();
    }
}

// Residual of a given trajectory (G == null: the zero trajectory).
template <typename TS>
__global__ void __launch_bounds__(NW * 32)
    k_residual(const TS *__restrict__ P, const float *__restrict__ params,
               const TS *__restrict__ G, int T, int d_h, const int32_t *cu, int S,
               uint32_t *residual_bits) {
    __shared__ uint32_t s_heads[L / 32];
    __shared__ uint32_t s_red[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int u = blockIdx.x * U + lane, t0 = blockIdx.y * L, b = blockIdx.z;
    if (tid < L / 32) s_heads[tid] = 0u;
    __syncthreads();
    if (tid == 0) mark_heads(cu, S, t0, L, s_heads);
    __syncthreads();
    const bool uok = u < d_h;
    const UnitParams prm = load_unit_params(params, d_h, u, uok);
    float m = 0.f;
    if (uok) {
        const int r0 = warp * SEG;
        const size_t row0 = static_cast<size_t>(b) * T;
        float hprev = (G != nullptr && t0 + r0 > 0) ? to_f32(G[(row0 + t0 + r0 - 1) * d_h + u]) : 0.f;
        for (int i = 0; i < SEG; ++i) {
            const int r = r0 + i, t = t0 + r;
            if (t >= T) break;
            const TS *p = P + (row0 + t) * 3 * d_h + u;
            const float g = (G != nullptr) ? to_f32(G[(row0 + t) * d_h + u]) : 0.f;
            const float hs = head_bit(s_heads, r) ? 0.f : hprev;
            const float f = cell_f(hs, to_f32(p[0]), to_f32(p[d_h]), to_f32(p[2 * d_h]), prm);
            m = fmaxf(m, abs_residual(g - f));
            hprev = g;
        }
    }
    const uint32_t v = __reduce_max_sync(FULL_MASK, __float_as_uint(m));
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    if (tid == 0) {
        uint32_t mx = 0u;
        for (int w = 0; w < NW; ++w) mx = max(mx, s_red[w]);
        atomicMax(residual_bits, mx);
    }
}

__global__ void k_head_mask(const int32_t *cu, int S, int64_t N, uint8_t *mask) {
    constexpr int SPAN = 1024;
    __shared__ uint32_t bits[SPAN / 32];
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * SPAN;
    if (threadIdx.x < SPAN / 32) bits[threadIdx.x] = 0u;
    __syncthreads();
    if (threadIdx.x == 0) mark_heads(cu, S, t0, SPAN, bits);
    __syncthreads();
    for (int i = threadIdx.x; i < SPAN; i += blockDim.x)
        if (t0 + i < N) mask[t0 + i] = head_bit(bits, i) ? 1 : 0;
}

__global__ void k_bounded_wait(const uint32_t *flag, uint64_t wait_ns, uint32_t *result) {
    const uint64_t ts = globaltimer_ns();
    while (ld_acquire_u32(flag) == 0u) {
        if (globaltimer_ns() - ts > wait_ns) {
            *result = 2u;
            return;
        }
        __nanosleep(256);
    }
    *result = 1u;
}

template <typename TS, bool FUSED>
size_t smem_bytes_for(bool with_h) {
    return FUSED ? static_cast<size_t>(3) * L * U * sizeof(float) + (with_h ? L * U * sizeof(TS) : 0)
                 : static_cast<size_t>(sizeof(TS) == 4 ? 3 : 4) * L * U * sizeof(TS);
}

// Early look-back reads pay when few chunks of each column (batch row x unit
// tile) are resident at once: then the nearest predecessor has usually
// published its inclusive prefix by the time a tile has its own aggregate.
// With many resident chunks per column (long sequences of few columns) the
// early read mostly finds a predecessor still at work.
bool early_lookback(const NewtonArgs &a, int ctas_per_sm, bool plan) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    const int64_t resident = static_cast<int64_t>(sms) * ctas_per_sm;
    // a segment-aligned pack has one look-back chain per segment and unit tile
    const int64_t columns = static_cast<int64_t>(plan ? a.S : a.B) * a.n_ut;
    return resident <= EARLY_LOOKBACK_CHUNKS * columns;
}

template <typename TS, bool FUSED, bool EARLY, bool PLAN, bool WARM>
cudaError_t launch_one(const CUtensorMap &tmP, const CUtensorMap &tmH, const CUtensorMap &tmO,
                       const NewtonArgs &a, int64_t n_ctas, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    const size_t smem = smem_bytes_for<TS, FUSED>(a.H_prev != nullptr);
    cudaError_t e = once_per_device(configured, [](int) {
        return cudaFuncSetAttribute(k_newton<TS, FUSED, false, EARLY, PLAN, WARM>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem_bytes_for<TS, FUSED>(true)));
    });
    if (e != cudaSuccess) return e;
    return launch_dependent(k_newton<TS, FUSED, false, EARLY, PLAN, WARM>,
                            static_cast<unsigned>(n_ctas), NW * 32, smem, stream, tmP, tmH, tmO, tmP,
                            tmP, a);
}

template <typename TS, bool FUSED, bool EARLY, bool PLAN>
cudaError_t launch_one(const CUtensorMap &tmP, const CUtensorMap &tmH, const CUtensorMap &tmO,
                       const NewtonArgs &a, int64_t n_ctas, cudaStream_t stream) {
    if (a.H_prev != nullptr)   // an iterate given: H^(0) (fused), H^(k-1) (per-iteration)
        return launch_one<TS, FUSED, EARLY, PLAN, true>(tmP, tmH, tmO, a, n_ctas, stream);
    return launch_one<TS, FUSED, EARLY, PLAN, false>(tmP, tmH, tmO, a, n_ctas, stream);
}

template <typename TS, bool FUSED>
cudaError_t launch_one(const CUtensorMap &tmP, const CUtensorMap &tmH, const CUtensorMap &tmO,
                       const NewtonArgs &a, int64_t n_ctas, cudaStream_t stream, bool plan) {
    const bool early = early_lookback(a, newton_min_blocks<TS, FUSED>(), plan);
    if (plan)
        return early ? launch_one<TS, FUSED, true, true>(tmP, tmH, tmO, a, n_ctas, stream)
                     : launch_one<TS, FUSED, false, true>(tmP, tmH, tmO, a, n_ctas, stream);
    return early ? launch_one<TS, FUSED, true, false>(tmP, tmH, tmO, a, n_ctas, stream)
                 : launch_one<TS, FUSED, false, false>(tmP, tmH, tmO, a, n_ctas, stream);
}

cudaError_t launch_x(const CUtensorMap &tmX, const CUtensorMap &tmW, const CUtensorMap &tmO,
                     const NewtonArgs &a, int64_t n_ctas, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    constexpr size_t smem = XP_RING_BYTES + 1024;   // stages alias the P' tile; + alignment
    static_assert(XP_RING_BYTES >= 3 * L * U * 4 && XP_RING_BYTES >= 2 * XP_STAGE_BYTES,
                  "the ring holds two stages and the P' tile");
    static_assert(XP_BK * 2 == 64 && XP_A_BYTES % 512 == 0 && XP_STAGE_BYTES % 512 == 0,
                  "64-byte swizzled tiles of 64-byte rows start on 512-byte boundaries");
    static_assert(XP_STAGE_BYTES >= 128 * XP_BK * 2, "the MMA's 128 A rows stay inside the stage");
    cudaError_t e = once_per_device(configured, [](int) {
        return cudaFuncSetAttribute(k_newton<__nv_bfloat16, true, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    });
    if (e != cudaSuccess) return e;
    return launch_dependent(k_newton<__nv_bfloat16, true, true>, static_cast<unsigned>(n_ctas),
                            NW * 32, smem, stream, tmX, tmX, tmO, tmX, tmW, a);
}

}  // namespace

size_t newton_smem_bytes(int dtype, bool fused) {
    if (dtype == 1)
        return fused ? smem_bytes_for<__nv_bfloat16, true>(true) : smem_bytes_for<__nv_bfloat16, false>(true);
    return fused ? smem_bytes_for<float, true>(true) : smem_bytes_for<float, false>(true);
}

int newton_lookback_form(int dtype, bool fused, const NewtonArgs &a, bool plan) {
    const int per_sm = dtype == 1 ? (fused ? newton_min_blocks<__nv_bfloat16, true>()
                                           : newton_min_blocks<__nv_bfloat16, false>())
                                  : (fused ? newton_min_blocks<float, true>()
                                           : newton_min_blocks<float, false>());
    return early_lookback(a, per_sm, plan) ? 1 : 0;
}

cudaError_t launch_newton(int dtype, bool fused, const CUtensorMap &tmP, const CUtensorMap &tmH,
                          const CUtensorMap &tmO, const NewtonArgs &a, int64_t n_ctas,
                          cudaStream_t stream, bool plan) {
    if (dtype == 1)
        return fused ? launch_one<__nv_bfloat16, true>(tmP, tmH, tmO, a, n_ctas, stream, plan)
                     : launch_one<__nv_bfloat16, false>(tmP, tmH, tmO, a, n_ctas, stream, plan);
    return fused ? launch_one<float, true>(tmP, tmH, tmO, a, n_ctas, stream, plan)
                 : launch_one<float, false>(tmP, tmH, tmO, a, n_ctas, stream, plan);
}

cudaError_t launch_newton_x(const CUtensorMap &tmX, const CUtensorMap &tmW, const CUtensorMap &tmO,
                            const NewtonArgs &a, int64_t n_ctas, cudaStream_t stream) {
    return launch_x(tmX, tmW, tmO, a, n_ctas, stream);
}

cudaError_t launch_residual(int dtype, const void *P, const float *params, const void *G, int B,
                            int T, int d_h, const int32_t *cu, int S, uint32_t *residual_bits,
                            cudaStream_t stream) {
    const dim3 grid((d_h + U - 1) / U, (T + L - 1) / L, B);
    if (dtype == 1)
        k_residual<__nv_bfloat16><<<grid, NW * 32, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(P), params, static_cast<const __nv_bfloat16 *>(G), T,
            d_h, cu, S, residual_bits);
    else
        k_residual<float><<<grid, NW * 32, 0, stream>>>(static_cast<const float *>(P), params,
                                                    static_cast<const float *>(G), T, d_h, cu, S,
                                                    residual_bits);
    return cudaGetLastError();
}

cudaError_t launch_head_mask(const int32_t *cu, int S, int64_t N, uint8_t *mask,
                             cudaStream_t stream) {
    const int64_t blocks = (N + 1023) / 1024;
    k_head_mask<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(cu, S, N, mask);
    return cudaGetLastError();
}

cudaError_t launch_bounded_wait(const uint32_t *flag, uint64_t wait_ns, uint32_t *result,
                                cudaStream_t stream) {
    k_bounded_wait<<<1, 1, 0, stream>>>(flag, wait_ns, result);
    return cudaGetLastError();
}

}  // namespace nrnn

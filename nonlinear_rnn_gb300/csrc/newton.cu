// Parallel Newton forward of the diagonal-mix GRU (sm_103a).
//
// One CTA owns a tile of 32 hidden units (one per lane) x L = 128 time steps
// of one batch row.  Per Newton iteration it
//   1. evaluates the cell at the shifted trajectory H_{t-1} for every step of
//      the tile: F_t = H_t - f(H_{t-1}, P_t), J_t = df/dh (J = 0 and shifted
//      state 0 at segment heads; pararnn-torch shapes_layout, "cu_seqlens");
//   2. composes the affine maps delta -> J_t delta - F_t serially inside each
//      warp's 16 steps, then across the 8 warps in shared memory;
//   3. obtains the carry delta_{t0-1} from earlier chunks by a decoupled
//      look-back over per-chunk published (A, b) pairs, each warp of the CTA
//      inspecting one predecessor of an 8-chunk window per round;
//   4. applies the carry and updates H <- H + delta.
// The fused variant repeats 1-4 for all K iterations on the tile held in
// shared memory/registers (the shifted state at the tile's first step is
// tracked as H^(k)_{t0-1} = H^(k-1)_{t0-1} + carry_k), so P is read once and
// H written once.  The per-iteration variant runs one iteration per launch
// and streams H^(k-1) in and H^(k) out.  The launch that produces H^(K)
// evaluates F(H^(K)) once more for the residual gate max|F| (numerics
// contract, "Two thresholds").
//
// Tiles of P (three gate blocks) and of H^(k-1) are staged in shared memory
// by TMA (cp.async.bulk.tensor, completion on an mbarrier).  CTAs take tiles
// from an atomic ticket in chunk-major order, so every CTA whose result a
// CTA waits for has already started: the look-back cannot deadlock.  Every
// wait is bounded by the caller's limit and reports a timeout in the error
// word instead of hanging.
#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

namespace {

constexpr int NW = NEWTON_NW;
constexpr int SEG = NEWTON_SEG;
constexpr int L = NEWTON_L;
constexpr int U = TILE_U;

constexpr uint32_t FLAG_AGGREGATE = 1u;
constexpr uint32_t FLAG_INCLUSIVE = 2u;

// Publishes one (A, b) pair per lane for a chunk, then its status flag.
__device__ __forceinline__ void publish(uint32_t *flag, unsigned long long *slot, float A,
                                        float b, uint32_t kind, int lane) {
    st_relaxed_u64(slot, pack_pair(A, b));
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_u32(flag, kind);
}

struct LookbackSmem {
    float winA[NW][32];
    float winB[NW][32];
    float cA[32];
    float cB[32];
    int done;
};

// Decoupled look-back for the chunk at `tile` (chunk index c > 0): returns the
// carry delta_{t0-1} for this lane's unit.  All warps of the CTA take part;
// warp w reads predecessor base - w of the current window.  Must be called by
// the whole CTA (it contains barriers); s.cA/s.cB must hold (1, 0).
__device__ __forceinline__ float lookback(const uint32_t *flags, const unsigned long long *slots,
                                          int tile, int c, LookbackSmem &s, uint64_t wait_ns,
                                          uint32_t *error) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int base = c - 1;; base -= NW) {
        const int p = base - warp;
        float pa = 0.f, pb = 0.f;   // p < 0: the sequence start, delta = 0
        if (p >= 0) {
            const int pt = tile - (c - p);
            uint32_t f = ld_acquire_u32(flags + pt);
            if (!__all_sync(FULL_MASK, f != 0u)) {
                const uint64_t ts = globaltimer_ns();
                for (;;) {
                    __nanosleep(32);
                    f = ld_acquire_u32(flags + pt);
                    if (__all_sync(FULL_MASK, f != 0u)) break;
                    const bool late = (globaltimer_ns() - ts) > wait_ns;
                    if (__any_sync(FULL_MASK, late)) {
                        if (lane == 0) atomicOr(error, 1u);
                        break;
                    }
                }
            }
            if (__all_sync(FULL_MASK, f != 0u)) {
                const unsigned long long v = ld_relaxed_u64(slots + static_cast<size_t>(pt) * 32 + lane);
                pa = pair_A(v);
                pb = pair_b(v);
            }
        }
        s.winA[warp][lane] = pa;
        s.winB[warp][lane] = pb;
        __syncthreads();
        if (warp == 0) {
            float cA = s.cA[lane], cB = s.cB[lane];
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                if (cA != 0.f) {
                    cB = fmaf(cA, s.winB[w][lane], cB);
                    cA *= s.winA[w][lane];
                }
            }
            s.cA[lane] = cA;
            s.cB[lane] = cB;
            // done when every lane's prefix is closed (A = 0) or the window has
            // reached chunk 0 (a NaN input keeps A = NaN, never 0)
            const bool all_done = __all_sync(FULL_MASK, cA == 0.f) || base - (NW - 1) <= 0;
            if (lane == 0) s.done = all_done ? 1 : 0;
        }
        __syncthreads();
        if (s.done) break;
    }
    return s.cB[lane];
}

template <typename TS, bool FUSED>
__global__ void __launch_bounds__(NW * 32)
    k_newton(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmH,
             const NewtonArgs a) {
    extern __shared__ __align__(128) unsigned char dsmem[];
    TS *Ps = reinterpret_cast<TS *>(dsmem);   // [3][L][U]
    TS *Hs = Ps + 3 * L * U;                  // [L][U] (per-iteration variant only)
    __shared__ float s_exA[NW][32], s_exB[NW][32];   // per-warp aggregate, then exclusive prefix
    __shared__ float s_last[NW][32];                 // last H of each warp's rows
    __shared__ float s_chunkA[32], s_chunkB[32];
    __shared__ LookbackSmem s_lb;
    __shared__ uint32_t s_heads[L / 32];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ uint32_t s_ticket;
    __shared__ uint32_t s_red[NW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_ticket = atomicAdd(a.ticket, 1u);
    if (tid < L / 32) s_heads[tid] = 0u;
    __syncthreads();

    const uint32_t per_chunk = static_cast<uint32_t>(a.B) * a.n_ut;
    const int c = static_cast<int>(s_ticket / per_chunk);
    const int rem = static_cast<int>(s_ticket - static_cast<uint32_t>(c) * per_chunk);
    const int b = rem / a.n_ut, ut = rem - (rem / a.n_ut) * a.n_ut;
    const int t0 = c * L, u0 = ut * U;
    const bool load_h = !FUSED && a.H_prev != nullptr;

    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
        const uint32_t bytes = (3u + (load_h ? 1u : 0u)) * L * U * sizeof(TS);
        mbar_arrive_expect_tx(&s_bar, bytes);
#pragma unroll
        for (int g = 0; g < 3; ++g)
            tma_load_3d(Ps + g * L * U, &tmP, &s_bar, g * a.d_h + u0, t0, b);
        if (load_h) tma_load_3d(Hs, &tmH, &s_bar, u0, t0, b);
        mark_heads(a.cu, a.S, t0, L, s_heads);
    }
    const int u = u0 + lane;
    const bool uok = u < a.d_h;
    const UnitParams prm = load_unit_params(a.params, a.d_h, u, uok);
    float hb = 0.f;   // H^(k-1) at t0 - 1, this lane's unit
    if (load_h && t0 > 0 && uok)
        hb = to_f32(reinterpret_cast<const TS *>(a.H_prev)[(static_cast<size_t>(b) * a.T + t0 - 1) *
                                                               a.d_h + u]);
    __syncthreads();   // barrier initialised, head bits visible
    mbar_wait_bounded(&s_bar, 0, a.wait_ns, a.error);

    const int r0 = warp * SEG;
    float Hreg[SEG];
#pragma unroll
    for (int i = 0; i < SEG; ++i) Hreg[i] = load_h ? to_f32(Hs[(r0 + i) * U + lane]) : 0.f;
    s_last[warp][lane] = Hreg[SEG - 1];
    __syncthreads();

    const int n_tiles = a.B * a.n_ut * a.n_chunks;
    const int tile = (b * a.n_ut + ut) * a.n_chunks + c;

    for (int k = a.k_first; k <= a.k_last; ++k) {
        // 1. pairs (J_t, -F_t) at the shifted iterate, composed over this warp's steps
        float Jr[SEG], Fr[SEG];
        float A = 1.f, Bv = 0.f;
        float hprev = (warp == 0) ? hb : s_last[warp - 1][lane];
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            const int r = r0 + i;
            const bool head = head_bit(s_heads, r);
            const float hs = head ? 0.f : hprev;
            float f, J;
            cell_fj(hs, to_f32(Ps[(0 * L + r) * U + lane]), to_f32(Ps[(1 * L + r) * U + lane]),
                    to_f32(Ps[(2 * L + r) * U + lane]), prm, f, J);
            float F = Hreg[i] - f;
            if (head) J = 0.f;
            if (t0 + r >= a.T) { J = 1.f; F = 0.f; }   // past the end: identity map
            Jr[i] = J;
            Fr[i] = F;
            Bv = fmaf(J, Bv, -F);
            A *= J;
            hprev = Hreg[i];
        }
        s_exA[warp][lane] = A;
        s_exB[warp][lane] = Bv;
        __syncthreads();

        // 2. chunk aggregate and per-warp exclusive prefixes; publish
        uint32_t *flags = a.flags + static_cast<size_t>(k - 1) * n_tiles;
        unsigned long long *slots = a.slots + static_cast<size_t>(k - 1) * n_tiles * 32;
        if (warp == 0) {
            float eA = 1.f, eB = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float wa = s_exA[w][lane], wb = s_exB[w][lane];
                s_exA[w][lane] = eA;
                s_exB[w][lane] = eB;
                eB = fmaf(wa, eB, wb);
                eA *= wa;
            }
            s_chunkA[lane] = eA;
            s_chunkB[lane] = eB;
            s_lb.cA[lane] = 1.f;
            s_lb.cB[lane] = 0.f;
            if (c == 0) publish(flags + tile, slots + static_cast<size_t>(tile) * 32 + lane, 0.f, eB,
                                FLAG_INCLUSIVE, lane);
            else publish(flags + tile, slots + static_cast<size_t>(tile) * 32 + lane, eA, eB,
                         FLAG_AGGREGATE, lane);
        }
        __syncthreads();

        // 3. carry from earlier chunks
        float C = 0.f;
        if (c > 0) {
            C = lookback(flags, slots, tile, c, s_lb, a.wait_ns, a.error);
            if (warp == 0)
                publish(flags + tile, slots + static_cast<size_t>(tile) * 32 + lane, 0.f,
                        fmaf(s_chunkA[lane], C, s_chunkB[lane]), FLAG_INCLUSIVE, lane);
        }

        // 4. delta_t = J_t delta_{t-1} - F_t from the carry; H <- H + delta
        float d = fmaf(s_exA[warp][lane], C, s_exB[warp][lane]);
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            d = fmaf(Jr[i], d, -Fr[i]);
            Hreg[i] = FUSED ? (Hreg[i] + d) : round_to<TS>(Hreg[i] + d);
        }
        hb = FUSED ? (hb + C) : round_to<TS>(hb + C);
        s_last[warp][lane] = Hreg[SEG - 1];
        __syncthreads();
    }

    // residual max|F(H^(K))| at the values as stored
    if (a.last && a.residual_bits != nullptr) {
        float m = 0.f;
        float hprev = round_to<TS>((warp == 0) ? hb : s_last[warp - 1][lane]);
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            const int r = r0 + i;
            const bool head = head_bit(s_heads, r);
            const float hq = round_to<TS>(Hreg[i]);
            const float f = cell_f(head ? 0.f : hprev, to_f32(Ps[(0 * L + r) * U + lane]),
                                   to_f32(Ps[(1 * L + r) * U + lane]),
                                   to_f32(Ps[(2 * L + r) * U + lane]), prm);
            if (uok && t0 + r < a.T) m = fmaxf(m, abs_residual(hq - f));
            hprev = hq;
        }
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

    TS *Hn = reinterpret_cast<TS *>(a.H_next);
    if (uok) {
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            const int t = t0 + r0 + i;
            if (t < a.T) Hn[(static_cast<size_t>(b) * a.T + t) * a.d_h + u] = from_f32<TS>(Hreg[i]);
        }
    }
}

// Residual of a given trajectory (G == null: the zero trajectory).
template <typename TS>
__global__ void __launch_bounds__(256)
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
size_t smem_bytes_for() {
    return static_cast<size_t>(FUSED ? 3 : 4) * L * U * sizeof(TS);
}

template <typename TS, bool FUSED>
cudaError_t launch_one(const CUtensorMap &tmP, const CUtensorMap &tmH, const NewtonArgs &a,
                       int64_t n_ctas, cudaStream_t stream) {
    static bool configured = false;
    const size_t smem = smem_bytes_for<TS, FUSED>();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_newton<TS, FUSED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    k_newton<TS, FUSED><<<static_cast<unsigned>(n_ctas), NW * 32, smem, stream>>>(tmP, tmH, a);
    return cudaGetLastError();
}

}  // namespace

size_t newton_smem_bytes(int dtype, bool fused) {
    if (dtype == 1) return fused ? smem_bytes_for<__nv_bfloat16, true>() : smem_bytes_for<__nv_bfloat16, false>();
    return fused ? smem_bytes_for<float, true>() : smem_bytes_for<float, false>();
}

cudaError_t launch_newton(int dtype, bool fused, const CUtensorMap &tmP, const CUtensorMap &tmH,
                          const NewtonArgs &a, int64_t n_ctas, cudaStream_t stream) {
    if (dtype == 1)
        return fused ? launch_one<__nv_bfloat16, true>(tmP, tmH, a, n_ctas, stream)
                     : launch_one<__nv_bfloat16, false>(tmP, tmH, a, n_ctas, stream);
    return fused ? launch_one<float, true>(tmP, tmH, a, n_ctas, stream)
                 : launch_one<float, false>(tmP, tmH, a, n_ctas, stream);
}

cudaError_t launch_residual(int dtype, const void *P, const float *params, const void *G, int B,
                            int T, int d_h, const int32_t *cu, int S, uint32_t *residual_bits,
                            cudaStream_t stream) {
    const dim3 grid((d_h + U - 1) / U, (T + L - 1) / L, B);
    if (dtype == 1)
        k_residual<__nv_bfloat16><<<grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(P), params, static_cast<const __nv_bfloat16 *>(G), T,
            d_h, cu, S, residual_bits);
    else
        k_residual<float><<<grid, 256, 0, stream>>>(static_cast<const float *>(P), params,
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

// Backward (adjoint) pass of the diagonal-mix GRU recurrence h_t = f(h_{t-1}, P_t)
// at a given trajectory H (e.g. the Newton result), for the training surface
// the pararnn-torch pages mention (shapes_layout: "train forward+backward";
// numerics contract: "backward-scan-cap.md -- long-T scan limits").
//
// With upstream gradient gH = dL/dH, the total derivative lambda_t = dL/dh_t
// obeys the reverse-time affine recurrence
//   nu_t = J_t (gH_t + nu_{t+1}),   lambda_t = gH_t + nu_{t+1},   nu after the end = 0,
// with J_t = df/dh at (H_{t-1}, P_t) and J = 0 at segment heads (no gradient
// crosses a segment boundary).  Then dL/dP_{t,g} = lambda_t df/dP_g and the
// parameter gradients are sums over (b, t) of lambda_t df/d(a_g, b_g).
//
// Same tiling as the Newton kernel (32 units x NEWTON_L steps, NEWTON_NW warps
// x 16 steps) run backwards in time: tiles of P, H and gH land in shared memory by TMA;
// each thread takes its rows as pairs (i, i + 8) on packed f32x2 arithmetic with
// the storage type's cell and composes the maps nu_{t+1} -> nu_t = (J_t, J_t gH_t)
// of each half from the last row upwards; warp aggregates meet in shared memory;
// warp 0 publishes the chunk aggregate and completes a decoupled look-back over
// LATER chunks (tickets are handed out from the last chunk backwards, so every
// chunk waited for has started); the carry nu at the chunk end is then applied,
// dL/dP staged in the P tile and stored by TMA.  Parameter gradients are reduced
// over the CTA and added with one atomicAdd per (gate, unit).  Every wait is
// bounded.  When few chunks of each column are resident at once, the next
// chunk in time (processed earlier) has usually finished: warp 0 then reads
// the look-back slots of chunks c + 1 and c + 2 as soon as the tile is known,
// and the look-back starts from what they held (EARLY).
#include "nrnn_device.cuh"
#include "nrnn_internal.h"
#include "tcgen05.cuh"

namespace nrnn {

namespace {

constexpr int NW = NEWTON_NW;
constexpr int SEG = NEWTON_SEG;
constexpr int L = NEWTON_L;
constexpr int U = TILE_U;

constexpr int HALF = SEG / 2;

// shared -> global store of one gate block of dL/dP through the 4-D map
// (d_h, gate, T, B); units past d_h and steps past T are not written
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int x, int y,
                                             int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

// Gates of a pair of steps in the storage type's formulation (the forward's:
// ex2/rcp for fp32, tanh.approx for bf16), from raw preactivations.
template <typename TS> struct BwCell;
template <> struct BwCell<float> {
    using Params = ScaledParams2;
    __device__ static Params make(const UnitParams &p) { return pair_params(scale_params(p)); }
    __device__ static void scale(float2 pz, float2 pr, float2 pc, const Params &q, float2 &sz,
                                 float2 &sr, float2 &sc) {
        scale_preact2(pz, pr, pc, q, sz, sr, sc);
    }
    __device__ static void gates(float2 h, float2 sz, float2 sr, float2 sc, const Params &q,
                                 float2 &z, float2 &omz, float2 &r, float2 &c) {
        float2 qc;
        gates2(h, sz, sr, sc, q, z, r, c, qc);
        omz = fma2(z, splat2(-1.0f), splat2(1.0f));
    }
};
template <> struct BwCell<__nv_bfloat16> {
    using Params = TanhCell::Params;
    __device__ static Params make(const UnitParams &p) { return TanhCell::make(p); }
    __device__ static void scale(float2 pz, float2 pr, float2 pc, const Params &q, float2 &sz,
                                 float2 &sr, float2 &sc) {
        TanhCell::scale(pz, pr, pc, q, sz, sr, sc);
    }
    __device__ static void gates(float2 h, float2 sz, float2 sr, float2 sc, const Params &q,
                                 float2 &z, float2 &omz, float2 &r, float2 &c) {
        float2 tz, tr;
        TanhCell::gates(h, sz, sr, sc, q, tz, tr, r, c);
        z = fma2(splat2(0.5f), tz, splat2(0.5f));
        omz = fma2(splat2(-0.5f), tz, splat2(0.5f));
    }
};

// The derivatives of a pair of steps at shifted states hs: J = df/dh and the
// factors of df/dP_g and df/d(a_g) that the gradient loop scales by lambda:
//   df/dP_z = z (1 - z) (c - h),  df/dP_c = z (1 - c^2),
//   df/dP_r = z (1 - c^2) a_c h r (1 - r),  df/da_g = df/dP_g * (h, h, r h)
struct Derivs2 {
    float2 J, dz, dr, dc, rh;
};
template <typename TS>
__device__ __forceinline__ Derivs2 derivs2(float2 hs, float2 pz, float2 pr, float2 pc,
                                           const typename BwCell<TS>::Params &q, float2 a_z,
                                           float2 a_r, float2 a_c) {
    const float2 one = splat2(1.0f), mone = splat2(-1.0f);
    float2 sz, sr, sc, z, omz, r, c;
    BwCell<TS>::scale(pz, pr, pc, q, sz, sr, sc);
    BwCell<TS>::gates(hs, sz, sr, sc, q, z, omz, r, c);
    const float2 cmh = fma2(hs, mone, c);
    const float2 omc2 = fma2(mul2(c, mone), c, one);       // 1 - c^2
    const float2 rr = fma2(mul2(r, mone), r, r);           // r (1 - r)
    const float2 dq = fma2(mul2(hs, a_r), rr, r);          // d(r h)/dh
    const float2 t3 = mul2(mul2(omc2, a_c), dq);
    Derivs2 d;
    d.J = fma2(z, fma2(mul2(omz, a_z), cmh, t3), omz);
    d.dz = mul2(mul2(z, omz), cmh);
    d.dc = mul2(z, omc2);
    d.dr = mul2(mul2(d.dc, a_c), mul2(hs, rr));
    d.rh = mul2(r, hs);
    return d;
}

// A thread keeps only the Jacobians of its rows across the look-back and
// evaluates the gates a second time for the gradients: one more cell
// evaluation per element buys twice the resident CTAs (64 registers and 8 CTAs
// per SM for bf16; 5 for fp32, whose 40 KB of tiles allow no more).
template <typename TS> constexpr int bw_min_blocks() { return sizeof(TS) == 2 ? 8 : 5; }

// PLAN: the chunks of a pack are segment-aligned, taken from a.plan (last
// chunks of the segments first).
template <typename TS, bool EARLY, bool PLAN>
__global__ void __launch_bounds__(NW * 32, bw_min_blocks<TS>())
    k_backward(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmH,
               const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmGP,
               const BackwardArgs a) {
    extern __shared__ __align__(128) unsigned char dsmem[];
    TS *Ps = reinterpret_cast<TS *>(dsmem);   // [3][L][U]
    TS *Hs = Ps + 3 * L * U;                  // [L][U] trajectory
    TS *Gs = Hs + L * U;                      // [L][U] dL/dH
    __shared__ float s_aggA[NW][32], s_aggB[NW][32];
    __shared__ float s_C[32];
    __shared__ float s_red[6][NW][32];
    __shared__ uint32_t s_heads[L / 32];
    __shared__ __align__(8) uint64_t s_bar;
    // this CTA's ticket: chunk (position in its look-back chain), batch row,
    // unit tile, first row, end of the rows it may write, chain index of the
    // look-back slots
    __shared__ int s_tile[PLAN ? 6 : 3];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        const uint32_t ticket = atomicAdd(a.ticket, 1u);
        if constexpr (PLAN) {
            // segment-aligned chunks, the last ones of the segments first; the
            // grid is sized for an upper bound of their number
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
            const uint32_t rem = ticket % per_chunk;
            s_tile[0] = a.n_chunks - 1 - static_cast<int>(ticket / per_chunk);   // last chunk first
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
    // t_end: rows at or past it are outside this tile's sequence; the chain
    // holds chunks 0 .. n_chain - 1, the slot of chunk c + d lies d slots on
    const int t0 = PLAN ? s_tile[3] : c * L, t_end = PLAN ? s_tile[4] : a.T;
    const int n_chain = PLAN ? c + (t_end - t0 + L - 1) / L : a.n_chunks;
    const int u0 = ut * U;
    const int tile = (b * a.n_ut + ut) * a.n_chunks + (PLAN ? s_tile[5] : c);
    unsigned long long *slot = a.slots + static_cast<size_t>(tile) * 32 + lane;

    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&s_bar, 5u * L * U * sizeof(TS));
#pragma unroll
        for (int g = 0; g < 3; ++g) tma_load_3d(Ps + g * L * U, &tmP, &s_bar, g * a.d_h + u0, t0, b);
        tma_load_3d(Hs, &tmH, &s_bar, u0, t0, b);
        tma_load_3d(Gs, &tmG, &s_bar, u0, t0, b);
        if constexpr (PLAN) {
            if (c == 0) s_heads[0] = 1u;   // a segment's first chunk starts at its head
        } else {
            mark_heads(a.cu, a.S, t0, L, s_heads);
        }
    }
    const int u = u0 + lane;
    const bool uok = u < a.d_h;
    const UnitParams up = load_unit_params(a.params, a.d_h, u, uok);
    const typename BwCell<TS>::Params q = BwCell<TS>::make(up);
    const float2 a_z = splat2(up.a_z), a_r = splat2(up.a_r), a_c = splat2(up.a_c);
    const int r0 = warp * SEG;
    float hb = 0.f;   // H at row r0 - 1
    if (warp == 0 && t0 > 0 && uok)
        hb = to_f32(reinterpret_cast<const TS *>(a.H)[(static_cast<size_t>(b) * a.T + t0 - 1) * a.d_h + u]);
    __syncthreads();
    mbar_wait_bounded(&s_bar, 0, a.wait_ns, a.error);
    if (warp > 0) hb = to_f32(Hs[(r0 - 1) * U + lane]);
    const uint32_t hm = (s_heads[r0 >> 5] >> (r0 & 31)) & ((1u << SEG) - 1u);
    const int nvalid = min(SEG, t_end - (t0 + r0));

    // Each thread takes its 16 rows as 8 pairs (i, i + 8) on packed f32x2
    // arithmetic: .x the lower half of the warp's rows, .y the upper half.
    // Shifted state of row r (0 at a head); H at row r0 - 1 is hb.
    auto shifted = [&](int i) {
        if ((hm >> i) & 1u) return 0.f;
        return i == 0 ? hb : to_f32(Hs[(r0 + i - 1) * U + lane]);
    };
    // per-row derivatives at (h~ = H_{t-1}, P_t) of both rows of pair i (read
    // from the P tile before the gradient loop overwrites them)
    auto row_derivs = [&](int i) {
        const int rl = r0 + i, ru = rl + HALF;
        const float2 hs = make_float2(shifted(i), shifted(i + HALF));
        const float2 pz = make_float2(to_f32(Ps[(0 * L + rl) * U + lane]), to_f32(Ps[(0 * L + ru) * U + lane]));
        const float2 pr = make_float2(to_f32(Ps[(1 * L + rl) * U + lane]), to_f32(Ps[(1 * L + ru) * U + lane]));
        const float2 pc = make_float2(to_f32(Ps[(2 * L + rl) * U + lane]), to_f32(Ps[(2 * L + ru) * U + lane]));
        return derivs2<TS>(hs, pz, pr, pc, q, a_z, a_r, a_c);
    };
    // J = 0 at a head and past the end
    float2 Jr[HALF];
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
        const float2 J = row_derivs(i).J;
        Jr[i] = make_float2(((hm >> i) & 1u) || i >= nvalid ? 0.f : J.x,
                            ((hm >> (i + HALF)) & 1u) || i + HALF >= nvalid ? 0.f : J.y);
    }

    // compose nu_{t+1} -> nu_t = J_t nu_{t+1} + J_t gH_t over each half, last
    // row first, then the lower half after the upper one
    float2 A2 = splat2(1.0f), B2 = splat2(0.0f);
#pragma unroll
    for (int i = HALF - 1; i >= 0; --i) {
        const float2 gh = make_float2(i < nvalid ? to_f32(Gs[(r0 + i) * U + lane]) : 0.f,
                                      i + HALF < nvalid ? to_f32(Gs[(r0 + i + HALF) * U + lane]) : 0.f);
        B2 = fma2(Jr[i], B2, mul2(Jr[i], gh));
        A2 = mul2(A2, Jr[i]);
    }
    // warp 0 reads the slots of chunks c + 1 and c + 2 before the barrier
    unsigned long long pre1 = SLOT_EMPTY, pre2 = SLOT_EMPTY;
    if (EARLY && warp == 0) {
        if (c + 1 < n_chain) pre1 = ld_relaxed_u64(slot + 32);
        if (c + 2 < n_chain) pre2 = ld_relaxed_u64(slot + 64);
    }
    s_aggA[warp][lane] = A2.x * A2.y;
    s_aggB[warp][lane] = fmaf(A2.x, B2.y, B2.x);
    __syncthreads();

    // carry into this warp from the later warps of the chunk
    float eA = 1.f, eB = 0.f;
    for (int w = NW - 1; w > warp; --w) {
        eB = fmaf(s_aggA[w][lane], eB, s_aggB[w][lane]);
        eA *= s_aggA[w][lane];
    }
    if (warp == 0) {
        float tA = 1.f, tB = 0.f;
#pragma unroll
        for (int w = NW - 1; w >= 0; --w) {
            tB = fmaf(s_aggA[w][lane], tB, s_aggB[w][lane]);
            tA *= s_aggA[w][lane];
        }
        float C = 0.f;   // nu at the first step after the chunk
        if (c == n_chain - 1) {
            publish(slot, 0.f, tB);
        } else {
            publish(slot, tA, tB);
            C = lookback_lane<4>(slot, c, +1, n_chain, a.wait_ns, a.error, pre1, pre2);
            publish(slot, 0.f, fmaf(tA, C, tB));
        }
        s_C[lane] = C;
    }
    __syncthreads();

    // lambda_t = gH_t + nu_{t+1}; nu_t = J_t lambda_t; gradients.  nu enters the
    // upper half from the later warps and the lower half from the upper half.
    const float nu_hi = fmaf(eA, s_C[lane], eB);
    float2 nu = make_float2(fmaf(A2.y, nu_hi, B2.y), nu_hi);
    float2 g_az = splat2(0.f), g_ar = splat2(0.f), g_ac = splat2(0.f);
    float2 g_bz = splat2(0.f), g_br = splat2(0.f), g_bc = splat2(0.f);
#pragma unroll
    for (int i = HALF - 1; i >= 0; --i) {
        const bool vl = i < nvalid, vu = i + HALF < nvalid;
        const float2 lam = make_float2(vl ? to_f32(Gs[(r0 + i) * U + lane]) + nu.x : 0.f,
                                       vu ? to_f32(Gs[(r0 + i + HALF) * U + lane]) + nu.y : 0.f);
        nu = mul2(Jr[i], lam);
        const float2 hs = make_float2(shifted(i), shifted(i + HALF));
        const Derivs2 d = row_derivs(i);   // the gate factors again
        const float2 gz = mul2(lam, d.dz), gr = mul2(lam, d.dr), gc = mul2(lam, d.dc);
        g_bz = add2(g_bz, gz);
        g_br = add2(g_br, gr);
        g_bc = add2(g_bc, gc);
        g_az = fma2(gz, hs, g_az);
        g_ar = fma2(gr, hs, g_ar);
        g_ac = fma2(gc, d.rh, g_ac);
        // dL/dP of both rows goes into the P tile, whose values are no longer
        // read (rows past T and units past d_h are clipped by the store)
        const int rl = r0 + i, ru = rl + HALF;
        Ps[(0 * L + rl) * U + lane] = from_f32<TS>(gz.x);
        Ps[(1 * L + rl) * U + lane] = from_f32<TS>(gr.x);
        Ps[(2 * L + rl) * U + lane] = from_f32<TS>(gc.x);
        Ps[(0 * L + ru) * U + lane] = from_f32<TS>(gz.y);
        Ps[(1 * L + ru) * U + lane] = from_f32<TS>(gr.y);
        Ps[(2 * L + ru) * U + lane] = from_f32<TS>(gc.y);
    }
    s_red[0][warp][lane] = g_az.x + g_az.y;
    s_red[1][warp][lane] = g_ar.x + g_ar.y;
    s_red[2][warp][lane] = g_ac.x + g_ac.y;
    s_red[3][warp][lane] = g_bz.x + g_bz.y;
    s_red[4][warp][lane] = g_br.x + g_br.y;
    s_red[5][warp][lane] = g_bc.x + g_bc.y;
    fence_proxy_async_smem();   // the staged dL/dP is visible to the TMA store
    __syncthreads();
    // a segment's short last chunk: the rows after it belong to the next
    // segment, so its rows of dL/dP are stored one by one
    const bool rowwise = PLAN && t_end - t0 < L;
    if (rowwise) {
        if (uok) {
            TS *o = static_cast<TS *>(a.gP) + static_cast<size_t>(t0) * 3 * a.d_h + u;
            for (int r = warp; r < t_end - t0; r += NW)
#pragma unroll
                for (int g = 0; g < 3; ++g)
                    o[static_cast<size_t>(r) * 3 * a.d_h + g * a.d_h] = Ps[(g * L + r) * U + lane];
        }
    } else if (tid == 0) {
#pragma unroll
        for (int g = 0; g < 3; ++g) tma_store_4d(&tmGP, Ps + g * L * U, u0, g, t0, b);
        bulk_commit();
    }
    if (uok) {   // warp w sums gate-parameters w, w + NW, ... over the NW warps
        for (int g = warp; g < 6; g += NW) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += s_red[g][w][lane];
            atomicAdd(a.gparams + g * a.d_h + u, s);
        }
    }
    if (tid == 0 && !rowwise) bulk_wait_read<0>();   // the tile outlives the store's reads
}

template <typename TS, bool EARLY, bool PLAN>
cudaError_t launch_bw(const CUtensorMap &tmP, const CUtensorMap &tmH, const CUtensorMap &tmG,
                      const CUtensorMap &tmGP, const BackwardArgs &a, int64_t n_ctas,
                      cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    constexpr size_t smem = static_cast<size_t>(5) * L * U * sizeof(TS);
    cudaError_t e = once_per_device(configured, [](int) {
        return cudaFuncSetAttribute(k_backward<TS, EARLY, PLAN>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    });
    if (e != cudaSuccess) return e;
    k_backward<TS, EARLY, PLAN><<<static_cast<unsigned>(n_ctas), NW * 32, smem, stream>>>(
        tmP, tmH, tmG, tmGP, a);
    return cudaGetLastError();
}

// the early reads pay when at most 4 chunks per column are resident at once;
// a segment-aligned pack has one column per segment and unit tile
bool bw_early(const BackwardArgs &a, bool plan, int ctas_per_sm) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    return static_cast<int64_t>(sms) * ctas_per_sm <= 4 * static_cast<int64_t>(plan ? a.S : a.B) * a.n_ut;
}

template <typename TS>
cudaError_t launch_bw(const CUtensorMap &tmP, const CUtensorMap &tmH, const CUtensorMap &tmG,
                      const CUtensorMap &tmGP, const BackwardArgs &a, int64_t n_ctas,
                      cudaStream_t stream, bool plan) {
    const bool early = bw_early(a, plan, bw_min_blocks<TS>());
    if (plan)
        return early ? launch_bw<TS, true, true>(tmP, tmH, tmG, tmGP, a, n_ctas, stream)
                     : launch_bw<TS, false, true>(tmP, tmH, tmG, tmGP, a, n_ctas, stream);
    return early ? launch_bw<TS, true, false>(tmP, tmH, tmG, tmGP, a, n_ctas, stream)
                 : launch_bw<TS, false, false>(tmP, tmH, tmG, tmGP, a, n_ctas, stream);
}

}  // namespace

cudaError_t launch_backward(int dtype, const CUtensorMap &tmP, const CUtensorMap &tmH,
                            const CUtensorMap &tmG, const CUtensorMap &tmGP, const BackwardArgs &a,
                            int64_t n_ctas, cudaStream_t stream, bool plan) {
    if (dtype == 1) return launch_bw<__nv_bfloat16>(tmP, tmH, tmG, tmGP, a, n_ctas, stream, plan);
    return launch_bw<float>(tmP, tmH, tmG, tmGP, a, n_ctas, stream, plan);
}

}  // namespace nrnn

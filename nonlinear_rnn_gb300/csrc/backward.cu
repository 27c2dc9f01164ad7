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
// each thread composes the maps nu_{t+1} -> nu_t = (J_t, J_t gH_t) of its rows
// from the last upwards; warp aggregates meet in shared memory; warp 0
// publishes the chunk aggregate and completes a decoupled look-back over
// LATER chunks (tickets are handed out from the last chunk backwards, so every
// chunk waited for has started); the carry nu at the chunk end is then applied
// and dL/dP written.  Parameter gradients are reduced over the CTA and added
// with one atomicAdd per (gate, unit).  Every wait is bounded.
#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

namespace {

constexpr int NW = NEWTON_NW;
constexpr int SEG = NEWTON_SEG;
constexpr int L = NEWTON_L;
constexpr int U = TILE_U;

template <typename TS>
__global__ void __launch_bounds__(NW * 32, 4)
    k_backward(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmH,
               const __grid_constant__ CUtensorMap tmG, const BackwardArgs a) {
    extern __shared__ __align__(128) unsigned char dsmem[];
    TS *Ps = reinterpret_cast<TS *>(dsmem);   // [3][L][U]
    TS *Hs = Ps + 3 * L * U;                  // [L][U] trajectory
    TS *Gs = Hs + L * U;                      // [L][U] dL/dH
    __shared__ float s_aggA[NW][32], s_aggB[NW][32];
    __shared__ float s_C[32];
    __shared__ float s_red[6][NW][32];
    __shared__ uint32_t s_heads[L / 32];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ int s_tile[3];   // chunk, batch row, unit tile of this CTA's ticket

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        const uint32_t ticket = atomicAdd(a.ticket, 1u);
        const uint32_t per_chunk = static_cast<uint32_t>(a.B) * a.n_ut;
        const uint32_t rem = ticket % per_chunk;
        s_tile[0] = a.n_chunks - 1 - static_cast<int>(ticket / per_chunk);   // last chunk first
        s_tile[1] = static_cast<int>(rem / a.n_ut);
        s_tile[2] = static_cast<int>(rem % a.n_ut);
    }
    if (tid < L / 32) s_heads[tid] = 0u;
    __syncthreads();

    const int c = s_tile[0], b = s_tile[1], ut = s_tile[2];
    const int t0 = c * L, u0 = ut * U;

    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&s_bar, 5u * L * U * sizeof(TS));
#pragma unroll
        for (int g = 0; g < 3; ++g) tma_load_3d(Ps + g * L * U, &tmP, &s_bar, g * a.d_h + u0, t0, b);
        tma_load_3d(Hs, &tmH, &s_bar, u0, t0, b);
        tma_load_3d(Gs, &tmG, &s_bar, u0, t0, b);
        mark_heads(a.cu, a.S, t0, L, s_heads);
    }
    const int u = u0 + lane;
    const bool uok = u < a.d_h;
    const UnitParams up = load_unit_params(a.params, a.d_h, u, uok);
    const ScaledParams prm = scale_params(up);
    const int r0 = warp * SEG;
    float hb = 0.f;   // H at row r0 - 1
    if (warp == 0 && t0 > 0 && uok)
        hb = to_f32(reinterpret_cast<const TS *>(a.H)[(static_cast<size_t>(b) * a.T + t0 - 1) * a.d_h + u]);
    __syncthreads();
    mbar_wait_bounded(&s_bar, 0, a.wait_ns, a.error);
    if (warp > 0) hb = to_f32(Hs[(r0 - 1) * U + lane]);
    const uint32_t hm = (s_heads[r0 >> 5] >> (r0 & 31)) & ((1u << SEG) - 1u);
    const int nvalid = min(SEG, a.T - (t0 + r0));

    // per-row derivatives at (h~ = H_{t-1}, P_t)
    float Jr[SEG], dz[SEG], dr[SEG], dc[SEG], rh[SEG];
    {
        float hprev = hb;
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            const int r = r0 + i;
            const bool head = (hm >> i) & 1u;
            const float hs = head ? 0.f : hprev;
            float sz, sr, sc;
            scale_preact(to_f32(Ps[(0 * L + r) * U + lane]), to_f32(Ps[(1 * L + r) * U + lane]),
                         to_f32(Ps[(2 * L + r) * U + lane]), prm, sz, sr, sc);
            float z, rg, cg;
            gates_scaled(hs, sz, sr, sc, prm, z, rg, cg);
            const float omz = 1.0f - z;
            const float cmh = cg - hs;
            const float omc2 = fmaf(-cg, cg, 1.0f);
            const float dPc = z * omc2;
            const float rr = fmaf(-rg, rg, rg);
            const float dq = fmaf(hs * up.a_r, rr, rg);
            float J = fmaf(z, fmaf(omz * up.a_z, cmh, omc2 * up.a_c * dq), omz);
            if (head || i >= nvalid) J = 0.f;   // no flow across a head or past the end
            Jr[i] = J;
            dz[i] = z * omz * cmh;
            dc[i] = dPc;
            dr[i] = dPc * up.a_c * hs * rr;
            rh[i] = rg * hs;
            hprev = to_f32(Hs[r * U + lane]);
        }
    }

    // compose nu_{t+1} -> nu_t = J_t nu_{t+1} + J_t gH_t over this warp's rows, last first
    float A = 1.f, Bv = 0.f;
#pragma unroll
    for (int i = SEG - 1; i >= 0; --i) {
        const float gh = (i < nvalid) ? to_f32(Gs[(r0 + i) * U + lane]) : 0.f;
        Bv = fmaf(Jr[i], Bv, Jr[i] * gh);
        A *= Jr[i];
    }
    s_aggA[warp][lane] = A;
    s_aggB[warp][lane] = Bv;
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
        const int tile = (b * a.n_ut + ut) * a.n_chunks + c;
        unsigned long long *slot = a.slots + static_cast<size_t>(tile) * 32 + lane;
        float C = 0.f;   // nu at the first step after the chunk
        if (c == a.n_chunks - 1) {
            publish(slot, 0.f, tB);
        } else {
            publish(slot, tA, tB);
            C = lookback_lane(slot, c, +1, a.n_chunks, a.wait_ns, a.error);
            publish(slot, 0.f, fmaf(tA, C, tB));
        }
        s_C[lane] = C;
    }
    __syncthreads();

    // lambda_t = gH_t + nu_{t+1}; nu_t = J_t lambda_t; gradients
    float nu = fmaf(eA, s_C[lane], eB);
    float g_az = 0.f, g_ar = 0.f, g_ac = 0.f, g_bz = 0.f, g_br = 0.f, g_bc = 0.f;
    TS *gP = reinterpret_cast<TS *>(a.gP);
#pragma unroll
    for (int i = SEG - 1; i >= 0; --i) {
        if (i >= nvalid) continue;
        const int r = r0 + i;
        const float lam = to_f32(Gs[r * U + lane]) + nu;
        nu = Jr[i] * lam;
        const float hs = ((hm >> i) & 1u) ? 0.f : (i == 0 ? hb : to_f32(Hs[(r - 1) * U + lane]));
        const float gz = lam * dz[i], gr = lam * dr[i], gc = lam * dc[i];
        g_bz += gz;
        g_br += gr;
        g_bc += gc;
        g_az = fmaf(gz, hs, g_az);
        g_ar = fmaf(gr, hs, g_ar);
        g_ac = fmaf(gc, rh[i], g_ac);
        if (uok) {
            TS *o = gP + (static_cast<size_t>(b) * a.T + t0 + r) * 3 * a.d_h + u;
            o[0] = from_f32<TS>(gz);
            o[a.d_h] = from_f32<TS>(gr);
            o[2 * a.d_h] = from_f32<TS>(gc);
        }
    }
    s_red[0][warp][lane] = g_az;
    s_red[1][warp][lane] = g_ar;
    s_red[2][warp][lane] = g_ac;
    s_red[3][warp][lane] = g_bz;
    s_red[4][warp][lane] = g_br;
    s_red[5][warp][lane] = g_bc;
    __syncthreads();
    if (uok) {   // warp w sums gate-parameters w, w + NW, ... over the NW warps
        for (int g = warp; g < 6; g += NW) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += s_red[g][w][lane];
            atomicAdd(a.gparams + g * a.d_h + u, s);
        }
    }
}

template <typename TS>
cudaError_t launch_bw(const CUtensorMap &tmP, const CUtensorMap &tmH, const CUtensorMap &tmG,
                      const BackwardArgs &a, int64_t n_ctas, cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    constexpr size_t smem = static_cast<size_t>(5) * L * U * sizeof(TS);
    cudaError_t e = once_per_device(configured, [](int) {
        return cudaFuncSetAttribute(k_backward<TS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    if (e != cudaSuccess) return e;
    k_backward<TS><<<static_cast<unsigned>(n_ctas), NW * 32, smem, stream>>>(tmP, tmH, tmG, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(int dtype, const CUtensorMap &tmP, const CUtensorMap &tmH,
                            const CUtensorMap &tmG, const BackwardArgs &a, int64_t n_ctas,
                            cudaStream_t stream) {
    if (dtype == 1) return launch_bw<__nv_bfloat16>(tmP, tmH, tmG, a, n_ctas, stream);
    return launch_bw<float>(tmP, tmH, tmG, a, n_ctas, stream);
}

}  // namespace nrnn

// Decode: one T = 1 step of the diagonal-mix GRU per slot, with the recurrent
// state carried between calls in a fixed (slots, d_h) buffer (pararnn-torch
// FAQs, "How do I pass recurrent state between decode steps?": a carry of
// size (slots, d_h), prefill then decode_wx + decode_step(..., out=) per token).
//
// k_decode_step: h_out = f(h_in, P) elementwise from given preactivations
// (k_decode_step_vec: the same on vectors of 4 units when shapes and
// alignment allow).
// k_decode_step_x: the same step with the input projection fused in, for
// small slot counts (a batched matrix-vector product per step; see below).
// k_decode_step_xtc: the same for bf16 on the tensor cores (see below).
// Every decode kernel evaluates the cell in the storage type's formulation,
// as the Newton kernels do: ex2/rcp for fp32, tanh.approx for bf16.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "nrnn_device.cuh"
#include "nrnn_internal.h"
#include "tcgen05.cuh"

namespace nrnn {

namespace {

template <typename TS>
__global__ void __launch_bounds__(256)
    k_decode_step(const TS *__restrict__ P, const float *__restrict__ params,
                  const TS *__restrict__ h_in, TS *__restrict__ h_out, int slots, int d_h) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(slots) * d_h) return;
    const int s = static_cast<int>(i / d_h), j = static_cast<int>(i - static_cast<int64_t>(s) * d_h);
    const UnitParams prm = load_unit_params(params, d_h, j, true);
    const TS *p = P + static_cast<int64_t>(s) * 3 * d_h + j;
    const float h = (h_in != nullptr) ? to_f32(h_in[i]) : 0.f;
    h_out[i] = from_f32<TS>(cell_f_storage<TS>(h, to_f32(p[0]), to_f32(p[d_h]), to_f32(p[2 * d_h]), prm));
}

__device__ __forceinline__ void unpack16(const uint4 &v, float (&o)[4]) {
    o[0] = __uint_as_float(v.x);
    o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z);
    o[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const uint4 &v, float (&o)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ void unpack8(const uint2 &v, float (&o)[4]) {
    o[0] = __uint_as_float(v.x << 16);
    o[1] = __uint_as_float(v.x & 0xffff0000u);
    o[2] = __uint_as_float(v.y << 16);
    o[3] = __uint_as_float(v.y & 0xffff0000u);
}
// The same step on vectors: a thread takes 4 adjacent units of one slot row
// (16-byte fp32 or 8-byte bf16 loads), keeps their parameters in registers
// and walks the slots with a stride of `lanes`, two slots per pass, so that
// eight loads are in flight and the parameters are read once per thread, not
// once per slot.  Four bf16 units rather than eight keep a thread at 64
// registers, so that 4 CTAs of 256 threads fit on an SM.  Needs d_h a
// multiple of 4 and 16-byte aligned P, params, h_in and h_out.
template <typename TS>
__global__ void __launch_bounds__(256)
    k_decode_step_vec(const TS *__restrict__ P, const float *__restrict__ params,
                      const TS *__restrict__ h_in, TS *__restrict__ h_out, int slots, int d_h,
                      int lanes) {
    constexpr int VEC = 4;
    using V = typename std::conditional<sizeof(TS) == 2, uint2, uint4>::type;
    const int groups = d_h / VEC;
    const int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (v >= static_cast<int64_t>(lanes) * groups) return;
    const int s_first = static_cast<int>(v / groups);
    const int j0 = static_cast<int>(v - static_cast<int64_t>(s_first) * groups) * VEC;
    float prm[6][VEC];
#pragma unroll
    for (int g = 0; g < 6; ++g) {
        const float4 w = *reinterpret_cast<const float4 *>(params + g * d_h + j0);
        prm[g][0] = w.x;
        prm[g][1] = w.y;
        prm[g][2] = w.z;
        prm[g][3] = w.w;
    }
    const V zero{};
    for (int64_t s = s_first; s < slots; s += 2 * static_cast<int64_t>(lanes)) {
        const bool two = s + lanes < slots;
        V in[2][4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int64_t sk = s + k * lanes;
            if (k == 0 || two) {
                const TS *p = P + sk * 3 * d_h + j0;
                in[k][0] = *reinterpret_cast<const V *>(p);
                in[k][1] = *reinterpret_cast<const V *>(p + d_h);
                in[k][2] = *reinterpret_cast<const V *>(p + 2 * d_h);
                in[k][3] = (h_in != nullptr) ? *reinterpret_cast<const V *>(h_in + sk * d_h + j0) : zero;
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (k == 1 && !two) break;
            float z[VEC], r[VEC], c[VEC], h[VEC];
            if constexpr (sizeof(TS) == 2) {
                unpack8(in[k][0], z);
                unpack8(in[k][1], r);
                unpack8(in[k][2], c);
                unpack8(in[k][3], h);
            } else {
                unpack16(in[k][0], z);
                unpack16(in[k][1], r);
                unpack16(in[k][2], c);
                unpack16(in[k][3], h);
            }
            __align__(16) TS o[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const UnitParams up{prm[0][e], prm[1][e], prm[2][e], prm[3][e], prm[4][e], prm[5][e]};
                o[e] = from_f32<TS>(cell_f_storage<TS>(h[e], z[e], r[e], c[e], up));
            }
            *reinterpret_cast<V *>(h_out + (s + k * lanes) * d_h + j0) = *reinterpret_cast<const V *>(o);
        }
    }
}

// k_decode_step_x: a CTA takes DX_UNITS units (one warp each) and a group of
// DX_SLOTS slots whose x rows it stages in shared memory once (or reads from
// global memory when they do not fit); each lane accumulates 16-byte slices of
// d_in for the three gate rows of its warp's unit against every slot of the
// group, so a W_x row is read once per slot group, not once per slot.  After
// the shuffle reduction lane s applies the cell to slot s.
constexpr int DX_UNITS = 8;
constexpr int DX_SLOTS = 8;
constexpr size_t DX_SMEM_MAX = 48 * 1024;

template <typename TS>
__global__ void __launch_bounds__(DX_UNITS * 32)
    k_decode_step_x(const TS *__restrict__ x, const TS *__restrict__ W, const float *__restrict__ params,
                    const TS *__restrict__ h_in, TS *__restrict__ h_out, int slots, int d_in,
                    int d_h, int stage_x) {
    constexpr int VEC = 16 / sizeof(TS);   // elements per 16-byte load
    extern __shared__ __align__(16) unsigned char dx_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = blockIdx.x * DX_UNITS + warp;
    const int s0 = blockIdx.y * DX_SLOTS;
    const int ns = min(DX_SLOTS, slots - s0);
    const TS *xg = x + static_cast<int64_t>(s0) * d_in;
    const TS *xs = xg;
    if (stage_x) {
        uint4 *dst = reinterpret_cast<uint4 *>(dx_smem);
        const uint4 *src = reinterpret_cast<const uint4 *>(xg);
        const int nvec = ns * d_in / VEC;
        for (int i = threadIdx.x; i < nvec; i += blockDim.x) dst[i] = src[i];
        __syncthreads();
        xs = reinterpret_cast<const TS *>(dx_smem);
    }
    if (j >= d_h) return;
    float acc[3][DX_SLOTS];
#pragma unroll
    for (int g = 0; g < 3; ++g)
#pragma unroll
        for (int s = 0; s < DX_SLOTS; ++s) acc[g][s] = 0.f;
    const TS *wr[3] = {W + static_cast<int64_t>(j) * d_in, W + static_cast<int64_t>(d_h + j) * d_in,
                       W + static_cast<int64_t>(2 * d_h + j) * d_in};
    for (int k = lane * VEC; k < d_in; k += 32 * VEC) {
        float wv[3][VEC];
#pragma unroll
        for (int g = 0; g < 3; ++g) unpack16(__ldg(reinterpret_cast<const uint4 *>(wr[g] + k)), wv[g]);
#pragma unroll
        for (int s = 0; s < DX_SLOTS; ++s) {
            if (s >= ns) break;
            float xv[VEC];
            unpack16(*reinterpret_cast<const uint4 *>(xs + s * d_in + k), xv);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
#pragma unroll
                for (int g = 0; g < 3; ++g) acc[g][s] = fmaf(xv[e], wv[g][e], acc[g][s]);
        }
    }
#pragma unroll
    for (int g = 0; g < 3; ++g)
#pragma unroll
        for (int s = 0; s < DX_SLOTS; ++s)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[g][s] += __shfl_xor_sync(FULL_MASK, acc[g][s], o);
    // lane s applies the cell to slot s0 + s; the preactivation is stored in TS
    // before the cell reads it, as on the projection path
    float pz = 0.f, pr = 0.f, pc = 0.f;
#pragma unroll
    for (int s = 0; s < DX_SLOTS; ++s)
        if (lane == s) {
            pz = acc[0][s];
            pr = acc[1][s];
            pc = acc[2][s];
        }
    if (lane < ns) {
        const int64_t i = static_cast<int64_t>(s0 + lane) * d_h + j;
        const float h = (h_in != nullptr) ? to_f32(h_in[i]) : 0.f;
        h_out[i] = from_f32<TS>(cell_f_storage<TS>(h, round_to<TS>(pz), round_to<TS>(pr), round_to<TS>(pc),
                                       load_unit_params(params, d_h, j, true)));
    }
}

// k_decode_step_xtc (bf16): the projection of a small batch of slots on the
// tensor cores, the step in the epilogue.  A CTA takes UNITS units (32, or 8
// when that leaves too few CTAs to keep W_x streaming from HBM) and 64 slots:
// D = W_tile x_tile^T with M = 128 TMEM lanes (gate g's UNITS rows of W_x at
// rows 32 g ..; the other rows unused), N = 64 slots, K = d_in in 64-wide
// slices through a ring of TMA stages (128-byte swizzle; rows past the slots
// or units and columns past d_in are zero-filled).  Warps 0..2 then read their
// gate's lanes (lane = unit, registers = slots), round them to bf16 as a
// stored preactivation would be, and pass them through shared memory; every
// thread applies the cell to (slot, unit) pairs, adjacent units of a slot on
// adjacent lanes.  A wait that gives up writes NaN.
constexpr int XT_SLOTS = 64;
constexpr int XT_BK = 64;
constexpr int XT_STAGES = 8;
constexpr int XT_A_BYTES = 128 * XT_BK * 2;                 // M = 128 rows
constexpr int XT_B_BYTES = XT_SLOTS * XT_BK * 2;
constexpr int XT_STAGE_BYTES = XT_A_BYTES + XT_B_BYTES;     // 24 KiB
constexpr uint32_t XT_TMEM_COLS = XT_SLOTS;
constexpr uint32_t XT_IDESC = idesc_kmajor<false>(128, XT_SLOTS);
constexpr uint64_t XT_WAIT_NS = 2000000000ull;
static_assert(XT_STAGES * XT_STAGE_BYTES >= 3 * XT_SLOTS * 32 * 4,
              "the gate values must fit in the stage ring");

template <int UNITS>
__global__ void __launch_bounds__(128)
    k_decode_step_xtc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const float *__restrict__ params, const __nv_bfloat16 *__restrict__ h_in,
                      __nv_bfloat16 *__restrict__ h_out, int slots, int d_in, int d_h) {
    constexpr int W_BOX_BYTES = UNITS * XT_BK * 2;   // one gate's UNITS rows of W_x
    extern __shared__ unsigned char xt_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(xt_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[XT_STAGES], empty_bar[XT_STAGES], acc_bar;
    __shared__ uint32_t s_tmem, s_err;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int u0 = blockIdx.x * UNITS, s0 = blockIdx.y * XT_SLOTS;
    const int kt_count = (d_in + XT_BK - 1) / XT_BK;
    if (tid == 0) {
        for (int i = 0; i < XT_STAGES; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        mbar_init(&acc_bar, 1);
        s_err = 0u;
        fence_mbar_init();
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(XT_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;
    if (warp == 0 && lane == 0) {
        // TMA producer: the three gates' W_x rows of this unit tile, x rows of these slots
        for (int kt = 0; kt < kt_count; ++kt) {
            const int st = kt % XT_STAGES;
            if (kt >= XT_STAGES)
                mbar_wait_bounded(&empty_bar[st], ((kt / XT_STAGES) - 1) & 1, XT_WAIT_NS, &s_err);
            unsigned char *A = smem + st * XT_STAGE_BYTES;
            mbar_arrive_expect_tx(&full_bar[st], 3 * W_BOX_BYTES + XT_B_BYTES);
#pragma unroll
            for (int g = 0; g < 3; ++g)   // gate g at rows 32 g (32 rows x 128 bytes apart)
                tma_load_2d(A + g * 32 * XT_BK * 2, &tmW, &full_bar[st], kt * XT_BK, g * d_h + u0);
            tma_load_2d(A + XT_A_BYTES, &tmX, &full_bar[st], kt * XT_BK, s0);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        for (int kt = 0; kt < kt_count; ++kt) {
            const int st = kt % XT_STAGES;
            mbar_wait_bounded(&full_bar[st], (kt / XT_STAGES) & 1, XT_WAIT_NS, &s_err);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t A = smem_u32(smem + st * XT_STAGE_BYTES);
#pragma unroll
            for (int kk = 0; kk < XT_BK / 16; ++kk)
                mma<false, XT_IDESC>(tmem, sw128_desc(A + kk * 32), sw128_desc(A + XT_A_BYTES + kk * 32),
                                     (kt > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&empty_bar[st]);
        }
        mma_commit(&acc_bar);
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(&acc_bar, 0, XT_WAIT_NS, &s_err);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    fence_proxy_async_smem();   // the gate values overwrite the stages
    float *Pg = reinterpret_cast<float *>(smem);   // [3 gates][64 slots][UNITS units]
    if (warp < 3) {
#pragma unroll 1
        for (int cc = 0; cc < XT_SLOTS / 32; ++cc) {
            uint32_t v[32];
            tmem_ld_cols<32>(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc * 32, v);
            if (lane < UNITS) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    Pg[(warp * XT_SLOTS + cc * 32 + i) * UNITS + lane] =
                        ok ? round_to<__nv_bfloat16>(__uint_as_float(v[i])) : __int_as_float(0x7fffffff);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 2) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(XT_TMEM_COLS)
                     : "memory");
    }
    // the step: thread t takes unit u0 + t % UNITS of slots t / UNITS, + 128 / UNITS, ...
    const int ul = tid % UNITS, u = u0 + ul;
    if (u >= d_h) return;
    const UnitParams prm = load_unit_params(params, d_h, u, true);
#pragma unroll 4
    for (int s = tid / UNITS; s < XT_SLOTS; s += 128 / UNITS) {
        const int slot = s0 + s;
        if (slot >= slots) break;
        const int64_t i = static_cast<int64_t>(slot) * d_h + u;
        const float h = (h_in != nullptr) ? to_f32(h_in[i]) : 0.f;
        h_out[i] = from_f32<__nv_bfloat16>(cell_f_storage<__nv_bfloat16>(h, Pg[(0 * XT_SLOTS + s) * UNITS + ul],
                                                  Pg[(1 * XT_SLOTS + s) * UNITS + ul],
                                                  Pg[(2 * XT_SLOTS + s) * UNITS + ul], prm));
    }
}

// k_decode_step_xtc_sk (bf16, one tile of at most 64 slots, 8-unit tiles):
// the same projection split along d_in over the KS CTAs of a thread-block
// cluster, for the small batches where one CTA per 8 units leaves most SMs
// idle and each CTA's K loop of d_in / 64 slices is the latency.  Rank r of
// the cluster accumulates the slices [r kt / KS, (r + 1) kt / KS) through a
// 2-stage ring, writes its fp32 partial sums (3 gates x 64 slots x 8 units)
// into its own shared memory, and after a cluster barrier sums the partials
// of all KS ranks for its quarter of the slots (distributed shared memory
// reads), rounds them to bf16 and applies the step.  No multicast: every CTA
// loads its own operand tiles.
constexpr int SK_UNITS = 8;
constexpr int SK_KS = 4;
constexpr int SK_STAGES = 2;
constexpr int SK_PART_FLOATS = 3 * XT_SLOTS * SK_UNITS;
static_assert(SK_STAGES * XT_STAGE_BYTES >= SK_PART_FLOATS * 4, "the partials fit in the ring");
static_assert(XT_SLOTS % SK_KS == 0 && (XT_SLOTS / SK_KS) * SK_UNITS == 128,
              "one (slot, unit) pair per thread in the epilogue");

__device__ __forceinline__ uint32_t sk_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float sk_ld_remote(const float *p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void sk_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(128)
    k_decode_step_xtc_sk(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                         const float *__restrict__ params, const __nv_bfloat16 *__restrict__ h_in,
                         __nv_bfloat16 *__restrict__ h_out, int slots, int d_in, int d_h) {
    constexpr int W_BOX_BYTES = SK_UNITS * XT_BK * 2;
    extern __shared__ unsigned char sk_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(sk_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[SK_STAGES], empty_bar[SK_STAGES], acc_bar;
    __shared__ uint32_t s_tmem, s_err;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = sk_rank();
    const int u0 = blockIdx.x * SK_UNITS;
    const int kt_all = (d_in + XT_BK - 1) / XT_BK;
    const int kt0 = static_cast<int>(rank) * kt_all / SK_KS;
    const int kt_count = (static_cast<int>(rank) + 1) * kt_all / SK_KS - kt0;
    if (tid == 0) {
        for (int i = 0; i < SK_STAGES; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        mbar_init(&acc_bar, 1);
        s_err = 0u;
        fence_mbar_init();
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(XT_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;
    if (kt_count > 0) {
        if (warp == 0 && lane == 0) {
            for (int k = 0; k < kt_count; ++k) {
                const int st = k % SK_STAGES, kt = kt0 + k;
                if (k >= SK_STAGES)
                    mbar_wait_bounded(&empty_bar[st], ((k / SK_STAGES) - 1) & 1, XT_WAIT_NS, &s_err);
                unsigned char *A = smem + st * XT_STAGE_BYTES;
                mbar_arrive_expect_tx(&full_bar[st], 3 * W_BOX_BYTES + XT_B_BYTES);
#pragma unroll
                for (int g = 0; g < 3; ++g)   // gate g at rows 32 g
                    tma_load_2d(A + g * 32 * XT_BK * 2, &tmW, &full_bar[st], kt * XT_BK, g * d_h + u0);
                tma_load_2d(A + XT_A_BYTES, &tmX, &full_bar[st], kt * XT_BK, 0);
            }
        } else if (warp == 1 && lane == 0) {
            for (int k = 0; k < kt_count; ++k) {
                const int st = k % SK_STAGES;
                mbar_wait_bounded(&full_bar[st], (k / SK_STAGES) & 1, XT_WAIT_NS, &s_err);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t A = smem_u32(smem + st * XT_STAGE_BYTES);
#pragma unroll
                for (int kk = 0; kk < XT_BK / 16; ++kk)
                    mma<false, XT_IDESC>(tmem, sw128_desc(A + kk * 32), sw128_desc(A + XT_A_BYTES + kk * 32),
                                         (k > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&empty_bar[st]);
            }
            mma_commit(&acc_bar);
        }
        __syncwarp();
    }
    const bool ok = kt_count == 0 || mbar_wait_bounded(&acc_bar, 0, XT_WAIT_NS, &s_err);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    fence_proxy_async_smem();   // the partials overwrite the stages
    float *part = reinterpret_cast<float *>(smem);   // [3 gates][64 slots][8 units]
    if (warp < 3) {
#pragma unroll 1
        for (int cc = 0; cc < XT_SLOTS / 32; ++cc) {
            uint32_t v[32];
            if (kt_count > 0) tmem_ld_cols<32>(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc * 32, v);
            if (lane < SK_UNITS) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    part[(warp * XT_SLOTS + cc * 32 + i) * SK_UNITS + lane] =
                        !ok ? __int_as_float(0x7fffffff) : (kt_count > 0 ? __uint_as_float(v[i]) : 0.f);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    // every rank's partials are complete and visible to the cluster (this also
    // makes sure every CTA of the cluster runs before any remote read)
    sk_cluster_sync();
    if (warp == 2) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(XT_TMEM_COLS)
                     : "memory");
    }
    // rank r finishes slots [16 r, 16 r + 16): thread t takes slot 16 r + t / 8, unit t % 8
    const int ul = tid % SK_UNITS, s = static_cast<int>(rank) * (XT_SLOTS / SK_KS) + tid / SK_UNITS;
    const int u = u0 + ul;
    if (u < d_h && s < slots) {
        float pg[3];
#pragma unroll
        for (int g = 0; g < 3; ++g) {
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < SK_KS; ++q)
                acc += sk_ld_remote(&part[(g * XT_SLOTS + s) * SK_UNITS + ul], static_cast<uint32_t>(q));
            pg[g] = round_to<__nv_bfloat16>(acc);
        }
        const int64_t i = static_cast<int64_t>(s) * d_h + u;
        const float h = (h_in != nullptr) ? to_f32(h_in[i]) : 0.f;
        h_out[i] = from_f32<__nv_bfloat16>(
            cell_f_storage<__nv_bfloat16>(h, pg[0], pg[1], pg[2], load_unit_params(params, d_h, u, true)));
    }
    // no CTA leaves while the others may still read its partials
    sk_cluster_sync();
}

// k_decode_step_xg (bf16, more slots than one 64-slot tile): the step's
// projection as a GEMM in the usual orientation, M = 128 slots and N = 192 =
// the z, r and c rows of W_x for 64 units (three TMA boxes of 64 rows, one per
// gate, stacked into one B tile), K = d_in through a 4-stage ring.  One
// persistent CTA per SM takes (slot tile, unit tile) pairs, unit tiles
// fastest (CTAs working at once share x tiles in L2), and keeps two TMEM
// accumulators: while the MMA thread fills one, four epilogue warps read the
// other (warp q: slots 32 q .. 32 q + 31 of the tile, one per lane), round
// the three gate preactivations to bf16 (the values the stored-P route reads)
// and apply the cell to h_in in groups of 8 units (16-byte loads and stores).
constexpr int XG_BM = 128;
constexpr int XG_UNITS = 64;
constexpr int XG_BN = 3 * XG_UNITS;
constexpr int XG_BK = 64;
constexpr int XG_STAGES = 4;
constexpr int XG_A_BYTES = XG_BM * XG_BK * 2;                       // 16 KiB
constexpr int XG_W_BOX_BYTES = XG_UNITS * XG_BK * 2;                // 8 KiB per gate
constexpr int XG_STAGE_BYTES = XG_A_BYTES + 3 * XG_W_BOX_BYTES;     // 40 KiB
constexpr uint32_t XG_ACC_STRIDE = 256;                             // TMEM columns per accumulator
constexpr uint32_t XG_TMEM_COLS = 2 * XG_ACC_STRIDE;
constexpr uint32_t XG_IDESC = idesc_kmajor<false>(XG_BM, XG_BN);
constexpr int XG_EPI_THREADS = 128;
constexpr size_t XG_SMEM = static_cast<size_t>(XG_STAGES) * XG_STAGE_BYTES + 1024;
static_assert(XG_STAGE_BYTES % 1024 == 0, "stages keep the 128-byte swizzle's 1024-byte alignment");

__global__ void __launch_bounds__(256, 1)
    k_decode_step_xg(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const float *__restrict__ params, const __nv_bfloat16 *__restrict__ h_in,
                     __nv_bfloat16 *__restrict__ h_out, int slots, int d_in, int d_h) {
    extern __shared__ unsigned char xg_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(xg_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[XG_STAGES], empty_bar[XG_STAGES], accf_bar[2],
        acce_bar[2];
    __shared__ uint32_t s_tmem, s_err;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = (d_h + XG_UNITS - 1) / XG_UNITS;
    const int n_tiles = ((slots + XG_BM - 1) / XG_BM) * tiles_n;
    const int kt_count = (d_in + XG_BK - 1) / XG_BK;
    if (threadIdx.x == 0) {
        for (int i = 0; i < XG_STAGES; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf_bar[b], 1);
            mbar_init(&acce_bar[b], XG_EPI_THREADS);
        }
        s_err = 0u;
        fence_mbar_init();
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(XG_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- TMA producer
        int it = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            const int m0 = (t / tiles_n) * XG_BM, n0 = (t % tiles_n) * XG_UNITS;
            for (int kt = 0; kt < kt_count; ++kt, ++it) {
                const int st = it % XG_STAGES;
                if (it >= XG_STAGES)
                    mbar_wait_bounded(&empty_bar[st], ((it / XG_STAGES) - 1) & 1, XT_WAIT_NS, &s_err);
                unsigned char *A = smem + st * XG_STAGE_BYTES;
                mbar_arrive_expect_tx(&full_bar[st], XG_STAGE_BYTES);
                tma_load_2d(A, &tmX, &full_bar[st], kt * XG_BK, m0);
#pragma unroll
                for (int g = 0; g < 3; ++g)   // gate g at rows 64 g of the B tile
                    tma_load_2d(A + XG_A_BYTES + g * XG_W_BOX_BYTES, &tmW, &full_bar[st], kt * XG_BK,
                                g * d_h + n0);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        int it = 0, j = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++j) {
            const int buf = j & 1;
            if (j >= 2) mbar_wait_bounded(&acce_bar[buf], ((j >> 1) - 1) & 1, XT_WAIT_NS, &s_err);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t d = tmem + buf * XG_ACC_STRIDE;
            for (int kt = 0; kt < kt_count; ++kt, ++it) {
                const int st = it % XG_STAGES;
                mbar_wait_bounded(&full_bar[st], (it / XG_STAGES) & 1, XT_WAIT_NS, &s_err);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t A = smem_u32(smem + st * XG_STAGE_BYTES);
#pragma unroll
                for (int kk = 0; kk < XG_BK / 16; ++kk)   // 32 bytes of K per MMA
                    mma<false, XG_IDESC>(d, sw128_desc(A + kk * 32), sw128_desc(A + XG_A_BYTES + kk * 32),
                                         (kt > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&empty_bar[st]);
            }
            mma_commit(&accf_bar[buf]);
        }
    } else if (warp >= 4) {
        // --------------------------------------------------------------- epilogue
        const int q = warp - 4;
        int j = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++j) {
            const int buf = j & 1;
            const int m0 = (t / tiles_n) * XG_BM, n0 = (t % tiles_n) * XG_UNITS;
            // a wait that ran out anywhere in the CTA (the producer's, the
            // MMA thread's or this one) turns this tile's outputs into NaN
            const bool ok = mbar_wait_bounded(&accf_bar[buf], (j >> 1) & 1, XT_WAIT_NS, &s_err) &&
                            *reinterpret_cast<volatile uint32_t *>(&s_err) == 0u;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int slot = m0 + 32 * q + lane;
            const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * XG_ACC_STRIDE;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t vz[32], vr[32], vc[32];
                tmem_ld_cols<32>(trow + 32 * half, vz);
                tmem_ld_cols<32>(trow + XG_UNITS + 32 * half, vr);
                tmem_ld_cols<32>(trow + 2 * XG_UNITS + 32 * half, vc);
                if (slot >= slots) continue;
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    const int u = n0 + 32 * half + 8 * g8;
                    if (u >= d_h) break;   // d_h is a multiple of 8
                    const int64_t i = static_cast<int64_t>(slot) * d_h + u;
                    float h[8];
                    if (h_in != nullptr) {
                        unpack16(*reinterpret_cast<const uint4 *>(h_in + i), h);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) h[e] = 0.f;
                    }
                    float prm[6][8];
#pragma unroll
                    for (int r = 0; r < 6; ++r) {
                        const float4 a = *reinterpret_cast<const float4 *>(params + r * d_h + u);
                        const float4 b = *reinterpret_cast<const float4 *>(params + r * d_h + u + 4);
                        prm[r][0] = a.x;
                        prm[r][1] = a.y;
                        prm[r][2] = a.z;
                        prm[r][3] = a.w;
                        prm[r][4] = b.x;
                        prm[r][5] = b.y;
                        prm[r][6] = b.z;
                        prm[r][7] = b.w;
                    }
                    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int c = 8 * g8 + e;
                        const float nan = __int_as_float(0x7fffffff);
                        const float pz = ok ? round_to<__nv_bfloat16>(__uint_as_float(vz[c])) : nan;
                        const float pr = ok ? round_to<__nv_bfloat16>(__uint_as_float(vr[c])) : nan;
                        const float pc = ok ? round_to<__nv_bfloat16>(__uint_as_float(vc[c])) : nan;
                        const UnitParams up{prm[0][e], prm[1][e], prm[2][e], prm[3][e], prm[4][e], prm[5][e]};
                        o[e] = from_f32<__nv_bfloat16>(cell_f_storage<__nv_bfloat16>(h[e], pz, pr, pc, up));
                    }
                    *reinterpret_cast<uint4 *>(h_out + i) = *reinterpret_cast<const uint4 *>(o);
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&acce_bar[buf]);
        }
    }
    __syncwarp();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 2) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(XG_TMEM_COLS)
                     : "memory");
    }
}

}  // namespace

int decode_xtc_units(int slots, int d_h) {
    // 32-unit tiles when they alone give about one CTA per SM, else 8-unit
    // tiles (four times the CTAs streaming W_x)
    const int64_t ctas32 = static_cast<int64_t>((d_h + 31) / 32) * ((slots + XT_SLOTS - 1) / XT_SLOTS);
    return ctas32 >= 128 ? 32 : 8;
}

template <int UNITS>
cudaError_t launch_xtc(const CUtensorMap &tmX, const CUtensorMap &tmW, const float *params,
                       const void *h_in, void *h_out, int slots, int d_in, int d_h,
                       cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    constexpr size_t smem = static_cast<size_t>(XT_STAGES) * XT_STAGE_BYTES + 1024;
    cudaError_t e = once_per_device(configured, [](int) {
        return cudaFuncSetAttribute(k_decode_step_xtc<UNITS>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    if (e != cudaSuccess) return e;
    const dim3 grid((d_h + UNITS - 1) / UNITS, (slots + XT_SLOTS - 1) / XT_SLOTS);
    k_decode_step_xtc<UNITS><<<grid, 128, smem, stream>>>(
        tmX, tmW, params, static_cast<const __nv_bfloat16 *>(h_in),
        static_cast<__nv_bfloat16 *>(h_out), slots, d_in, d_h);
    return cudaGetLastError();
}

// The split-K cluster form for one slot tile of 8-unit CTAs that leave most
// SMs idle and have at least SK_KS slices of d_in each.
bool decode_split_k(int slots, int d_in, int d_h) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    const int64_t ctas = (d_h + SK_UNITS - 1) / SK_UNITS;   // 4 fit an SM (shared memory)
    return slots <= XT_SLOTS && (d_in + XT_BK - 1) / XT_BK >= SK_KS &&
           ctas * SK_KS <= 4 * static_cast<int64_t>(sms) && decode_xtc_units(slots, d_h) == SK_UNITS;
}

cudaError_t launch_xtc_sk(const CUtensorMap &tmX, const CUtensorMap &tmW, const float *params,
                          const void *h_in, void *h_out, int slots, int d_in, int d_h,
                          cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    constexpr size_t smem = static_cast<size_t>(SK_STAGES) * XT_STAGE_BYTES + 1024;
    cudaError_t e = once_per_device(configured, [](int) {
        return cudaFuncSetAttribute(k_decode_step_xtc_sk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((d_h + SK_UNITS - 1) / SK_UNITS, 1, SK_KS);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = SK_KS;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_decode_step_xtc_sk, tmX, tmW, params,
                              static_cast<const __nv_bfloat16 *>(h_in),
                              static_cast<__nv_bfloat16 *>(h_out), slots, d_in, d_h);
}

cudaError_t launch_decode_step_xtc(const CUtensorMap &tmX, const CUtensorMap &tmW,
                                   const float *params, const void *h_in, void *h_out, int slots,
                                   int d_in, int d_h, cudaStream_t stream) {
    if (slots == 0) return cudaSuccess;
    if (decode_split_k(slots, d_in, d_h))
        return launch_xtc_sk(tmX, tmW, params, h_in, h_out, slots, d_in, d_h, stream);
    if (decode_xtc_units(slots, d_h) == 32)
        return launch_xtc<32>(tmX, tmW, params, h_in, h_out, slots, d_in, d_h, stream);
    return launch_xtc<8>(tmX, tmW, params, h_in, h_out, slots, d_in, d_h, stream);
}

cudaError_t launch_decode_step_xg(const CUtensorMap &tmX, const CUtensorMap &tmW,
                                  const float *params, const void *h_in, void *h_out, int slots,
                                  int d_in, int d_h, cudaStream_t stream) {
    if (slots == 0) return cudaSuccess;
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = once_per_device(configured, [](int) {
        return cudaFuncSetAttribute(k_decode_step_xg, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(XG_SMEM));
    });
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorUnknown;
    const int64_t tiles = static_cast<int64_t>((slots + XG_BM - 1) / XG_BM) * ((d_h + XG_UNITS - 1) / XG_UNITS);
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, sms));
    k_decode_step_xg<<<grid, 256, XG_SMEM, stream>>>(tmX, tmW, params,
                                                     static_cast<const __nv_bfloat16 *>(h_in),
                                                     static_cast<__nv_bfloat16 *>(h_out), slots,
                                                     d_in, d_h);
    return cudaGetLastError();
}

cudaError_t launch_decode_step(int dtype, const void *P, const float *params, const void *h_in,
                               void *h_out, int slots, int d_h, cudaStream_t stream) {
    const int64_t n = static_cast<int64_t>(slots) * d_h;
    if (n == 0) return cudaSuccess;
    const int vec = 4;
    const auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    if (d_h % vec == 0 && a16(P) && a16(params) && a16(h_out) && (h_in == nullptr || a16(h_in))) {
        // one resident wave of threads, each taking an equal number of two-slot passes
        static std::atomic<int> resident[2] = {0, 0};   // CTAs per SM, by dtype
        int dev = 0, sms = 0, per_sm = resident[dtype == 1].load();
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaErrorUnknown;
        if (per_sm == 0) {
            const cudaError_t oe =
                dtype == 1
                    ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_step_vec<__nv_bfloat16>, 256, 0)
                    : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_step_vec<float>, 256, 0);
            if (oe != cudaSuccess) return oe;
            resident[dtype == 1].store(per_sm);
        }
        const int64_t groups = d_h / vec;
        const int64_t target =
            std::max<int64_t>(1, static_cast<int64_t>(sms) * std::max(per_sm, 1) * 256 / groups);
        const int64_t passes = (slots + 2 * target - 1) / (2 * target);
        const int lanes = static_cast<int>((slots + 2 * passes - 1) / (2 * passes));
        const unsigned vblocks = static_cast<unsigned>((groups * lanes + 255) / 256);
        if (dtype == 1)
            k_decode_step_vec<__nv_bfloat16><<<vblocks, 256, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(P), params,
                static_cast<const __nv_bfloat16 *>(h_in), static_cast<__nv_bfloat16 *>(h_out),
                slots, d_h, lanes);
        else
            k_decode_step_vec<float><<<vblocks, 256, 0, stream>>>(
                static_cast<const float *>(P), params, static_cast<const float *>(h_in),
                static_cast<float *>(h_out), slots, d_h, lanes);
        return cudaGetLastError();
    }
    const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
    if (dtype == 1)
        k_decode_step<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(P), params, static_cast<const __nv_bfloat16 *>(h_in),
            static_cast<__nv_bfloat16 *>(h_out), slots, d_h);
    else
        k_decode_step<float><<<blocks, 256, 0, stream>>>(static_cast<const float *>(P), params,
                                                         static_cast<const float *>(h_in),
                                                         static_cast<float *>(h_out), slots, d_h);
    return cudaGetLastError();
}

cudaError_t launch_decode_step_x(int dtype, const void *x, const void *W, const float *params,
                                 const void *h_in, void *h_out, int slots, int d_in, int d_h,
                                 cudaStream_t stream) {
    if (slots == 0) return cudaSuccess;
    const dim3 grid((d_h + DX_UNITS - 1) / DX_UNITS, (slots + DX_SLOTS - 1) / DX_SLOTS);
    const size_t xbytes = static_cast<size_t>(DX_SLOTS) * d_in * (dtype == 1 ? 2 : 4);
    const int stage = xbytes <= DX_SMEM_MAX ? 1 : 0;
    const size_t smem = stage ? xbytes : 0;
    if (dtype == 1)
        k_decode_step_x<__nv_bfloat16><<<grid, DX_UNITS * 32, smem, stream>>>(
            static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(W), params,
            static_cast<const __nv_bfloat16 *>(h_in), static_cast<__nv_bfloat16 *>(h_out), slots,
            d_in, d_h, stage);
    else
        k_decode_step_x<float><<<grid, DX_UNITS * 32, smem, stream>>>(
            static_cast<const float *>(x), static_cast<const float *>(W), params,
            static_cast<const float *>(h_in), static_cast<float *>(h_out), slots, d_in, d_h, stage);
    return cudaGetLastError();
}

}  // namespace nrnn

// Input projection P = x W_x^T on the 5th-generation tensor cores.
//
// Persistent kernel, one CTA per SM, tiles of P taken round-robin (gate
// columns fastest, so CTAs working at the same time share the x rows in L2).
// Both operands are K-major (x is (rows, d_in), W_x is (3 d_h, d_in), both
// row-major); TMA stages K slices of 128-byte rows with the 128-byte swizzle
// into a ring of shared-memory stages that runs on across tiles.  Warp roles:
//   warp 0      TMA producer (one thread)
//   warp 1      MMA issuer (one thread): tcgen05.mma into one of two TMEM
//               accumulators, tcgen05.commit returns stages and hands a
//               finished accumulator to the epilogue
//   warp 2      owns the tensor-memory allocation
//   warps 4..7  epilogue: tcgen05.ld of their 32-lane quarter, 32 x 32
//               blocks staged in shared memory and sent out by TMA stores,
//               then release the accumulator; it overlaps the next K loop
//   warps 8..15 (fp32 only) split each staged x tile for split-TF32
// bf16: kind::f16, 128 x 256 tiles, 64-wide K slices, 4 stages, fp32
// accumulation rounded to bf16.  fp32: split-TF32 ("3xTF32") -- each fp32
// operand v is read by kind::tf32 as hi = v with its low 13 mantissa bits
// dropped (the tensor core ignores them, so a staged tile serves as hi
// unchanged), lo = v - hi is exact with |lo| < 2^-10 |v|, and
//   A B ~ A_hi B_hi + A_hi B_lo + A_lo B_hi
// (the dropped A_lo B_lo and the TF32 reading of lo are of order 2^-20
// relative).  The low part of the static operand W_x is computed once per
// call into global memory (k_split_low) and staged by TMA like its high part;
// the splitter warps write the low part of each staged x tile beside it with
// 16-byte accesses.  128 x 128 tiles in 3 stages, or 128 x 256 in 2, with
// 32-wide K slices.
// Out-of-range rows, columns and K are zero-filled by TMA loads and clipped
// by TMA stores.  Every wait is bounded; a wait that gives up sets
// g_projection_tc_error and the epilogue writes NaN, which the Newton residual
// gate downstream reports as divergence.
#include <type_traits>

#include "nrnn_device.cuh"
#include "nrnn_internal.h"
#include "tcgen05.cuh"

namespace nrnn {

namespace {

constexpr uint64_t TC_WAIT_NS = 2000000000ull;

__device__ uint32_t g_projection_tc_error;

// MODE 0: bf16; MODE 1: fp32 split-TF32, 128-column tiles; MODE 2: fp32
// split-TF32, 256-column tiles (half the A-operand traffic per product, two
// stages)
template <int MODE> struct ProjCfg;

template <> struct ProjCfg<0> {
    static constexpr bool F32 = false;
    static constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
    static constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int THREADS = 256;
    static constexpr int MMA_K = 16;   // elements per instruction (32 bytes)
    // D fp32, A and B bf16, both K-major, N = BN, M = BM
    static constexpr uint32_t IDESC = idesc_kmajor<false>(BM, BN);
};

template <int BN_, int STAGES_> struct ProjCfgTf32 {   // fp32 split-TF32
    static constexpr bool F32 = true;
    static constexpr int BM = 128, BN = BN_, BK = 32, STAGES = STAGES_;
    static constexpr int A_BYTES = BM * BK * 4, B_BYTES = BN * BK * 4;
    static constexpr int STAGE_BYTES = 2 * (A_BYTES + B_BYTES);   // A | B | lo A | lo B
    static constexpr int THREADS = 512;
    static constexpr int MMA_K = 8;    // elements per instruction (32 bytes)
    // D fp32, A and B TF32, both K-major, N = BN, M = BM
    static constexpr uint32_t IDESC = idesc_kmajor<true>(BM, BN);
};
template <> struct ProjCfg<1> : ProjCfgTf32<128, 3> {};
template <> struct ProjCfg<2> : ProjCfgTf32<256, 2> {};

constexpr int SPLIT_THREADS = 256;

// v - (v with its low 13 mantissa bits cleared): what kind::tf32 drops, exact
__device__ __forceinline__ float low_part(uint32_t bits) {
    return __uint_as_float(bits) - __uint_as_float(bits & 0xffffe000u);
}

__global__ void k_split_low(const uint32_t *__restrict__ w, float *__restrict__ lo, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n; i += stride)
        lo[i] = low_part(w[i]);
}
constexpr int EPI_THREADS = 128;

// The epilogue writes each 32 x 32 block of the accumulator, converted to the
// output type, into a shared-memory buffer in the layout of a TMA box with the
// 64-byte (bf16: 64-byte rows) or 128-byte (fp32: 128-byte rows) swizzle, and
// one TMA store sends it to P in whole lines: the row-per-thread layout of
// tcgen05.ld would otherwise store 16-byte pieces of 32 different rows.  The
// swizzle moves 16-byte piece q of row r to q ^ ((r >> 1) & 3) (64-byte) or
// q ^ (r & 7) (128-byte), so the 32 row-writes of a warp hit distinct banks.
constexpr int OUT_BOX = PROJ_OUT_BOX;   // rows and columns of one stored block

// this thread's row (32 accumulator columns) -> the staged block
__device__ __forceinline__ void stage_row(unsigned char *blk, int r, const uint32_t (&v)[32],
                                          bool ok, __nv_bfloat16 *) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 pk;
        uint32_t *w = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = ok ? __uint_as_float(v[q * 8 + 2 * e]) : __int_as_float(0x7fffffff);
            const float hi = ok ? __uint_as_float(v[q * 8 + 2 * e + 1]) : __int_as_float(0x7fffffff);
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
            w[e] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        *reinterpret_cast<uint4 *>(blk + r * 64 + 16 * (q ^ ((r >> 1) & 3))) = pk;
    }
}
__device__ __forceinline__ void stage_row(unsigned char *blk, int r, const uint32_t (&v)[32],
                                          bool ok, float *) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        uint4 o;
        o.x = ok ? v[4 * q + 0] : 0x7fffffffu;
        o.y = ok ? v[4 * q + 1] : 0x7fffffffu;
        o.z = ok ? v[4 * q + 2] : 0x7fffffffu;
        o.w = ok ? v[4 * q + 3] : 0x7fffffffu;
        *reinterpret_cast<uint4 *>(blk + r * 128 + 16 * (q ^ (r & 7))) = o;
    }
}

template <int MODE>
__global__ void __launch_bounds__(ProjCfg<MODE>::THREADS, 1)
    k_projection_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBlo, const __grid_constant__ CUtensorMap tmP,
                    int64_t rows, int K, int N) {
    using C = ProjCfg<MODE>;
    constexpr bool F32 = C::F32;
    using Out = typename std::conditional<F32, float, __nv_bfloat16>::type;
    constexpr uint32_t TMEM_COLS = 2 * C::BN;   // two accumulators
    uint32_t *error = &g_projection_tc_error;
    extern __shared__ unsigned char dsmem_raw[];
    // the 128-byte swizzle needs 1024-byte aligned tiles
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[C::STAGES], split_bar[C::STAGES],
        empty_bar[C::STAGES], accf_bar[2], acce_bar[2];
    __shared__ uint32_t s_tmem;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = (N + C::BN - 1) / C::BN;
    const int64_t tiles_m = (rows + C::BM - 1) / C::BM;
    const int kt_count = (K + C::BK - 1) / C::BK;
    // tiles in order, gate columns fastest, round-robin over the CTAs
    const int64_t n_tiles = tiles_m * tiles_n;
    const int64_t tile0 = blockIdx.x, tile_step = gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&split_bar[s], SPLIT_THREADS);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf_bar[b], 1);
            mbar_init(&acce_bar[b], EPI_THREADS);
        }
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (F32) prefetch_tensormap(&tmBlo);
        prefetch_tensormap(&tmP);
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(TMEM_COLS)
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
        for (int64_t u = tile0; u < n_tiles; u += tile_step) {
            const int64_t m0 = (u / tiles_n) * C::BM;
            const int n0 = static_cast<int>(u % tiles_n) * C::BN;
            for (int kt = 0; kt < kt_count; ++kt, ++it) {
                const int s = it % C::STAGES;
                if (it >= C::STAGES)
                    mbar_wait_bounded(&empty_bar[s], ((it / C::STAGES) - 1) & 1, TC_WAIT_NS, error);
                unsigned char *st = smem + s * C::STAGE_BYTES;
                // stage layout: A | B | lo A | lo B
                mbar_arrive_expect_tx(&full_bar[s], C::A_BYTES + (F32 ? 2 : 1) * C::B_BYTES);
                tma_load_2d(st, &tmA, &full_bar[s], kt * C::BK, static_cast<int>(m0));
                tma_load_2d(st + C::A_BYTES, &tmB, &full_bar[s], kt * C::BK, n0);
                if (F32)
                    tma_load_2d(st + 2 * C::A_BYTES + C::B_BYTES, &tmBlo, &full_bar[s], kt * C::BK, n0);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        int it = 0, j = 0;
        for (int64_t u = tile0; u < n_tiles; u += tile_step, ++j) {
            const int buf = j & 1;
            if (j >= 2) mbar_wait_bounded(&acce_bar[buf], ((j >> 1) - 1) & 1, TC_WAIT_NS, error);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t d = tmem + buf * C::BN;
            for (int kt = 0; kt < kt_count; ++kt, ++it) {
                const int s = it % C::STAGES;
                mbar_wait_bounded(F32 ? &split_bar[s] : &full_bar[s], (it / C::STAGES) & 1,
                                  TC_WAIT_NS, error);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a_hi = smem_u32(smem + s * C::STAGE_BYTES);
                const uint32_t b_hi = a_hi + C::A_BYTES;
#pragma unroll
                for (int kk = 0; kk < C::BK / C::MMA_K; ++kk) {   // 32 bytes of K per MMA
                    const uint32_t o = kk * 32;
                    const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
                    if (F32) {
                        const uint32_t a_lo = a_hi + C::A_BYTES + C::B_BYTES;
                        const uint32_t b_lo = a_lo + C::A_BYTES;
                        mma<F32, C::IDESC>(d, sw128_desc(a_lo + o), sw128_desc(b_hi + o), acc);
                        mma<F32, C::IDESC>(d, sw128_desc(a_hi + o), sw128_desc(b_lo + o), 1u);
                        mma<F32, C::IDESC>(d, sw128_desc(a_hi + o), sw128_desc(b_hi + o), 1u);
                    } else {
                        mma<F32, C::IDESC>(d, sw128_desc(a_hi + o), sw128_desc(b_hi + o), acc);
                    }
                }
                mma_commit(&empty_bar[s]);
            }
            mma_commit(&accf_bar[buf]);
        }
    } else if (F32 && warp >= 8) {
        // ------------------------------------------- split-TF32 operand splitter
        const int t = threadIdx.x - 8 * 32;
        int it = 0;
        for (int64_t u = tile0; u < n_tiles; u += tile_step) {
            for (int kt = 0; kt < kt_count; ++kt, ++it) {
                const int s = it % C::STAGES;
                mbar_wait_bounded(&full_bar[s], (it / C::STAGES) & 1, TC_WAIT_NS, error);
                const uint4 *raw = reinterpret_cast<const uint4 *>(smem + s * C::STAGE_BYTES);
                float4 *lo = reinterpret_cast<float4 *>(smem + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES);
#pragma unroll 4
                for (int e = t; e < C::A_BYTES / 16; e += SPLIT_THREADS) {
                    const uint4 v = raw[e];
                    lo[e] = make_float4(low_part(v.x), low_part(v.y), low_part(v.z), low_part(v.w));
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(&split_bar[s]);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // --------------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        constexpr int BLK_BYTES = OUT_BOX * OUT_BOX * static_cast<int>(sizeof(Out));
        // two staged blocks per warp: one is filled while the other is stored
        unsigned char *stage_out = smem + C::STAGES * C::STAGE_BYTES + quarter * 2 * BLK_BYTES;
        int nblk = 0;
        int j = 0;
        for (int64_t u = tile0; u < n_tiles; u += tile_step, ++j) {
            const int buf = j & 1;
            const int64_t m0 = (u / tiles_n) * C::BM;
            const int n0 = static_cast<int>(u % tiles_n) * C::BN;
            const bool ok = mbar_wait_bounded(&accf_bar[buf], (j >> 1) & 1, TC_WAIT_NS, error);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int64_t row0 = m0 + quarter * 32;
#pragma unroll 1
            for (int c = 0; c < C::BN; c += OUT_BOX) {
                uint32_t v[32];
                tmem_ld_cols<32>(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * C::BN + c, v);
                if (row0 >= rows || n0 + c >= N) continue;   // block wholly outside P
                unsigned char *blk = stage_out + (nblk & 1) * BLK_BYTES;
                if (lane == 0) bulk_wait_read<1>();   // this buffer's previous store has read it
                __syncwarp();
                stage_row(blk, lane, v, ok, static_cast<Out *>(nullptr));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmP, blk, n0 + c, static_cast<int>(row0));
                    bulk_commit();
                }
                ++nblk;
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&acce_bar[buf]);
        }
        if (lane == 0) bulk_wait_all();   // the stores are done before the CTA exits
    }
    __syncwarp();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 2) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

template <int MODE>
cudaError_t launch_tc(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmBlo,
                      const CUtensorMap &tmP, int64_t rows, int d_in, int n_out,
                      cudaStream_t stream) {
    using C = ProjCfg<MODE>;
    static std::atomic<unsigned long long> configured{0};
    static int sms_of[64];   // SMs per device: one persistent CTA each
    // operand ring + two staged output blocks per epilogue warp + alignment slack
    constexpr size_t smem = static_cast<size_t>(C::STAGES) * C::STAGE_BYTES +
                            (EPI_THREADS / 32) * 2 * OUT_BOX * OUT_BOX * (C::F32 ? 4 : 2) + 1024;
    cudaError_t e = once_per_device(configured, [](int dev) {
        cudaError_t r = cudaFuncSetAttribute(k_projection_tc<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        int n = 0;
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess && n <= 0) r = cudaErrorInvalidConfiguration;
        if (r == cudaSuccess && dev < 64) sms_of[dev] = n;
        return r;
    });
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    const int64_t n_tiles = ((rows + C::BM - 1) / C::BM) * ((n_out + C::BN - 1) / C::BN);
    const int64_t grid = n_tiles < sms_of[dev] ? n_tiles : sms_of[dev];
    k_projection_tc<MODE><<<static_cast<unsigned>(grid), C::THREADS, smem, stream>>>(
        tmA, tmB, tmBlo, tmP, rows, d_in, n_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_projection_tc(const CUtensorMap &tmA, const CUtensorMap &tmB,
                                 const CUtensorMap &tmP, int64_t rows, int d_in, int n_out,
                                 cudaStream_t stream) {
    return launch_tc<0>(tmA, tmB, tmB, tmP, rows, d_in, n_out, stream);
}

int projection_tf32x3_bn(int n_out) { return n_out >= 512 ? 256 : 128; }

cudaError_t launch_projection_tf32x3(const CUtensorMap &tmA, const CUtensorMap &tmB,
                                     const CUtensorMap &tmBlo, const CUtensorMap &tmP,
                                     int64_t rows, int d_in, int n_out, cudaStream_t stream) {
    if (projection_tf32x3_bn(n_out) == 256)
        return launch_tc<2>(tmA, tmB, tmBlo, tmP, rows, d_in, n_out, stream);
    return launch_tc<1>(tmA, tmB, tmBlo, tmP, rows, d_in, n_out, stream);
}

cudaError_t launch_split_low(const void *w, void *lo, int64_t n, cudaStream_t stream) {
    const int64_t blocks = (n + 255) / 256;
    k_split_low<<<static_cast<unsigned>(blocks < 1216 ? blocks : 1216), 256, 0, stream>>>(
        static_cast<const uint32_t *>(w), static_cast<float *>(lo), n);
    return cudaGetLastError();
}

}  // namespace nrnn

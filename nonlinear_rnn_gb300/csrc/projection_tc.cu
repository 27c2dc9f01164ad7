// Input projection P = x W_x^T on the 5th-generation tensor cores (bf16
// operands, fp32 accumulation in tensor memory, bf16 result).
//
// One CTA computes a 128 x 256 tile of P (rows x gate columns).  Both operands
// are K-major (x is (rows, d_in), W_x is (3 d_h, d_in), both row-major), so
// TMA stages 64-wide K slices of each with the 128-byte swizzle into a
// 4-deep shared-memory ring.  One thread issues the TMA copies, one thread
// issues tcgen05.mma (M = 128, N = 256, K = 16 per instruction) into a
// 128-lane x 256-column fp32 accumulator in TMEM and returns each stage to
// the producer with tcgen05.commit; after the last K slice the four warps
// read the accumulator back (tcgen05.ld, one 32-lane quarter per warp),
// round to bf16 and store their rows.  Out-of-range rows, columns and K are
// zero-filled by TMA and masked on store.  Every mbarrier wait is bounded;
// a wait that gives up sets g_projection_tc_error and the tile is written as
// NaN, which the Newton residual gate downstream reports as divergence.
#include "nrnn_device.cuh"
#include "nrnn_internal.h"

namespace nrnn {

namespace {

constexpr int TC_BM = 128;
constexpr int TC_BN = 256;
constexpr int TC_BK = 64;                     // 64 bf16 = 128 bytes: one swizzle row
constexpr int TC_STAGES = 4;
constexpr int TC_THREADS = 128;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;   // 16 KiB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;   // 32 KiB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;
constexpr int TC_TMEM_COLS = 256;
constexpr uint64_t TC_WAIT_NS = 2000000000ull;

__device__ uint32_t g_projection_tc_error;

// Shared-memory matrix descriptor of a K-major tile with the 128-byte swizzle:
// 8-row x 128-byte core blocks stacked along M/N every 1024 bytes (SBO), start
// address in 16-byte units, descriptor version 1, layout type 2 (SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3ffffu) >> 4);          // start address
    d |= static_cast<uint64_t>(16u >> 4) << 16;                        // LBO (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;                      // SBO
    d |= static_cast<uint64_t>(1u) << 46;                              // version
    d |= static_cast<uint64_t>(2u) << 61;                              // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N = TC_BN, M = TC_BM.
constexpr uint32_t TC_IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                              (static_cast<uint32_t>(TC_BN >> 3) << 17) |
                              (static_cast<uint32_t>(TC_BM >> 4) << 24);

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(TC_IDESC), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    k_projection_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    int64_t rows, int K, int N, __nv_bfloat16 *__restrict__ P) {
    uint32_t *error = &g_projection_tc_error;
    extern __shared__ unsigned char dsmem_raw[];
    // the 128-byte swizzle needs 1024-byte aligned tiles
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[TC_STAGES], empty_bar[TC_STAGES], acc_bar;
    __shared__ uint32_t s_tmem;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * TC_BN;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TC_BM;
    const int kt_count = (K + TC_BK - 1) / TC_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(&acc_bar, 1);
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 2) {   // one warp owns the tensor-memory allocation
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;

    if (warp == 0 && lane == 0) {
        // TMA producer
        for (int kt = 0; kt < kt_count; ++kt) {
            const int s = kt % TC_STAGES;
            if (kt >= TC_STAGES)
                mbar_wait_bounded(&empty_bar[s], ((kt / TC_STAGES) - 1) & 1, TC_WAIT_NS, error);
            unsigned char *sa = smem + s * TC_STAGE_BYTES;
            unsigned char *sb = sa + TC_A_BYTES;
            mbar_arrive_expect_tx(&full_bar[s], TC_STAGE_BYTES);
            tma_load_2d(sa, &tmA, &full_bar[s], kt * TC_BK, static_cast<int>(m0));
            tma_load_2d(sb, &tmB, &full_bar[s], kt * TC_BK, n0);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        for (int kt = 0; kt < kt_count; ++kt) {
            const int s = kt % TC_STAGES;
            mbar_wait_bounded(&full_bar[s], (kt / TC_STAGES) & 1, TC_WAIT_NS, error);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t sa = smem_u32(smem + s * TC_STAGE_BYTES);
            const uint32_t sb = sa + TC_A_BYTES;
#pragma unroll
            for (int kk = 0; kk < TC_BK / 16; ++kk)   // 16 bf16 = 32 bytes per MMA
                mma_bf16(tmem, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32),
                         (kt > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&empty_bar[s]);
        }
        mma_commit(&acc_bar);
    }
    __syncwarp();

    // epilogue: warp w reads accumulator lanes 32 w .. 32 w + 31 (tile rows)
    const bool acc_ok = mbar_wait_bounded(&acc_bar, 0, TC_WAIT_NS, error);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int64_t row = m0 + warp * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < TC_BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32cols(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 32, v);
        const int col0 = n0 + c * 32;
        if (row < rows) {
            __nv_bfloat16 *dst = P + row * N + col0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // 8 columns (16 bytes) per store
                if (col0 + q * 8 + 8 <= N) {
                    uint4 pk;
                    uint32_t *w = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = acc_ok ? __uint_as_float(v[q * 8 + 2 * e]) : __int_as_float(0x7fffffff);
                        const float hi = acc_ok ? __uint_as_float(v[q * 8 + 2 * e + 1]) : __int_as_float(0x7fffffff);
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
                        w[e] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                    *reinterpret_cast<uint4 *>(dst + q * 8) = pk;
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 2) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TC_TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// fp32 projection on the tensor cores with split-TF32 ("3xTF32"): each fp32
// operand x is split into hi = x rounded to the nearest TF32 value (low 13
// mantissa bits cleared after adding half of their range; exactly
// representable in TF32, so the tensor core reads it unchanged) and lo = x - hi
// (exact, |lo| <= 2^-11 |x|), and
//   A B ~ A_hi B_hi + A_hi B_lo + A_lo B_hi
// (the dropped A_lo B_lo term and the TF32 reading of lo are of order 2^-21
// relative), which keeps fp32-level accuracy where a single TF32 product would
// not.  128 x 128 tiles, 32-wide fp32 K slices (128-byte swizzle rows), three
// stages.  Warp 0 issues TMA, warp 1 issues tcgen05.mma kind::tf32 (M 128,
// N 128, K 8), warps 4..7 split each staged tile in place (hi into the TMA
// buffer, lo into a second buffer), fence the generic-to-async proxy and
// release the stage to the MMA thread.
constexpr int T3_BM = 128;
constexpr int T3_BN = 128;
constexpr int T3_BK = 32;                       // 32 fp32 = 128 bytes
constexpr int T3_STAGES = 3;
constexpr int T3_THREADS = 256;
constexpr int T3_TILE_BYTES = 128 * T3_BK * 4;  // 16 KiB (A or B, hi or lo)
constexpr int T3_STAGE_BYTES = 4 * T3_TILE_BYTES;   // A_hi, B_hi, A_lo, B_lo
constexpr int T3_TMEM_COLS = 128;
constexpr int T3_SPLIT_THREADS = 128;

constexpr uint32_t T3_IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                              (static_cast<uint32_t>(T3_BN >> 3) << 17) |
                              (static_cast<uint32_t>(T3_BM >> 4) << 24);

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(T3_IDESC), "r"(accumulate)
        : "memory");
}

__global__ void __launch_bounds__(T3_THREADS, 1)
    k_projection_tf32x3(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        int64_t rows, int K, int N, float *__restrict__ P) {
    uint32_t *error = &g_projection_tc_error;
    extern __shared__ unsigned char dsmem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full_bar[T3_STAGES], split_bar[T3_STAGES],
        empty_bar[T3_STAGES], acc_bar;
    __shared__ uint32_t s_tmem;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * T3_BN;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * T3_BM;
    const int kt_count = (K + T3_BK - 1) / T3_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < T3_STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&split_bar[s], T3_SPLIT_THREADS);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(&acc_bar, 1);
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(T3_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;

    if (warp == 0 && lane == 0) {
        for (int kt = 0; kt < kt_count; ++kt) {
            const int s = kt % T3_STAGES;
            if (kt >= T3_STAGES)
                mbar_wait_bounded(&empty_bar[s], ((kt / T3_STAGES) - 1) & 1, TC_WAIT_NS, error);
            unsigned char *st = smem + s * T3_STAGE_BYTES;
            mbar_arrive_expect_tx(&full_bar[s], 2 * T3_TILE_BYTES);
            tma_load_2d(st, &tmA, &full_bar[s], kt * T3_BK, static_cast<int>(m0));
            tma_load_2d(st + T3_TILE_BYTES, &tmB, &full_bar[s], kt * T3_BK, n0);
        }
    } else if (warp == 1 && lane == 0) {
        for (int kt = 0; kt < kt_count; ++kt) {
            const int s = kt % T3_STAGES;
            mbar_wait_bounded(&split_bar[s], (kt / T3_STAGES) & 1, TC_WAIT_NS, error);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t a_hi = smem_u32(smem + s * T3_STAGE_BYTES);
            const uint32_t b_hi = a_hi + T3_TILE_BYTES;
            const uint32_t a_lo = a_hi + 2 * T3_TILE_BYTES;
            const uint32_t b_lo = a_hi + 3 * T3_TILE_BYTES;
#pragma unroll
            for (int kk = 0; kk < T3_BK / 8; ++kk) {   // 8 fp32 = 32 bytes per MMA
                const uint32_t o = kk * 32;
                mma_tf32(tmem, sw128_desc(a_lo + o), sw128_desc(b_hi + o), (kt > 0 || kk > 0) ? 1u : 0u);
                mma_tf32(tmem, sw128_desc(a_hi + o), sw128_desc(b_lo + o), 1u);
                mma_tf32(tmem, sw128_desc(a_hi + o), sw128_desc(b_hi + o), 1u);
            }
            mma_commit(&empty_bar[s]);
        }
        mma_commit(&acc_bar);
    } else if (warp >= 4) {
        // split the staged fp32 tiles in place: hi (TF32-exact) stays, lo goes to the second half
        const int t = threadIdx.x - 4 * 32;
        for (int kt = 0; kt < kt_count; ++kt) {
            const int s = kt % T3_STAGES;
            mbar_wait_bounded(&full_bar[s], (kt / T3_STAGES) & 1, TC_WAIT_NS, error);
            uint32_t *hi = reinterpret_cast<uint32_t *>(smem + s * T3_STAGE_BYTES);
            float *lo = reinterpret_cast<float *>(smem + s * T3_STAGE_BYTES + 2 * T3_TILE_BYTES);
#pragma unroll 4
            for (int e = t; e < 2 * T3_TILE_BYTES / 4; e += T3_SPLIT_THREADS) {
                const uint32_t bits = hi[e];
                const uint32_t hb = (bits + 0x1000u) & 0xffffe000u;
                lo[e] = __uint_as_float(bits) - __uint_as_float(hb);
                hi[e] = hb;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&split_bar[s]);
        }
    }
    __syncwarp();

    const bool acc_ok = mbar_wait_bounded(&acc_bar, 0, TC_WAIT_NS, error);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int quarter = warp & 3, half = warp >> 2;
    const int64_t row = m0 + quarter * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
        const int colc = half * 64 + c * 32;
        uint32_t v[32];
        tmem_ld_32cols(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + colc, v);
        const int col0 = n0 + colc;
        if (row < rows) {
            float *dst = P + row * N + col0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {   // 4 columns (16 bytes) per store
                if (col0 + q * 4 + 4 <= N) {
                    float4 o;
                    o.x = acc_ok ? __uint_as_float(v[4 * q + 0]) : __int_as_float(0x7fffffff);
                    o.y = acc_ok ? __uint_as_float(v[4 * q + 1]) : __int_as_float(0x7fffffff);
                    o.z = acc_ok ? __uint_as_float(v[4 * q + 2]) : __int_as_float(0x7fffffff);
                    o.w = acc_ok ? __uint_as_float(v[4 * q + 3]) : __int_as_float(0x7fffffff);
                    *reinterpret_cast<float4 *>(dst + q * 4) = o;
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 2) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(T3_TMEM_COLS)
                     : "memory");
    }
}

}  // namespace

size_t projection_tc_smem_bytes() { return static_cast<size_t>(TC_STAGES) * TC_STAGE_BYTES + 1024; }

cudaError_t launch_projection_tc(const CUtensorMap &tmA, const CUtensorMap &tmB, int64_t rows,
                                 int d_in, int n_out, void *P, cudaStream_t stream) {
    static bool configured = false;
    const size_t smem = projection_tc_smem_bytes();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_projection_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const dim3 grid((n_out + TC_BN - 1) / TC_BN, static_cast<unsigned>((rows + TC_BM - 1) / TC_BM));
    k_projection_tc<<<grid, TC_THREADS, smem, stream>>>(tmA, tmB, rows, d_in, n_out,
                                                        static_cast<__nv_bfloat16 *>(P));
    return cudaGetLastError();
}

cudaError_t launch_projection_tf32x3(const CUtensorMap &tmA, const CUtensorMap &tmB, int64_t rows,
                                     int d_in, int n_out, float *P, cudaStream_t stream) {
    static bool configured = false;
    const size_t smem = static_cast<size_t>(T3_STAGES) * T3_STAGE_BYTES + 1024;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_projection_tf32x3,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const dim3 grid((n_out + T3_BN - 1) / T3_BN, static_cast<unsigned>((rows + T3_BM - 1) / T3_BM));
    k_projection_tf32x3<<<grid, T3_THREADS, smem, stream>>>(tmA, tmB, rows, d_in, n_out, P);
    return cudaGetLastError();
}

}  // namespace nrnn

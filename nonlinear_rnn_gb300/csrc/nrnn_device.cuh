// Device helpers for the diagonal-GRU Newton kernels (sm_103a).
//
// Cell of ParaGRU(mix='diag') (pararnn-torch; equations as stated for its
// diag-GRU benches): z = sig(P_z + a_z h + b_z), r = sig(P_r + a_r h + b_r),
// c = tanh(P_c + a_c (r h) + b_c), f = (1 - z) h + z c.  Its derivative with
// respect to h (chain rule) is
//   J = (1 - z) + z (1 - z) a_z (c - h) + z (1 - c^2) a_c (r + h r (1 - r) a_r).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nrnn {

constexpr unsigned FULL_MASK = 0xffffffffu;

// ---------------------------------------------------------------- storage types
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename TS> __device__ __forceinline__ TS from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
// value of v after a round trip through the storage type
template <typename TS> __device__ __forceinline__ float round_to(float v) {
    return to_f32(from_f32<TS>(v));
}
// both values of a pair rounded to the storage type and widened back (bf16:
// one packed conversion instead of two)
template <typename TS> __device__ __forceinline__ float2 round2_to(float2 v);
template <> __device__ __forceinline__ float2 round2_to<float>(float2 v) { return v; }
template <> __device__ __forceinline__ float2 round2_to<__nv_bfloat16>(float2 v) {
    return __bfloat1622float2(__floats2bfloat162_rn(v.x, v.y));
}

// ------------------------------------------------------------- PTX primitives
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// min that propagates NaN (a NaN input must reach the residual gate)
__device__ __forceinline__ float min_nan(float a, float b) {
    float y;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}
// max that propagates NaN (a NaN residual must reach the gate)
__device__ __forceinline__ float max_nan(float a, float b) {
    float y;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// mbarrier + TMA (cp.async.bulk.tensor) for one CTA
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// shared -> global tile store; elements outside the tensor are not written
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y,
                                             int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// commit this thread's bulk stores and wait until their shared-memory sources
// have been read (the CTA may then exit or reuse the buffer)
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Bounded wait on an mbarrier phase; sets *error bit 2 and returns false on timeout.
// try_wait that suspends the thread until the phase completes or about
// hint_ns nanoseconds pass (no issue slots spent spinning)
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns, uint32_t *error) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint32_t hint = static_cast<uint32_t>(limit_ns < 1000000u ? limit_ns : 1000000u);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_hint(bar, parity, hint)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(error, 2u);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ the cell
struct UnitParams {
    float a_z, a_r, a_c, b_z, b_r, b_c;
};

__device__ __forceinline__ UnitParams load_unit_params(const float *params, int d_h, int u,
                                                       bool valid) {
    UnitParams p{0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid) {
        p.a_z = __ldg(params + 0 * d_h + u);
        p.a_r = __ldg(params + 1 * d_h + u);
        p.a_c = __ldg(params + 2 * d_h + u);
        p.b_z = __ldg(params + 3 * d_h + u);
        p.b_r = __ldg(params + 4 * d_h + u);
        p.b_c = __ldg(params + 5 * d_h + u);
    }
    return p;
}

constexpr float LOG2E = 1.4426950408889634f;

// logistic sigmoid: 1 / (1 + 2^(-x log2 e)); saturates to exactly 0 / 1
__device__ __forceinline__ float sigmoid_f(float x) {
    return rcp_approx(1.0f + ex2_approx(-LOG2E * x));
}
// tanh(x) = 1 - 2 / (1 + e^(2x)); saturates to exactly -1 / +1
__device__ __forceinline__ float tanh_f(float x) {
    return fmaf(-2.0f, rcp_approx(1.0f + ex2_approx((2.0f * LOG2E) * x)), 1.0f);
}

// f(h, P) only
__device__ __forceinline__ float cell_f(float h, float pz, float pr, float pc,
                                        const UnitParams &p) {
    const float z = sigmoid_f(fmaf(p.a_z, h, pz + p.b_z));
    const float r = sigmoid_f(fmaf(p.a_r, h, pr + p.b_r));
    const float c = tanh_f(fmaf(p.a_c, r * h, pc + p.b_c));
    return fmaf(z, c - h, h);
}

// ---------------------------------------------- cell on pre-scaled arguments
// The gate arguments are carried in exponent-2 units:
//   sz = -log2(e) (P_z + b_z),  sr = -log2(e) (P_r + b_r),  sc = 2 log2(e) (P_c + b_c)
// so that z = 1 / (1 + 2^(sz - log2(e) a_z h)) and tanh(x) = 1 - 2 / (1 + 2^(2 log2(e) x))
// each start from one FFMA.  z and the tanh share one reciprocal:
// 1/(dz dc) times dc gives 1/dz and times dz gives 1/dc; the arguments are
// clamped at 63 so that dz dc stays finite (below 2^126); the clamp moves
// sigmoid by less than 1e-19 and leaves tanh at exactly 1 in fp32.
struct ScaledParams {
    float na_z, na_r, a_c2;   // -log2(e) a_z, -log2(e) a_r, 2 log2(e) a_c
    float a_z, a_r, a_c;      // for the Jacobian
    float nb_z, nb_r, b_c2;   // -log2(e) b_z, -log2(e) b_r, 2 log2(e) b_c
};

__device__ __forceinline__ ScaledParams scale_params(const UnitParams &p) {
    ScaledParams s;
    s.na_z = -LOG2E * p.a_z;
    s.na_r = -LOG2E * p.a_r;
    s.a_c2 = 2.0f * LOG2E * p.a_c;
    s.a_z = p.a_z;
    s.a_r = p.a_r;
    s.a_c = p.a_c;
    s.nb_z = -LOG2E * p.b_z;
    s.nb_r = -LOG2E * p.b_r;
    s.b_c2 = 2.0f * LOG2E * p.b_c;
    return s;
}

// pre-scaled arguments of one step from raw preactivations
__device__ __forceinline__ void scale_preact(float pz, float pr, float pc, const ScaledParams &p,
                                             float &sz, float &sr, float &sc) {
    sz = fmaf(pz, -LOG2E, p.nb_z);
    sr = fmaf(pr, -LOG2E, p.nb_r);
    sc = fmaf(pc, 2.0f * LOG2E, p.b_c2);
}

constexpr float EXP2_CLAMP = 63.0f;

// gates z, r, c at state h
__device__ __forceinline__ void gates_scaled(float h, float sz, float sr, float sc,
                                             const ScaledParams &p, float &z, float &r,
                                             float &c) {
    const float dz = 1.0f + ex2_approx(min_nan(fmaf(p.na_z, h, sz), EXP2_CLAMP));
    r = rcp_approx(1.0f + ex2_approx(fmaf(p.na_r, h, sr)));
    const float dc = 1.0f + ex2_approx(min_nan(fmaf(p.a_c2, r * h, sc), EXP2_CLAMP));
    const float inv = rcp_approx(dz * dc);
    z = dc * inv;
    c = fmaf(-2.0f, dz * inv, 1.0f);
}

// ------------------------------------------------ the cell on pairs of steps
// sm_100 and later execute fma / mul / add on a pair of fp32 values as one
// instruction (f32x2: two FMA lanes for one issue slot).  The Newton kernel
// evaluates two independent time steps per thread with them; ex2 / rcp and the
// clamps stay scalar.  Each lane of a pair computes exactly what the scalar
// formulas below compute, up to the order of a few roundings.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 ex2_2(float2 x) {
    return make_float2(ex2_approx(x.x), ex2_approx(x.y));
}
__device__ __forceinline__ float2 rcp_2(float2 x) {
    return make_float2(rcp_approx(x.x), rcp_approx(x.y));
}
__device__ __forceinline__ float2 clamp2(float2 x) {
    return make_float2(min_nan(x.x, EXP2_CLAMP), min_nan(x.y, EXP2_CLAMP));
}

struct ScaledParams2 {
    float2 na_z, na_r, a_c2;   // state coefficients of the exponent-2 gate arguments
    float2 a_z, ma_z, a_r, a_c4;   // Jacobian: a_z, -a_z, a_r, 4 a_c
    float2 nb_z, nb_r, b_c2;   // scaled biases (raw preactivations only)
};

__device__ __forceinline__ ScaledParams2 pair_params(const ScaledParams &p) {
    ScaledParams2 q;
    q.na_z = splat2(p.na_z);
    q.na_r = splat2(p.na_r);
    q.a_c2 = splat2(p.a_c2);
    q.a_z = splat2(p.a_z);
    q.ma_z = splat2(-p.a_z);
    q.a_r = splat2(p.a_r);
    q.a_c4 = splat2(4.0f * p.a_c);
    q.nb_z = splat2(p.nb_z);
    q.nb_r = splat2(p.nb_r);
    q.b_c2 = splat2(p.b_c2);
    return q;
}

// pre-scaled arguments of a pair of steps from raw preactivations
__device__ __forceinline__ void scale_preact2(float2 pz, float2 pr, float2 pc,
                                              const ScaledParams2 &p, float2 &sz, float2 &sr,
                                              float2 &sc) {
    sz = fma2(pz, splat2(-LOG2E), p.nb_z);
    sr = fma2(pr, splat2(-LOG2E), p.nb_r);
    sc = fma2(pc, splat2(2.0f * LOG2E), p.b_c2);
}

// gates at a pair of states (gates_scaled on each lane); q = 1 / (1 + 2^(arg_c)),
// so that c = 1 - 2 q and 1 - c^2 = 4 q (1 - q)
__device__ __forceinline__ void gates2(float2 h, float2 sz, float2 sr, float2 sc,
                                       const ScaledParams2 &p, float2 &z, float2 &r, float2 &c,
                                       float2 &q) {
    const float2 one = splat2(1.0f);
    const float2 dz = add2(ex2_2(clamp2(fma2(p.na_z, h, sz))), one);
    r = rcp_2(add2(ex2_2(fma2(p.na_r, h, sr)), one));
    const float2 dc = add2(ex2_2(clamp2(fma2(p.a_c2, mul2(r, h), sc))), one);
    const float2 inv = rcp_2(mul2(dz, dc));
    z = mul2(dc, inv);
    q = mul2(dz, inv);
    c = fma2(splat2(-2.0f), q, one);
}

// gates2 with two signs folded in, for the Jacobian below: z, mr = -r, c and
// mq = -q.  -(1 + 2^x) costs the same one fma as 1 + 2^x, and the negated
// values save the (1 - r), (1 - q) steps of the derivative (r (1 - r) =
// -(mr + mr^2), q (1 - q) = -(mq + mq^2)).  nh = -h.
__device__ __forceinline__ void gates2_neg(float2 h, float2 nh, float2 sz, float2 sr, float2 sc,
                                           const ScaledParams2 &p, float2 &z, float2 &mr,
                                           float2 &c, float2 &mq) {
    const float2 one = splat2(1.0f), mone = splat2(-1.0f);
    const float2 dz = add2(ex2_2(clamp2(fma2(p.na_z, h, sz))), one);
    mr = rcp_2(fma2(ex2_2(fma2(p.na_r, h, sr)), mone, mone));
    const float2 mdc = fma2(ex2_2(clamp2(fma2(p.a_c2, mul2(mr, nh), sc))), mone, mone);
    const float2 minv = rcp_2(mul2(dz, mdc));   // -1 / (dz dc)
    z = mul2(mdc, minv);
    mq = mul2(dz, minv);
    c = fma2(splat2(2.0f), mq, one);
}

// J = df/dh and the Newton pair's offset g = f(h) - J h for a pair of shifted
// states.  With inner = (1 - z) a_z (c - h) + (1 - c^2) a_c d(rh)/dh one has
// J = (1 - z) + z inner = 1 + z (inner - 1) and f - J h = z (c - h inner)
// = z ((c - h) - h (inner - 1)); the kernels use inner - 1 directly.  With
// D = -d(rh)/dh = mr + h a_r (mr + mr^2) and 1 - c^2 = 4 q (1 - q):
// (1 - c^2) a_c d(rh)/dh = 4 a_c (mq + mq^2) D.
__device__ __forceinline__ void cell_jg2(float2 h, float2 sz, float2 sr, float2 sc,
                                         const ScaledParams2 &p, float2 &J, float2 &g) {
    const float2 one = splat2(1.0f), mone = splat2(-1.0f);
    const float2 nh = mul2(h, mone);
    float2 z, mr, c, mq;
    gates2_neg(h, nh, sz, sr, sc, p, z, mr, c, mq);
    const float2 cmh = add2(c, nh);
    const float2 D = fma2(mul2(h, p.a_r), fma2(mr, mr, mr), mr);
    const float2 t3m1 = fma2(mul2(p.a_c4, fma2(mq, mq, mq)), D, mone);   // (1 - c^2) a_c dq - 1
    const float2 im1 = fma2(fma2(z, p.ma_z, p.a_z), cmh, t3m1);           // inner - 1
    J = fma2(z, im1, one);
    g = mul2(z, fma2(nh, im1, cmh));
}

// the same at the zero state: g = f(0) = z c, J = (1 - z) + z ((1 - z) a_z c + (1 - c^2) a_c r)
__device__ __forceinline__ void cell_jg2_at_zero(float2 sz, float2 sr, float2 sc,
                                                 const ScaledParams2 &p, float2 &J, float2 &g) {
    const float2 one = splat2(1.0f), mone = splat2(-1.0f);
    const float2 dz = add2(ex2_2(clamp2(sz)), one);
    const float2 mr = rcp_2(fma2(ex2_2(sr), mone, mone));
    const float2 mdc = fma2(ex2_2(clamp2(sc)), mone, mone);
    const float2 minv = rcp_2(mul2(dz, mdc));
    const float2 z = mul2(mdc, minv);
    const float2 mq = mul2(dz, minv);
    const float2 c = fma2(splat2(2.0f), mq, one);
    const float2 t3m1 = fma2(mul2(p.a_c4, fma2(mq, mq, mq)), mr, mone);   // (1 - c^2) a_c r - 1
    J = fma2(z, fma2(fma2(z, p.ma_z, p.a_z), c, t3m1), one);
    g = mul2(z, c);
}

// f(h) for a pair of states
__device__ __forceinline__ float2 cell_f2(float2 h, float2 sz, float2 sr, float2 sc,
                                          const ScaledParams2 &p) {
    float2 z, r, c, q;
    gates2(h, sz, sr, sc, p, z, r, c, q);
    return fma2(z, fma2(h, splat2(-1.0f), c), h);
}

// --------------------------------------------- cell formulations per storage
// ExpCell (fp32 storage): the exponent-2 form above, ex2.approx and
// rcp.approx, a few ulp.  TanhCell (bf16 storage): sig(x) = (1 + tanh(x/2))/2
// and tanh on tanh.approx.f32 (max relative error about 2^-11, four times
// below the bf16 storage step), three MUFU operations per evaluation and no
// clamps (tanh saturates).  Both present the same interface to the kernels:
// pre-scaled gate arguments, (J, g) of a pair of steps, f of a pair.
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float2 tanh_2(float2 x) {
    return make_float2(tanh_approx(x.x), tanh_approx(x.y));
}

struct ExpCell {
    using Params = ScaledParams2;
    __device__ static Params make(const UnitParams &p) { return pair_params(scale_params(p)); }
    // pre-scaled argument of gate g from a raw preactivation: p * mul + add
    __device__ static void gate_affine(int g, const UnitParams &p, float &mul, float &add) {
        mul = g == 2 ? 2.0f * LOG2E : -LOG2E;
        add = g == 0 ? -LOG2E * p.b_z : (g == 1 ? -LOG2E * p.b_r : 2.0f * LOG2E * p.b_c);
    }
    __device__ static void scale(float2 pz, float2 pr, float2 pc, const Params &q, float2 &sz,
                                 float2 &sr, float2 &sc) {
        scale_preact2(pz, pr, pc, q, sz, sr, sc);
    }
    __device__ static void jg(float2 h, float2 sz, float2 sr, float2 sc, const Params &q, float2 &J,
                              float2 &g) {
        cell_jg2(h, sz, sr, sc, q, J, g);
    }
    __device__ static void jg_zero(float2 sz, float2 sr, float2 sc, const Params &q, float2 &J,
                                   float2 &g) {
        cell_jg2_at_zero(sz, sr, sc, q, J, g);
    }
    __device__ static float2 f(float2 h, float2 sz, float2 sr, float2 sc, const Params &q) {
        return cell_f2(h, sz, sr, sc, q);
    }
};

struct TanhCell {
    struct Params {
        float2 hz, hr;           // a_z / 2, a_r / 2: state terms of the halved z, r arguments
        float2 a_c, na_c;        // a_c, -a_c
        float2 a_z, a_r;         // Jacobian
        float2 bz, br, bc;       // b_z / 2, b_r / 2, b_c
    };
    __device__ static Params make(const UnitParams &p) {
        Params q;
        q.hz = splat2(0.5f * p.a_z);
        q.hr = splat2(0.5f * p.a_r);
        q.a_c = splat2(p.a_c);
        q.na_c = splat2(-p.a_c);
        q.a_z = splat2(p.a_z);
        q.a_r = splat2(p.a_r);
        q.bz = splat2(0.5f * p.b_z);
        q.br = splat2(0.5f * p.b_r);
        q.bc = splat2(p.b_c);
        return q;
    }
    __device__ static void gate_affine(int g, const UnitParams &p, float &mul, float &add) {
        mul = g == 2 ? 1.0f : 0.5f;
        add = g == 0 ? 0.5f * p.b_z : (g == 1 ? 0.5f * p.b_r : p.b_c);
    }
    __device__ static void scale(float2 pz, float2 pr, float2 pc, const Params &q, float2 &sz,
                                 float2 &sr, float2 &sc) {
        sz = fma2(pz, splat2(0.5f), q.bz);
        sr = fma2(pr, splat2(0.5f), q.br);
        sc = add2(pc, q.bc);
    }
    // tz = tanh(arg_z / 2 ...): z = (1 + tz) / 2, 1 - z = (1 - tz) / 2; likewise r
    __device__ static void gates(float2 h, float2 sz, float2 sr, float2 sc, const Params &q,
                                 float2 &tz, float2 &tr, float2 &r, float2 &c) {
        tz = tanh_2(fma2(q.hz, h, sz));
        tr = tanh_2(fma2(q.hr, h, sr));
        r = fma2(splat2(0.5f), tr, splat2(0.5f));
        c = tanh_2(fma2(q.a_c, mul2(r, h), sc));
    }
    __device__ static void jg(float2 h, float2 sz, float2 sr, float2 sc, const Params &q, float2 &J,
                              float2 &g) {
        float2 tz, tr, r, c;
        gates(h, sz, sr, sc, q, tz, tr, r, c);
        const float2 half = splat2(0.5f), mhalf = splat2(-0.5f), mone = splat2(-1.0f);
        const float2 z = fma2(half, tz, half), omz = fma2(mhalf, tz, half);
        const float2 omr = fma2(mhalf, tr, half);
        const float2 nh = mul2(h, mone);
        const float2 cmh = add2(c, nh);
        const float2 dq = fma2(mul2(mul2(h, q.a_r), omr), r, r);      // d(r h)/dh
        const float2 t2 = fma2(mul2(c, q.na_c), c, q.a_c);            // a_c (1 - c^2)
        const float2 inner = fma2(mul2(omz, q.a_z), cmh, mul2(t2, dq));
        J = fma2(z, inner, omz);
        g = mul2(z, fma2(nh, inner, c));
    }
    __device__ static void jg_zero(float2 sz, float2 sr, float2 sc, const Params &q, float2 &J,
                                   float2 &g) {
        const float2 half = splat2(0.5f), mhalf = splat2(-0.5f);
        const float2 tz = tanh_2(sz), tr = tanh_2(sr), c = tanh_2(sc);
        const float2 z = fma2(half, tz, half), omz = fma2(mhalf, tz, half);
        const float2 r = fma2(half, tr, half);
        const float2 t2 = fma2(mul2(c, q.na_c), c, q.a_c);
        J = fma2(z, fma2(mul2(omz, q.a_z), c, mul2(t2, r)), omz);
        g = mul2(z, c);
    }
    __device__ static float2 f(float2 h, float2 sz, float2 sr, float2 sc, const Params &q) {
        float2 tz, tr, r, c;
        gates(h, sz, sr, sc, q, tz, tr, r, c);
        const float2 z = fma2(splat2(0.5f), tz, splat2(0.5f));
        return fma2(z, fma2(h, splat2(-1.0f), c), h);
    }
};

template <typename TS> struct CellOf { using type = ExpCell; };
template <> struct CellOf<__nv_bfloat16> { using type = TanhCell; };

// f(h, P) from raw preactivations in the storage type's formulation: the
// ex2/rcp form for fp32, tanh.approx for bf16 (sig(x) = (1 + tanh(x/2))/2)
template <typename TS>
__device__ __forceinline__ float cell_f_storage(float h, float pz, float pr, float pc,
                                                const UnitParams &p) {
    if constexpr (sizeof(TS) == 2) {
        const float z = fmaf(0.5f, tanh_approx(0.5f * fmaf(p.a_z, h, pz + p.b_z)), 0.5f);
        const float r = fmaf(0.5f, tanh_approx(0.5f * fmaf(p.a_r, h, pr + p.b_r)), 0.5f);
        const float c = tanh_approx(fmaf(p.a_c, r * h, pc + p.b_c));
        return fmaf(z, c - h, h);
    } else {
        return cell_f(h, pz, pr, pc, p);
    }
}

// |F| for the residual gate; NaN counts as +inf
__device__ __forceinline__ float abs_residual(float F) {
    const float a = fabsf(F);
    return (a <= 3.402823466e38f) ? a : __int_as_float(0x7f800000);
}

// ----------------------------------------------------------- segment heads
// Sets bit (t - t0) of bits[] for every head t in [t0, t0 + len): t = 0, or
// t = cu[i] with cu[i] < cu[i + 1] (shapes_layout page: segment heads of a
// cu_seqlens pack use J = 0).  bits[] must be zeroed by the caller.  Stays
// inside cu[0 .. S] and inside bits[] for any contents of cu.
__device__ __forceinline__ void mark_heads(const int32_t *cu, int S, int64_t t0, int len,
                                           uint32_t *bits) {
    if (t0 == 0 && len > 0) bits[0] |= 1u;
    if (cu == nullptr || S <= 0) return;
    int lo = 0, hi = S + 1;  // first i in [0, S] with cu[i] >= t0
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(__ldg(cu + mid)) < t0) lo = mid + 1;
        else hi = mid;
    }
    for (int i = lo; i < S; ++i) {
        const int64_t s = __ldg(cu + i);
        if (s >= t0 + len) break;
        if (s >= t0 && s < static_cast<int64_t>(__ldg(cu + i + 1))) {
            const int o = static_cast<int>(s - t0);
            bits[o >> 5] |= 1u << (o & 31);
        }
    }
}

__device__ __forceinline__ bool head_bit(const uint32_t *bits, int r) {
    return (bits[r >> 5] >> (r & 31)) & 1u;
}

// pack / unpack an affine pair (A, b) into one 64-bit word (single-copy atomic)
__device__ __forceinline__ unsigned long long pack_pair(float A, float b) {
    return (static_cast<unsigned long long>(__float_as_uint(b)) << 32) | __float_as_uint(A);
}
__device__ __forceinline__ float pair_A(unsigned long long v) {
    return __uint_as_float(static_cast<uint32_t>(v));
}
__device__ __forceinline__ float pair_b(unsigned long long v) {
    return __uint_as_float(static_cast<uint32_t>(v >> 32));
}

// ------------------------------------------------- decoupled look-back slots
// One 64-bit word per (chunk, unit) holds the chunk's affine pair (A, b) and is
// its own ready flag: SLOT_EMPTY (all zero bits, from the per-call clear that
// also zeroes the counters) means not yet published.  Published pairs
// never take that value: publish() writes the pair (+0, +0) as (+0, -0),
// which composes identically.  Because a 64-bit aligned access is single-copy
// atomic, a reader sees either SLOT_EMPTY, the chunk aggregate, or the
// inclusive prefix (A = 0), and the latter two both compose correctly: no
// fence is needed on either side.
constexpr unsigned long long SLOT_EMPTY = 0ull;

__device__ __forceinline__ void publish(unsigned long long *slot, float A, float b) {
    unsigned long long v = pack_pair(A, b);
    if (v == SLOT_EMPTY) v = pack_pair(0.f, -0.f);
    st_relaxed_u64(slot, v);
}

// Decoupled look-back for one unit (one lane) of chunk c: composes the pairs
// of chunks c + dir, c + 2 dir, ... (dir = -1: earlier chunks, forward scan;
// dir = +1: later chunks, reverse scan) until a closed prefix (A = 0) or the
// end of the sequence, and returns the carry into chunk c.  `slot` is this
// lane's slot of chunk c; chunk c + dir d has slot + dir d 32.  Up to WIN
// neighbours are read per round with independent loads; while nothing is
// ready only the nearest is polled.  pre1, pre2: the slots of chunks c + dir
// and c + 2 dir as the caller read them earlier (SLOT_EMPTY if it did not,
// or if they were not published then): what they hold is folded first, so a
// caller that issues those loads before waiting for other work hides their
// latency.  Bounded: gives up after wait_ns without progress, sets bit 0 of
// *error and returns the partial prefix.
template <int WIN>
__device__ __forceinline__ float lookback_lane(const unsigned long long *slot, int c, int dir,
                                               int n_chunks, uint64_t wait_ns, uint32_t *error,
                                               unsigned long long pre1 = SLOT_EMPTY,
                                               unsigned long long pre2 = SLOT_EMPTY) {
    float cA = 1.f, cB = 0.f;
    int d = 1;   // distance of the next neighbour to fold
    if (pre1 != SLOT_EMPTY) {
        cB = pair_b(pre1);
        cA = pair_A(pre1);
        d = 2;
        if (cA == 0.f) return cB;
        if (pre2 != SLOT_EMPTY) {
            cB = fmaf(cA, pair_b(pre2), cB);
            cA *= pair_A(pre2);
            d = 3;
            if (cA == 0.f) return cB;
        }
    }
    for (;;) {
        const int q = c + dir * d;
        if (q < 0 || q >= n_chunks) break;
        unsigned long long v[WIN];
#pragma unroll
        for (int i = 0; i < WIN; ++i) {
            const int qi = c + dir * (d + i);
            v[i] = (qi >= 0 && qi < n_chunks)
                       ? ld_relaxed_u64(slot + static_cast<ptrdiff_t>(dir) * (d + i) * 32)
                       : pack_pair(0.f, -0.f);   // before the first chunk: closed, zero
        }
        int folded = 0;
#pragma unroll
        for (int i = 0; i < WIN; ++i) {
            if (folded < i || v[i] == SLOT_EMPTY) break;
            cB = fmaf(cA, pair_b(v[i]), cB);
            cA *= pair_A(v[i]);
            ++folded;
        }
        if (cA == 0.f) break;          // closed prefix (an inclusive or a head)
        d += folded;
        if (folded == 0) {
            const unsigned long long *nq = slot + static_cast<ptrdiff_t>(dir) * d * 32;
            const uint64_t t_wait = globaltimer_ns();
            while (ld_relaxed_u64(nq) == SLOT_EMPTY) {
                __nanosleep(64);
                if (globaltimer_ns() - t_wait > wait_ns) {
                    atomicOr(error, 1u);
                    return cB;
                }
            }
        }
    }
    return cB;
}

}  // namespace nrnn

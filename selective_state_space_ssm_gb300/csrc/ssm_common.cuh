// ssm_common.cuh -- device helpers shared by the sm_103a kernels of libssm_gb300.
//
//  * activation storage types (fp32 / bf16) and conversions
//  * the scalar functions of src/training/cpu_ops.ts (softplus, sigmoid, silu,
//    siluGrad), evaluated in fp32 with the hardware ex2 / rcp units
//  * TMA (cp.async.bulk.tensor) and mbarrier wrappers in inline PTX; every
//    mbarrier wait is bounded and reports a timeout through g_ssm_fault
//    instead of spinning forever.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through cudart)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

// ---------------------------------------------------------------- constants

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kALogLo = -10.0f;   // mamba1_cpu.ts A_LOG_CLAMP_LO
constexpr float kALogHi = 5.0f;     // mamba1_cpu.ts A_LOG_CLAMP_HI

// Fault codes written to g_ssm_fault (bitwise OR) by a bounded wait that ran out.
constexpr unsigned kFaultFwdWait = 1u;
constexpr unsigned kFaultBwdWait = 2u;
constexpr unsigned kFaultDrain = 4u;
constexpr unsigned kFaultSelftest = 16u;   // the bounded-wait self-test (probe.cu)

// mbarrier polls before a wait gives up (each try_wait may itself suspend for
// a hardware-chosen time slice, so this is far beyond any legitimate wait).
constexpr uint32_t kWaitLimit = 1u << 24;

}  // namespace ssm

// Fault word of the kernels in one translation unit (each .cu file that waits
// on an mbarrier has its own copy; the C ABI reads and clears them).
static __device__ unsigned int g_ssm_fault;

namespace ssm {

// ---------------------------------------------------------------- storage types

template <typename T> struct Act;
template <> struct Act<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Act<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) {
        return __float2bfloat16_rn(v);
    }
};

// ---------------------------------------------------------------- scalar math

// 2^x on the MUFU unit (flushes results below 2^-126 to 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log1p(e) for 0 <= e <= 1 from the identity log1p(e) = 2 atanh(s), s = e/(2+e)
// in [0, 1/3], and the Taylor series atanh(s) = sum_k s^(2k+1)/(2k+1) cut after
// k = 7 (next term below 3e-9 relative).  `inv2pe` is 1/(2+e).
__device__ __forceinline__ float log1p_unit(float e, float inv2pe) {
    const float s = e * inv2pe;
    const float s2 = s * s;
    float p = 1.0f / 15.0f;
    p = fmaf(p, s2, 1.0f / 13.0f);
    p = fmaf(p, s2, 1.0f / 11.0f);
    p = fmaf(p, s2, 1.0f / 9.0f);
    p = fmaf(p, s2, 1.0f / 7.0f);
    p = fmaf(p, s2, 1.0f / 5.0f);
    p = fmaf(p, s2, 1.0f / 3.0f);
    p = fmaf(p, s2, 1.0f);
    return 2.0f * s * p;
}

// softplus(x) = max(x, 0) + log1p(exp(-|x|))  (cpu_ops.ts softplus, no threshold
// branch).  Also returns e = exp(-|x|), from which sigmoid(x) follows.
__device__ __forceinline__ float softplus_e(float x, float& e) {
    e = ex2(-fabsf(x) * kLog2e);
    return fmaxf(x, 0.0f) + log1p_unit(e, rcp(2.0f + e));
}
// sigmoid(x) from e = exp(-|x|):  x >= 0 -> 1/(1+e),  x < 0 -> e/(1+e).
__device__ __forceinline__ float sigmoid_from_e(float x, float e) {
    float r = rcp(1.0f + e);
    return x >= 0.0f ? r : e * r;
}
__device__ __forceinline__ float sigmoidf_(float x) {
    float e = ex2(-fabsf(x) * kLog2e);
    return sigmoid_from_e(x, e);
}

// softplus(x) and sigmoid(z) with one reciprocal between them:
// r = 1/((2+e)(1+ez)) gives 1/(2+e) = r(1+ez) and 1/(1+ez) = r(2+e).  ez is
// capped at 2^100 (z > -69.3); below that sigmoid(z) < 1e-30 and the capped
// value stays below 1e-30 as well.
__device__ __forceinline__ void softplus_sigmoid(float x, float z, float& sp, float& sig_z) {
    const float e = ex2(-fabsf(x) * kLog2e);
    const float ez = ex2(fminf(-z * kLog2e, 100.0f));
    const float a = 2.0f + e, b = 1.0f + ez;
    const float r = rcp(a * b);
    sp = fmaxf(x, 0.0f) + log1p_unit(e, r * b);
    sig_z = r * a;
}

// softplus(x) together with sigmoid(x) and sigmoid(z), from e = exp(-|x|),
// ez = exp(-z) and one reciprocal r = 1/((2+e)(1+ez)(1+e)): 1/(2+e) =
// r(1+ez)(1+e), sigmoid(z) = 1/(1+ez) = r(2+e)(1+e), 1/(1+e) = r(2+e)(1+ez).
// ez is capped at 2^100 as in softplus_sigmoid; the product stays below 2^103.
__device__ __forceinline__ void softplus_sig_xz(float x, float z, float& sp, float& sig_x,
                                                float& sig_z) {
    const float e = ex2(-fabsf(x) * kLog2e);
    const float ez = ex2(fminf(-z * kLog2e, 100.0f));
    const float a = 2.0f + e, b = 1.0f + ez, c = 1.0f + e;
    const float ab = a * b;
    const float r = rcp(ab * c);
    const float inv_c = r * ab;
    sig_z = r * (a * c);
    sp = fmaxf(x, 0.0f) + log1p_unit(e, r * (b * c));
    sig_x = x >= 0.0f ? inv_c : e * inv_c;
}
// The same without a gate: r = 1/((2+e)(1+e)).
__device__ __forceinline__ void softplus_sig_x(float x, float& sp, float& sig_x) {
    const float e = ex2(-fabsf(x) * kLog2e);
    const float a = 2.0f + e, c = 1.0f + e;
    const float r = rcp(a * c);
    const float inv_c = r * a;
    sp = fmaxf(x, 0.0f) + log1p_unit(e, r * c);
    sig_x = x >= 0.0f ? inv_c : e * inv_c;
}

// A = -exp(clamp(A_log, -10, 5)), returned pre-scaled by log2(e) so that
// exp(delta * A) = ex2(delta * A2).
__device__ __forceinline__ float a2_from_alog(float a_log) {
    float c = fminf(fmaxf(a_log, kALogLo), kALogHi);
    return -expf(c) * kLog2e;
}
__device__ __forceinline__ float a_from_alog(float a_log) {
    float c = fminf(fmaxf(a_log, kALogLo), kALogHi);
    return -expf(c);
}

// phi1(x) = expm1(x)/x and phi2(x) = (x e^x - e^x + 1)/x^2 for |x| < 1/2, by
// their Taylor series sum x^k/(k+1)! and sum (k+1) x^k/(k+2)! (truncation
// below 1e-9 relative there).  Used by the ZOH discretisation, where
// beta/B = delta*phi1(delta A) and d(beta/B)/dA = delta^2 * phi2(delta A).
__device__ __forceinline__ float phi1_series(float x) {
    float p = 1.0f / 40320.0f;                 // 1/8!
    p = fmaf(p, x, 1.0f / 5040.0f);
    p = fmaf(p, x, 1.0f / 720.0f);
    p = fmaf(p, x, 1.0f / 120.0f);
    p = fmaf(p, x, 1.0f / 24.0f);
    p = fmaf(p, x, 1.0f / 6.0f);
    p = fmaf(p, x, 0.5f);
    return fmaf(p, x, 1.0f);
}
__device__ __forceinline__ float phi2_series(float x) {
    float p = 9.0f / 3628800.0f;               // (k+1)/(k+2)! at k = 8
    p = fmaf(p, x, 8.0f / 362880.0f);
    p = fmaf(p, x, 7.0f / 40320.0f);
    p = fmaf(p, x, 6.0f / 5040.0f);
    p = fmaf(p, x, 5.0f / 720.0f);
    p = fmaf(p, x, 4.0f / 120.0f);
    p = fmaf(p, x, 3.0f / 24.0f);
    p = fmaf(p, x, 2.0f / 6.0f);
    return fmaf(p, x, 0.5f);
}

// ---------------------------------------------------------------- packed fp32

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// softplus_sig_xz / softplus_sig_x / softplus_sigmoid / softplus for two
// elements at once: the same
// formulas, the fp32 arithmetic on f32x2 pairs and the ex2 / rcp per element.
__device__ __forceinline__ float2 log1p_unit2(float2 e, float2 inv2pe) {
    const float2 s = mul2(e, inv2pe);
    const float2 s2 = mul2(s, s);
    float2 p = f2(1.0f / 15.0f);
    p = fma2(p, s2, f2(1.0f / 13.0f));
    p = fma2(p, s2, f2(1.0f / 11.0f));
    p = fma2(p, s2, f2(1.0f / 9.0f));
    p = fma2(p, s2, f2(1.0f / 7.0f));
    p = fma2(p, s2, f2(1.0f / 5.0f));
    p = fma2(p, s2, f2(1.0f / 3.0f));
    p = fma2(p, s2, f2(1.0f));
    return mul2(mul2(f2(2.0f), s), p);
}
__device__ __forceinline__ void softplus_sig_xz2(float2 x, float2 z, float2& sp, float2& sig_x,
                                                 float2& sig_z) {
    const float2 ax = mul2(make_float2(fabsf(x.x), fabsf(x.y)), f2(-kLog2e));
    const float2 e = make_float2(ex2(ax.x), ex2(ax.y));
    const float2 zz = mul2(z, f2(-kLog2e));
    const float2 ez = make_float2(ex2(fminf(zz.x, 100.0f)), ex2(fminf(zz.y, 100.0f)));
    const float2 a = add2(f2(2.0f), e), b = add2(f2(1.0f), ez), c = add2(f2(1.0f), e);
    const float2 ab = mul2(a, b);
    const float2 abc = mul2(ab, c);
    const float2 r = make_float2(rcp(abc.x), rcp(abc.y));
    const float2 inv_c = mul2(r, ab);
    sig_z = mul2(r, mul2(a, c));
    sp = add2(make_float2(fmaxf(x.x, 0.0f), fmaxf(x.y, 0.0f)), log1p_unit2(e, mul2(r, mul2(b, c))));
    const float2 ei = mul2(e, inv_c);
    sig_x = make_float2(x.x >= 0.0f ? inv_c.x : ei.x, x.y >= 0.0f ? inv_c.y : ei.y);
}
__device__ __forceinline__ void softplus_sigmoid2(float2 x, float2 z, float2& sp, float2& sig_z) {
    const float2 ax = mul2(make_float2(fabsf(x.x), fabsf(x.y)), f2(-kLog2e));
    const float2 e = make_float2(ex2(ax.x), ex2(ax.y));
    const float2 zz = mul2(z, f2(-kLog2e));
    const float2 ez = make_float2(ex2(fminf(zz.x, 100.0f)), ex2(fminf(zz.y, 100.0f)));
    const float2 a = add2(f2(2.0f), e), b = add2(f2(1.0f), ez);
    const float2 ab = mul2(a, b);
    const float2 r = make_float2(rcp(ab.x), rcp(ab.y));
    sp = add2(make_float2(fmaxf(x.x, 0.0f), fmaxf(x.y, 0.0f)), log1p_unit2(e, mul2(r, b)));
    sig_z = mul2(r, a);
}
__device__ __forceinline__ float2 softplus2(float2 x) {
    const float2 ax = mul2(make_float2(fabsf(x.x), fabsf(x.y)), f2(-kLog2e));
    const float2 e = make_float2(ex2(ax.x), ex2(ax.y));
    const float2 a = add2(f2(2.0f), e);
    return add2(make_float2(fmaxf(x.x, 0.0f), fmaxf(x.y, 0.0f)),
                log1p_unit2(e, make_float2(rcp(a.x), rcp(a.y))));
}
__device__ __forceinline__ void softplus_sig_x2(float2 x, float2& sp, float2& sig_x) {
    const float2 ax = mul2(make_float2(fabsf(x.x), fabsf(x.y)), f2(-kLog2e));
    const float2 e = make_float2(ex2(ax.x), ex2(ax.y));
    const float2 a = add2(f2(2.0f), e), c = add2(f2(1.0f), e);
    const float2 ac = mul2(a, c);
    const float2 r = make_float2(rcp(ac.x), rcp(ac.y));
    const float2 inv_c = mul2(r, a);
    sp = add2(make_float2(fmaxf(x.x, 0.0f), fmaxf(x.y, 0.0f)), log1p_unit2(e, mul2(r, c)));
    const float2 ei = mul2(e, inv_c);
    sig_x = make_float2(x.x >= 0.0f ? inv_c.x : ei.x, x.y >= 0.0f ? inv_c.y : ei.y);
}

// ---------------------------------------------------------------- mbarrier / TMA

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// Bounded wait for the phase with the given parity to complete.  Returns false
// (and records `fault`) if it did not complete within `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned fault,
                                          uint32_t limit = kWaitLimit) {
    const uint32_t a = smem_u32(bar);
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    atomicOr(&g_ssm_fault, fault);
    return false;
}
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 3-D tiled TMA load global -> shared, completion counted on `bar`.
// Coordinates are in elements (x innermost).  x * elemsize must be a multiple
// of 16 bytes (callers only pass tile starts that are multiples of 32 elements).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// Tile stores shared -> global (bulk-group completion).  Elements of the box
// outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(smem_u32(src))
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most one committed store group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Wait until every committed store group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace ssm

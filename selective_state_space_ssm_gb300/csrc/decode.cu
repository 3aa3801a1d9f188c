// decode.cu -- single-token decode kernels for sm_103a: one step of the
// selective scan with the state carried between calls, and one step of the
// causal conv1d + SiLU with the previous inputs kept in a ring.
//
// The recurrence is that of mamba1_cpu.ts mamba1CpuForward steps 8-9 (page
// "@seanhogg/builderforce-memory-engine 2026.7.12 -> 2026.9.27") taken at one
// position:
//   delta = softplus(delta_raw);  A = -exp(clamp(A_log, -10, 5))
//   h[n] <- exp(delta A_n) h[n] + beta_n u;  y = sum_n C_n h[n] + D u;
//   out = y * silu(z)
// and the conv that of steps 4-5 at one position (tap 0 = current input).
//
// Design (GB300): a decode step touches every state once, so it is bound by
// HBM: 2 * dstate * 4 bytes of state per (batch row, channel) against a few
// bytes of activations.  The state is laid out [batch][dstate][dinner] so that
// a thread owning 2 adjacent channels reads and writes one 8-byte vector per
// state (256 contiguous bytes per warp instruction); all dstate loads of a
// thread are issued before any arithmetic, which keeps 128 bytes per thread in
// flight at about 80 registers (7 CTAs of 128 threads per SM).
#include "decode_args.cuh"
#include "ssm_common.cuh"

namespace ssm {

namespace {

constexpr int kStepThreads = 128;

__device__ __forceinline__ float4 ld4f(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4f(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// 2 adjacent activations (8-byte aligned for fp32, 4-byte for bf16).
__device__ __forceinline__ void load2(const float* p, float (&v)[2]) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
}
__device__ __forceinline__ void load2(const __nv_bfloat16* p, float (&v)[2]) {
    const uint32_t t = *reinterpret_cast<const uint32_t*>(p);
    v[0] = __uint_as_float(t << 16);
    v[1] = __uint_as_float(t & 0xffff0000u);
}
__device__ __forceinline__ void store2(float* p, const float (&v)[2]) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}
__device__ __forceinline__ void store2(__nv_bfloat16* p, const float (&v)[2]) {
    __nv_bfloat162 t = __floats2bfloat162_rn(v[0], v[1]);
    *reinterpret_cast<__nv_bfloat162*>(p) = t;
}

__device__ __forceinline__ float silu_f(float x) { return x * rcp(1.0f + ex2(-x * kLog2e)); }

}  // namespace

// One thread = 2 adjacent channels of one batch row (blockIdx.y), all dstate
// states of them.
template <typename T, int NT, int DISC, bool GATE>
__global__ void __launch_bounds__(kStepThreads, 7)
scan_step_kernel(const ScanStepArgs a) {
    const int b = blockIdx.y;
    const int d0 = 2 * (blockIdx.x * kStepThreads + threadIdx.x);
    if (d0 >= a.dinner) return;
    const int N = a.dstate, Dn = a.dinner;
    float* hrow = a.h + static_cast<size_t>(b) * N * Dn + d0;

    // loads first: the states, the row's B and C, the channels' inputs
    float h[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float2 v = n < N ? *reinterpret_cast<const float2*>(hrow + static_cast<size_t>(n) * Dn)
                               : make_float2(0.f, 0.f);
        h[n][0] = v.x; h[n][1] = v.y;
    }
    // B and C of the row: the same addresses for every thread (cache hits),
    // read where they are used
    const T* Bp = static_cast<const T*>(a.B) + b * a.ld_B;
    const T* Cp = static_cast<const T*>(a.C) + b * a.ld_C;
    float uv[2], xr[2], zv[2] = {0.f, 0.f};
    load2(static_cast<const T*>(a.u) + b * a.ld_u + d0, uv);
    load2(static_cast<const T*>(a.dr) + b * a.ld_dr + d0, xr);
    if (GATE) load2(static_cast<const T*>(a.z) + b * a.ld_z + d0, zv);

    float y[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int d = d0 + c;
        float dt, gz = 1.0f;
        if (GATE) {
            float sz;
            softplus_sigmoid(xr[c], zv[c], dt, sz);
            gz = zv[c] * sz;                                   // silu(z)
        } else {
            float e;
            dt = softplus_e(xr[c], e);
        }
        const float bs = DISC == 0 ? dt * uv[c] : uv[c];       // Euler: delta*u; ZOH: u
        float acc = 0.0f;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            if (n >= N) break;
            const float A = a_from_alog(a.A_log[static_cast<size_t>(d) * N + n]);
            const float av = ex2(dt * A * kLog2e);
            float bu;
            if (DISC == 0) {
                bu = bs * Act<T>::load(Bp + n);
            } else {
                // beta/B = expm1(delta A)/A, without cancellation for small delta A
                const float xn = dt * A;
                const float cf = fabsf(xn) < 0.5f ? dt * phi1_series(xn) : (av - 1.0f) / A;
                bu = cf * bs * Act<T>::load(Bp + n);
            }
            h[n][c] = fmaf(av, h[n][c], bu);
            acc = fmaf(Act<T>::load(Cp + n), h[n][c], acc);
        }
        const float yv = (a.D ? fmaf(a.D[d], uv[c], acc) : acc);
        y[c] = GATE ? yv * gz : yv;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
        if (n < N) *reinterpret_cast<float2*>(hrow + static_cast<size_t>(n) * Dn) = make_float2(h[n][0], h[n][1]);
    store2(static_cast<T*>(a.out) + b * a.ld_out + d0, y);
}

// One thread = 4 adjacent channels of one batch row.
__global__ void __launch_bounds__(kStepThreads)
conv_step_kernel(const ConvStepArgs a) {
    const int nq = a.dinner / 4;
    const long long gid = static_cast<long long>(blockIdx.x) * kStepThreads + threadIdx.x;
    if (gid >= static_cast<long long>(nq) * a.batch) return;
    const int b = static_cast<int>(gid / nq);
    const int d0 = 4 * static_cast<int>(gid % nq);
    const int K = a.kconv, R = K - 1;
    const float4 x = ld4f(a.x + b * a.ld_x + d0);
    float4 acc = a.bias ? ld4f(a.bias + d0) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float* w = a.w + static_cast<size_t>(d0) * K;
    acc.x = fmaf(w[0], x.x, acc.x);
    acc.y = fmaf(w[K], x.y, acc.y);
    acc.z = fmaf(w[2 * K], x.z, acc.z);
    acc.w = fmaf(w[3 * K], x.w, acc.w);
    float* ring = a.ring + static_cast<size_t>(b) * R * a.dinner + d0;
    for (int k = 1; k < K; ++k) {
        const long long p = a.pos - k;
        if (p < 0) break;                                      // before the sequence: nothing
        const float4 v = ld4f(ring + static_cast<size_t>(p % R) * a.dinner);
        acc.x = fmaf(w[k], v.x, acc.x);
        acc.y = fmaf(w[K + k], v.y, acc.y);
        acc.z = fmaf(w[2 * K + k], v.z, acc.z);
        acc.w = fmaf(w[3 * K + k], v.w, acc.w);
    }
    st4f(a.out + b * a.ld_out + d0, make_float4(silu_f(acc.x), silu_f(acc.y), silu_f(acc.z), silu_f(acc.w)));
    // the slot of position pos held position pos-R, read above by this thread
    if (R > 0) st4f(ring + static_cast<size_t>(a.pos % R) * a.dinner, x);
}

// One thread = 4 adjacent channels of one (batch row, prompt position) among
// the last kconv-1 positions.
__global__ void __launch_bounds__(kStepThreads)
ring_fill_kernel(const RingFillArgs a) {
    const int R = a.kconv - 1;
    const int nq = a.dinner / 4;
    const long long gid = static_cast<long long>(blockIdx.x) * kStepThreads + threadIdx.x;
    if (gid >= static_cast<long long>(nq) * R * a.batch) return;
    const int q = static_cast<int>(gid % nq);
    const int i = static_cast<int>((gid / nq) % R);
    const int b = static_cast<int>(gid / (static_cast<long long>(nq) * R));
    const long long p = static_cast<long long>(a.seqlen) - R + i;   // prompt position
    if (p < 0) return;
    const float4 v = ld4f(a.x + (static_cast<size_t>(b) * a.seqlen + p) * a.ld_x + 4 * q);
    st4f(a.ring + (static_cast<size_t>(b) * R + static_cast<size_t>(p % R)) * a.dinner + 4 * q, v);
}

template <typename T, int NT>
static cudaError_t launch_step_nt(int disc, bool gate, const ScanStepArgs& a, cudaStream_t st) {
    const dim3 grid((a.dinner / 2 + kStepThreads - 1) / kStepThreads, a.batch);
    if (disc == 0) {
        if (gate) scan_step_kernel<T, NT, 0, true><<<grid, kStepThreads, 0, st>>>(a);
        else scan_step_kernel<T, NT, 0, false><<<grid, kStepThreads, 0, st>>>(a);
    } else {
        if (gate) scan_step_kernel<T, NT, 1, true><<<grid, kStepThreads, 0, st>>>(a);
        else scan_step_kernel<T, NT, 1, false><<<grid, kStepThreads, 0, st>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_scan_step(int dtype, int nt, int disc, bool gate, const ScanStepArgs& a,
                             cudaStream_t st) {
    if (a.batch == 0 || a.dinner == 0) return cudaSuccess;
    if (dtype == 0)
        return nt == 8 ? launch_step_nt<float, 8>(disc, gate, a, st)
                       : launch_step_nt<float, 16>(disc, gate, a, st);
    return nt == 8 ? launch_step_nt<__nv_bfloat16, 8>(disc, gate, a, st)
                   : launch_step_nt<__nv_bfloat16, 16>(disc, gate, a, st);
}

cudaError_t launch_conv_step(const ConvStepArgs& a, cudaStream_t st) {
    const long long total = static_cast<long long>(a.dinner / 4) * a.batch;
    if (total == 0) return cudaSuccess;
    conv_step_kernel<<<static_cast<unsigned>((total + kStepThreads - 1) / kStepThreads), kStepThreads, 0,
                       st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_ring_fill(const RingFillArgs& a, cudaStream_t st) {
    const long long total = static_cast<long long>(a.dinner / 4) * (a.kconv - 1) * a.batch;
    if (total == 0) return cudaSuccess;
    ring_fill_kernel<<<static_cast<unsigned>((total + kStepThreads - 1) / kStepThreads), kStepThreads, 0,
                       st>>>(a);
    return cudaGetLastError();
}

}  // namespace ssm

// decode.cu -- single-token decode kernels for sm_103a: one step of the
// selective scan with the state carried between calls, and one step of the
// causal conv1d + SiLU with the previous inputs kept in a shift register.
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
constexpr int kStepRows = 2;     // batch rows per decode-step CTA
constexpr int kConvRows = 4;     // batch rows per conv-step thread

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

// One thread = 2 adjacent channels, all dstate states of them, for the
// kStepRows batch rows of its CTA.  A log2(e) of its channels is computed once
// (vector loads of their A_log rows) and kept in shared memory for the rows;
// the states of the next row are loaded while the current one is computed and
// stored, so reads and writes of the state overlap within a CTA.  FULL:
// dstate == NT, so the per-state guards and strides are compile-time.
template <typename T, int NT, int DISC, bool GATE, bool FULL>
__global__ void __launch_bounds__(kStepThreads, 4)
scan_step_kernel(const ScanStepArgs a) {
    constexpr int CH = 2 * kStepThreads;          // channels per CTA
    constexpr int AS = CH + 2;                    // padded row
    constexpr int RB = kStepRows;
    __shared__ __align__(16) float As[NT * AS];   // A log2(e), [n][local channel]
    __shared__ float Bs[RB][NT], Cs[RB][NT];
    const int b0 = blockIdx.y * RB;
    const int nrow = min(RB, a.batch - b0);
    const int cbase = blockIdx.x * CH;
    const int N = FULL ? NT : a.dstate, Dn = a.dinner;
    const int d0 = cbase + 2 * threadIdx.x;
    const bool active = d0 < Dn;

    // one row's inputs: the states and the channels' u, delta_raw, z
    struct Row {
        float2 h[NT];                              // (channel d0, channel d0+1) per state
        float u[2], xr[2], z[2];
    };
    auto load_row = [&](Row& w, int b) {
        const float* hp = a.h + static_cast<size_t>(b) * N * Dn + d0;
#pragma unroll
        for (int n = 0; n < NT; ++n)
            w.h[n] = n < N ? *reinterpret_cast<const float2*>(hp + static_cast<size_t>(n) * Dn)
                           : make_float2(0.f, 0.f);
        load2(static_cast<const T*>(a.u) + b * a.ld_u + d0, w.u);
        load2(static_cast<const T*>(a.dr) + b * a.ld_dr + d0, w.xr);
        if (GATE) load2(static_cast<const T*>(a.z) + b * a.ld_z + d0, w.z);
    };
    // the longest loads first
    Row cur, nxt;
    if (active) load_row(cur, b0);

    for (int i = threadIdx.x; i < nrow * N; i += kStepThreads) {
        const int r = i / N, n = i - r * N;
        Bs[r][n] = Act<T>::load(static_cast<const T*>(a.B) + (b0 + r) * a.ld_B + n);
        Cs[r][n] = Act<T>::load(static_cast<const T*>(a.C) + (b0 + r) * a.ld_C + n);
    }
    // A log2(e) = -2^(clamp(A_log) log2(e)) log2(e) of this thread's two channels
    // (the 2N contiguous floats of their A_log rows), kept in shared memory
    // [n][channel] for the rows; only this thread reads its entries back
    if (active) {
        const float* al = a.A_log + static_cast<size_t>(d0) * N;
        auto a2 = [](float v) { return -ex2(fminf(fmaxf(v, kALogLo), kALogHi) * kLog2e) * kLog2e; };
        if (NT == 16 && N == 16 && (reinterpret_cast<uintptr_t>(al) & 15u) == 0) {   // 8 x 16-byte loads
            float4 q[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) q[k] = reinterpret_cast<const float4*>(al)[k];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 c0 = q[k], c1 = q[4 + k];         // states 4k..4k+3 of each channel
                *reinterpret_cast<float2*>(&As[(4 * k + 0) * AS + 2 * threadIdx.x]) = make_float2(a2(c0.x), a2(c1.x));
                *reinterpret_cast<float2*>(&As[(4 * k + 1) * AS + 2 * threadIdx.x]) = make_float2(a2(c0.y), a2(c1.y));
                *reinterpret_cast<float2*>(&As[(4 * k + 2) * AS + 2 * threadIdx.x]) = make_float2(a2(c0.z), a2(c1.z));
                *reinterpret_cast<float2*>(&As[(4 * k + 3) * AS + 2 * threadIdx.x]) = make_float2(a2(c0.w), a2(c1.w));
            }
        } else {
#pragma unroll
            for (int n = 0; n < NT; ++n)
                if (n < N)
                    *reinterpret_cast<float2*>(&As[n * AS + 2 * threadIdx.x]) = make_float2(a2(al[n]), a2(al[N + n]));
        }
    }
    __syncthreads();
    if (!active) return;
    const float Dv[2] = {a.D ? a.D[d0] : 0.0f, a.D ? a.D[d0 + 1] : 0.0f};

#pragma unroll
    for (int r = 0; r < RB; ++r) {
        if (r >= nrow) break;
        const int b = b0 + r;
        if (r + 1 < nrow) load_row(nxt, b + 1);   // next row in flight during this one

        float dt[2], bs[2], gz[2] = {1.0f, 1.0f};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            if (GATE) {
                float sz;
                softplus_sigmoid(cur.xr[c], cur.z[c], dt[c], sz);
                gz[c] = cur.z[c] * sz;                         // silu(z)
            } else {
                float e;
                dt[c] = softplus_e(cur.xr[c], e);
            }
            bs[c] = DISC == 0 ? dt[c] * cur.u[c] : cur.u[c];   // Euler: delta*u; ZOH: u
        }
        // both channels at once: packed f32x2 multiplies and FMAs
        const float2 dt2 = make_float2(dt[0], dt[1]), bs2 = make_float2(bs[0], bs[1]);
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            if (n >= N) break;
            const float2 A2 = *reinterpret_cast<const float2*>(&As[n * AS + 2 * threadIdx.x]);  // A log2(e)
            const float Bn = Bs[r][n], Cn = Cs[r][n];
            const float2 x = mul2(dt2, A2);
            const float2 av = make_float2(ex2(x.x), ex2(x.y));
            float2 bu;
            if (DISC == 0) {
                bu = mul2(bs2, f2(Bn));
            } else {
                // beta/B = expm1(delta A)/A, without cancellation for small delta A
                float cf[2];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float Ac = (c ? A2.y : A2.x) * kLn2;
                    const float xn = dt[c] * Ac;
                    const float ae = c ? av.y : av.x;
                    cf[c] = fabsf(xn) < 0.5f ? dt[c] * phi1_series(xn) : (ae - 1.0f) / Ac;
                }
                bu = mul2(mul2(make_float2(cf[0], cf[1]), bs2), f2(Bn));
            }
            cur.h[n] = fma2(av, cur.h[n], bu);
            acc = fma2(f2(Cn), cur.h[n], acc);
        }
        float y[2];
        const float accv[2] = {acc.x, acc.y};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const float yv = fmaf(Dv[c], cur.u[c], accv[c]);
            y[c] = GATE ? yv * gz[c] : yv;
        }
        float* hp = a.h + static_cast<size_t>(b) * N * Dn + d0;
#pragma unroll
        for (int n = 0; n < NT; ++n)
            if (n < N) *reinterpret_cast<float2*>(hp + static_cast<size_t>(n) * Dn) = cur.h[n];
        store2(static_cast<T*>(a.out) + b * a.ld_out + d0, y);
        if (r + 1 < nrow) cur = nxt;
    }
}

// One thread = 4 adjacent channels of kConvRows batch rows (the taps and bias
// loaded once for them); K taps unrolled so that every state load is in
// flight at once.
template <int K>
__global__ void __launch_bounds__(kStepThreads)
conv_step_kernel(const ConvStepArgs a) {
    constexpr int R = K - 1;
    constexpr int RB = kConvRows;
    const int nq = a.dinner / 4;
    const long long gid = static_cast<long long>(blockIdx.x) * kStepThreads + threadIdx.x;
    const int ngroups = (a.batch + RB - 1) / RB;
    if (gid >= static_cast<long long>(nq) * ngroups) return;
    const int b0 = static_cast<int>(gid / nq) * RB;
    const int d0 = 4 * static_cast<int>(gid % nq);
    const int nrow = min(RB, a.batch - b0);
    float4 x[RB], v[RB][K > 1 ? K - 1 : 1];                   // v[r][j]: input R-j steps back
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        if (r >= nrow) break;
        x[r] = ld4f(a.x + (b0 + r) * a.ld_x + d0);
        const float* st = a.state + static_cast<size_t>(b0 + r) * R * a.dinner + d0;
#pragma unroll
        for (int j = 0; j < R; ++j) v[r][j] = ld4f(st + static_cast<size_t>(j) * a.dinner);
    }
    const float4 bias = a.bias ? ld4f(a.bias + d0) : make_float4(0.f, 0.f, 0.f, 0.f);
    float wt[4][K];
    const float* w = a.w + static_cast<size_t>(d0) * K;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int k = 0; k < K; ++k) wt[c][k] = w[c * K + k];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        if (r >= nrow) break;
        float4 acc = bias;
        acc.x = fmaf(wt[0][0], x[r].x, acc.x);
        acc.y = fmaf(wt[1][0], x[r].y, acc.y);
        acc.z = fmaf(wt[2][0], x[r].z, acc.z);
        acc.w = fmaf(wt[3][0], x[r].w, acc.w);
#pragma unroll
        for (int k = 1; k < K; ++k) {
            const float4 s = v[r][R - k];
            acc.x = fmaf(wt[0][k], s.x, acc.x);
            acc.y = fmaf(wt[1][k], s.y, acc.y);
            acc.z = fmaf(wt[2][k], s.z, acc.z);
            acc.w = fmaf(wt[3][k], s.w, acc.w);
        }
        st4f(a.out + (b0 + r) * a.ld_out + d0,
             make_float4(silu_f(acc.x), silu_f(acc.y), silu_f(acc.z), silu_f(acc.w)));
        // shift: every slot one step older, the current input last
        float* st = a.state + static_cast<size_t>(b0 + r) * R * a.dinner + d0;
#pragma unroll
        for (int j = 0; j + 1 < R; ++j) st4f(st + static_cast<size_t>(j) * a.dinner, v[r][j + 1]);
        if (R > 0) st4f(st + static_cast<size_t>(R - 1) * a.dinner, x[r]);
    }
}

// One thread = 4 adjacent channels of one (batch row, state slot).
__global__ void __launch_bounds__(kStepThreads)
conv_state_fill_kernel(const ConvStateFillArgs a) {
    const int R = a.kconv - 1;
    const int nq = a.dinner / 4;
    const long long gid = static_cast<long long>(blockIdx.x) * kStepThreads + threadIdx.x;
    if (gid >= static_cast<long long>(nq) * R * a.batch) return;
    const int q = static_cast<int>(gid % nq);
    const int j = static_cast<int>((gid / nq) % R);
    const int b = static_cast<int>(gid / (static_cast<long long>(nq) * R));
    const long long p = static_cast<long long>(a.seqlen) - R + j;   // prompt position of slot j
    const float4 v = p >= 0 ? ld4f(a.x + (static_cast<size_t>(b) * a.seqlen + p) * a.ld_x + 4 * q)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    st4f(a.state + (static_cast<size_t>(b) * R + j) * a.dinner + 4 * q, v);
}

template <typename T, int NT>
static cudaError_t launch_step_nt(int disc, bool gate, const ScanStepArgs& a, cudaStream_t st) {
    const dim3 grid((a.dinner / 2 + kStepThreads - 1) / kStepThreads, (a.batch + kStepRows - 1) / kStepRows);
    // compile-time dstate for Euler B when the states fill NT (the ZOH path
    // would spill with it)
    const bool full = a.dstate == NT;
    if (disc == 0) {
        if (gate) {
            if (full) scan_step_kernel<T, NT, 0, true, true><<<grid, kStepThreads, 0, st>>>(a);
            else scan_step_kernel<T, NT, 0, true, false><<<grid, kStepThreads, 0, st>>>(a);
        } else {
            if (full) scan_step_kernel<T, NT, 0, false, true><<<grid, kStepThreads, 0, st>>>(a);
            else scan_step_kernel<T, NT, 0, false, false><<<grid, kStepThreads, 0, st>>>(a);
        }
    } else {
        if (gate) scan_step_kernel<T, NT, 1, true, false><<<grid, kStepThreads, 0, st>>>(a);
        else scan_step_kernel<T, NT, 1, false, false><<<grid, kStepThreads, 0, st>>>(a);
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
    const long long total = static_cast<long long>(a.dinner / 4) * ((a.batch + kConvRows - 1) / kConvRows);
    if (total == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((total + kStepThreads - 1) / kStepThreads);
    switch (a.kconv) {
        case 1: conv_step_kernel<1><<<grid, kStepThreads, 0, st>>>(a); break;
        case 2: conv_step_kernel<2><<<grid, kStepThreads, 0, st>>>(a); break;
        case 3: conv_step_kernel<3><<<grid, kStepThreads, 0, st>>>(a); break;
        case 4: conv_step_kernel<4><<<grid, kStepThreads, 0, st>>>(a); break;
        case 5: conv_step_kernel<5><<<grid, kStepThreads, 0, st>>>(a); break;
        case 6: conv_step_kernel<6><<<grid, kStepThreads, 0, st>>>(a); break;
        case 7: conv_step_kernel<7><<<grid, kStepThreads, 0, st>>>(a); break;
        default: conv_step_kernel<8><<<grid, kStepThreads, 0, st>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_conv_state_fill(const ConvStateFillArgs& a, cudaStream_t st) {
    const long long total = static_cast<long long>(a.dinner / 4) * (a.kconv - 1) * a.batch;
    if (total == 0) return cudaSuccess;
    conv_state_fill_kernel<<<static_cast<unsigned>((total + kStepThreads - 1) / kStepThreads), kStepThreads,
                             0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ssm

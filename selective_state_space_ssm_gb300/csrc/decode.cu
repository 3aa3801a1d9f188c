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
// the lanes of a warp (consecutive channels) read and write 128 contiguous
// bytes per state; every state load of a row is issued before its arithmetic
// and the next row's loads overlap the current row's work.
#include "decode_args.cuh"
#include "ssm_common.cuh"

namespace ssm {

namespace {

constexpr int kStepThreads = 128;
constexpr int kStepRows = 2;     // batch rows per decode-step CTA
constexpr int kConvRows = 2;     // batch rows per conv-step thread

__device__ __forceinline__ float4 ld4f(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4f(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

__device__ __forceinline__ float silu_f(float x) { return x * rcp(1.0f + ex2(-x * kLog2e)); }

}  // namespace

// One thread = one channel, all dstate states of it (in packed pairs), for the
// kStepRows batch rows of its CTA (a 64 x 4096 batch: 1024 CTAs of 128
// threads, 7 per SM by the 72-register budget).  A log2(e) of the channel is computed once
// into shared memory; the first two rows' states are both loaded before that
// set-up (more bytes in flight from the start), and each later row while the
// one before it is computed and stored.  FULL: dstate == NT.
template <typename T, int NT, int DISC, bool GATE, bool FULL>
__global__ void __launch_bounds__(kStepThreads, 7)
scan_step_kernel(const ScanStepArgs a) {
    constexpr int NP = NT / 2;                    // state pairs
    constexpr int RB = kStepRows;
    __shared__ float2 As[NP * kStepThreads];      // A log2(e), [pair][local channel]
    __shared__ __align__(8) float Bs[RB][NT];
    __shared__ __align__(8) float Cs[RB][NT];
    const int b0 = blockIdx.y * RB;
    const int nrow = min(RB, a.batch - b0);
    const int N = FULL ? NT : a.dstate, Dn = a.dinner;
    const int d = blockIdx.x * kStepThreads + threadIdx.x;
    const bool active = d < Dn;

    struct Row {
        float2 h[NP];                              // states (2p, 2p+1)
        float u, xr, z;
    };
    auto load_row = [&](Row& w, int b) {
        const float* hp = a.h + static_cast<size_t>(b) * N * Dn + d;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            w.h[p].x = 2 * p < N ? hp[static_cast<size_t>(2 * p) * Dn] : 0.0f;
            w.h[p].y = 2 * p + 1 < N ? hp[static_cast<size_t>(2 * p + 1) * Dn] : 0.0f;
        }
        w.u = Act<T>::load(static_cast<const T*>(a.u) + b * a.ld_u + d);
        w.xr = Act<T>::load(static_cast<const T*>(a.dr) + b * a.ld_dr + d);
        w.z = GATE ? Act<T>::load(static_cast<const T*>(a.z) + b * a.ld_z + d) : 0.0f;
    };
    Row cur, nxt;
    if (active) load_row(cur, b0);                 // the longest loads first
    if (active && nrow > 1) load_row(nxt, b0 + 1);

    // the rows' B and C, zero past dstate so that packed pairs need no guard
    for (int i = threadIdx.x; i < nrow * NT; i += kStepThreads) {
        const int r = i / NT, n = i % NT;
        Bs[r][n] = n < N ? Act<T>::load(static_cast<const T*>(a.B) + (b0 + r) * a.ld_B + n) : 0.0f;
        Cs[r][n] = n < N ? Act<T>::load(static_cast<const T*>(a.C) + (b0 + r) * a.ld_C + n) : 0.0f;
    }
    // A log2(e) = -2^(clamp(A_log) log2(e)) log2(e) of this channel (0 past
    // dstate: a = 1 there, and B = C = 0 keep those states at 0)
    if (active) {
        const float* al = a.A_log + static_cast<size_t>(d) * N;
        auto a2 = [](float v) { return -ex2(fminf(fmaxf(v, kALogLo), kALogHi) * kLog2e) * kLog2e; };
        if (FULL && NT == 16 && (reinterpret_cast<uintptr_t>(al) & 15u) == 0) {   // 4 x 16-byte loads
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 q = reinterpret_cast<const float4*>(al)[k];
                As[(2 * k) * kStepThreads + threadIdx.x] = make_float2(a2(q.x), a2(q.y));
                As[(2 * k + 1) * kStepThreads + threadIdx.x] = make_float2(a2(q.z), a2(q.w));
            }
        } else {
#pragma unroll
            for (int p = 0; p < NP; ++p)
                As[p * kStepThreads + threadIdx.x] =
                    make_float2(2 * p < N ? a2(al[2 * p]) : 0.0f, 2 * p + 1 < N ? a2(al[2 * p + 1]) : 0.0f);
        }
    }
    __syncthreads();
    if (!active) return;
    const float Dv = a.D ? a.D[d] : 0.0f;

#pragma unroll
    for (int r = 0; r < RB; ++r) {
        if (r >= nrow) break;
        const int b = b0 + r;
        if (r > 0 && r + 1 < nrow) load_row(nxt, b + 1);   // next row in flight during this one

        float dt, gz = 1.0f;
        if (GATE) {
            float sz;
            softplus_sigmoid(cur.xr, cur.z, dt, sz);
            gz = cur.z * sz;                               // silu(z)
        } else {
            float e;
            dt = softplus_e(cur.xr, e);
        }
        const float bs = DISC == 0 ? dt * cur.u : cur.u;   // Euler: delta*u; ZOH: u
        const float2 dt2 = f2(dt), bs2 = f2(bs);
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            if (2 * p >= N) break;
            const float2 A2 = As[p * kStepThreads + threadIdx.x];
            const float2 Bp = *reinterpret_cast<const float2*>(&Bs[r][2 * p]);
            const float2 Cp = *reinterpret_cast<const float2*>(&Cs[r][2 * p]);
            const float2 x = mul2(dt2, A2);
            const float2 av = make_float2(ex2(x.x), ex2(x.y));
            float2 bu;
            if (DISC == 0) {
                bu = mul2(bs2, Bp);
            } else {
                // beta/B = expm1(delta A)/A, without cancellation for small delta A
                float cf[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float Ae = (e ? A2.y : A2.x) * kLn2;
                    const float xn = dt * Ae;
                    const float ae = e ? av.y : av.x;
                    cf[e] = fabsf(xn) < 0.5f ? dt * phi1_series(xn) : (Ae != 0.0f ? (ae - 1.0f) / Ae : dt);
                }
                bu = mul2(mul2(make_float2(cf[0], cf[1]), bs2), Bp);
            }
            cur.h[p] = fma2(av, cur.h[p], bu);
            acc = fma2(Cp, cur.h[p], acc);
        }
        const float yv = fmaf(Dv, cur.u, acc.x + acc.y);
        float* hp = a.h + static_cast<size_t>(b) * N * Dn + d;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            if (2 * p < N) hp[static_cast<size_t>(2 * p) * Dn] = cur.h[p].x;
            if (2 * p + 1 < N) hp[static_cast<size_t>(2 * p + 1) * Dn] = cur.h[p].y;
        }
        static_cast<T*>(a.out)[b * a.ld_out + d] = Act<T>::from_f(GATE ? yv * gz : yv);
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
    if constexpr (K == 4) {
        // the 4 channels' taps are 16 contiguous floats: four 16-byte loads
        if ((reinterpret_cast<uintptr_t>(w) & 15u) == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 q = ld4f(w + 4 * c);
                wt[c][0] = q.x;
                wt[c][1] = q.y;
                wt[c][2] = q.z;
                wt[c][3] = q.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int k = 0; k < K; ++k) wt[c][k] = w[c * K + k];
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int k = 0; k < K; ++k) wt[c][k] = w[c * K + k];
    }
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
    const dim3 grid((a.dinner + kStepThreads - 1) / kStepThreads, (a.batch + kStepRows - 1) / kStepRows);
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

// conv1d.cu -- causal depthwise conv1d + SiLU, forward and backward, for sm_103a.
//
// mamba1_cpu.ts (page "@seanhogg/builderforce-memory-engine 2026.7.12 ->
// 2026.9.27"), mamba1CpuForward steps 4-5 and mamba1CpuBackward steps 5-4:
//   pre[r, d] = bias[d] + sum_{k < K, t >= k} w[d*K + k] * x[r - k, d]
//   out       = silu(pre)
//   dpre      = dout * silu'(pre);  dbias[d] = sum_r dpre;  dw[d,k] = sum_r dpre[r] x[r-k]
//   dx[r, d]  = sum_{k < K, t + k < L} w[d*K + k] * dpre[r + k, d]
// Tap k = 0 multiplies the CURRENT step.
//
// Design: the op is bound by HBM (one read of x and one write of out per
// element).  A thread owns 4 adjacent channels (one 16-byte access per row,
// 512 contiguous bytes per warp) and walks a run of kConvRun rows, keeping the
// last K rows of x (and, backward, of dpre) in registers, so each element is
// read from HBM once plus a (K-1)/kConvRun halo.  The rows are taken in small
// groups whose loads are all issued before the group's first store, so that
// several loads per thread are in flight (one at a time, the kernels reached
// about half of the HBM bandwidth).
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "conv_args.cuh"
#include "ssm_common.cuh"

namespace ssm {

// rows whose loads a thread issues together before it uses them (measured
// best: 4 forward, 8 backward; 4 backward for kconv > 4, whose larger
// register windows would spill with 8)
constexpr int kConvGroupFwd = 4;
constexpr int kConvGroupBwd = 8;
constexpr int kConvThreads = 128;

__device__ __forceinline__ float silu_f(float x) { return x * rcp(1.0f + ex2(-x * kLog2e)); }
__device__ __forceinline__ float silu_grad_f(float x) {
    const float s = rcp(1.0f + ex2(-x * kLog2e));
    return s * (1.0f + x * (1.0f - s));
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// The 4 channels' taps (4 x K contiguous floats at w + d0*K) as w4[k] = tap k
// of the 4 channels: K 16-byte loads when aligned.
template <int K>
__device__ __forceinline__ void load_taps(const float* wp, float4 (&w4)[K]) {
    float f[4 * K];
    if ((reinterpret_cast<uintptr_t>(wp) & 15u) == 0) {
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const float4 v = ld4(wp + 4 * i);
            f[4 * i] = v.x;
            f[4 * i + 1] = v.y;
            f[4 * i + 2] = v.z;
            f[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4 * K; ++i) f[i] = wp[i];
    }
#pragma unroll
    for (int k = 0; k < K; ++k) w4[k] = make_float4(f[k], f[K + k], f[2 * K + k], f[3 * K + k]);
}

template <int K>
__global__ void __launch_bounds__(kConvThreads)
conv1d_silu_fwd_kernel(const ConvArgs a) {
    constexpr int G = kConvGroupFwd;
    const int nq = a.dinner / 4;
    const int runs = (a.seqlen + kConvRun - 1) / kConvRun;
    const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long total = static_cast<long long>(nq) * runs * a.batch;
    if (gid >= total) return;
    const int q = static_cast<int>(gid % nq);
    const long long rest = gid / nq;
    const int run = static_cast<int>(rest % runs);
    const int b = static_cast<int>(rest / runs);
    const int d0 = 4 * q;
    const float* __restrict__ x = a.x;
    float* __restrict__ out = a.out;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 w[K];
    load_taps<K>(a.w + static_cast<size_t>(d0) * K, w);
    const float4 bias = a.bias ? ld4(a.bias + d0) : z4;
    const int t0 = run * kConvRun;
    const int t1 = min(a.seqlen, t0 + kConvRun);
    const size_t row0 = static_cast<size_t>(b) * a.seqlen;
    float4 xw[K];   // xw[k] = x[t - 1 - k] before step t's shift; zeros before the sequence
#pragma unroll
    for (int k = 0; k < K; ++k) xw[k] = z4;
    if constexpr (K > 1) {
        float4 hl[K - 1];   // halo rows t0-K+1 .. t0-1, loaded at once
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            const int t = t0 - (K - 1) + j;
            hl[j] = t >= 0 ? ld4(x + (row0 + t) * a.ld_x + d0) : z4;
        }
#pragma unroll
        for (int k = 0; k < K - 1; ++k) xw[k] = hl[K - 2 - k];
    }
    // groups of G rows: the group's loads are issued before any of its stores
    for (int tb = t0; tb < t1; tb += G) {
        float4 xn[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int t = tb + g;
            xn[g] = t < t1 ? ld4(x + (row0 + t) * a.ld_x + d0) : z4;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int t = tb + g;
            if (t < t1) {
#pragma unroll
                for (int k = K - 1; k > 0; --k) xw[k] = xw[k - 1];
                xw[0] = xn[g];
                float4 acc = bias;
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    acc.x = fmaf(w[k].x, xw[k].x, acc.x);
                    acc.y = fmaf(w[k].y, xw[k].y, acc.y);
                    acc.z = fmaf(w[k].z, xw[k].z, acc.z);
                    acc.w = fmaf(w[k].w, xw[k].w, acc.w);
                }
                st4(out + (row0 + t) * a.ld_out + d0,
                    make_float4(silu_f(acc.x), silu_f(acc.y), silu_f(acc.z), silu_f(acc.w)));
            }
        }
    }
}

// Backward: per run, dx for its rows and partial dw / dbias (written to the
// workspace, reduced over runs by conv1d_reduce_kernel).  Rows are taken in
// groups of kConvGroupBwd whose x and dout loads are issued together.
template <int K>
__global__ void __launch_bounds__(kConvThreads)
conv1d_silu_bwd_kernel(const ConvArgs a) {
    constexpr int G = K <= 4 ? kConvGroupBwd : kConvGroupFwd;
    const int nq = a.dinner / 4;
    const int runs = (a.seqlen + kConvRun - 1) / kConvRun;
    const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long total = static_cast<long long>(nq) * runs * a.batch;
    if (gid >= total) return;
    const int q = static_cast<int>(gid % nq);
    const long long rest = gid / nq;
    const int run = static_cast<int>(rest % runs);
    const int b = static_cast<int>(rest / runs);
    const int d0 = 4 * q;
    const int L = a.seqlen;
    const float* __restrict__ x = a.x;
    const float* __restrict__ dout = a.dout;
    float* __restrict__ dx = a.dx;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 w[K];
    load_taps<K>(a.w + static_cast<size_t>(d0) * K, w);
    const float4 bias = a.bias ? ld4(a.bias + d0) : z4;
    const int t0 = run * kConvRun;
    const int t1 = min(L, t0 + kConvRun);
    const size_t row0 = static_cast<size_t>(b) * L;
    float4 xw[K], gw[K];   // xw[k] = x[s-k], gw[k] = dpre[s-k]
#pragma unroll
    for (int k = 0; k < K; ++k) xw[k] = gw[k] = z4;
    float4 dwa[K], dba = z4;
#pragma unroll
    for (int k = 0; k < K; ++k) dwa[k] = z4;

    const int s_begin = max(0, t0 - K + 1), s_end = t1 + K - 1;
    for (int sb = s_begin; sb < s_end; sb += G) {
        float4 xn[G], gn[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int s = sb + g;
            const bool in = s < s_end && s < L;
            xn[g] = in ? ld4(x + (row0 + s) * a.ld_x + d0) : z4;
            gn[g] = in && s >= t0 ? ld4(dout + (row0 + s) * a.ld_dout + d0) : z4;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int s = sb + g;
            if (s < s_end) {
#pragma unroll
                for (int k = K - 1; k > 0; --k) {
                    xw[k] = xw[k - 1];
                    gw[k] = gw[k - 1];
                }
                xw[0] = xn[g];
                float4 gv = z4;
                if (s < L && s >= t0) {
                    float4 p = bias;
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        p.x = fmaf(w[k].x, xw[k].x, p.x);
                        p.y = fmaf(w[k].y, xw[k].y, p.y);
                        p.z = fmaf(w[k].z, xw[k].z, p.z);
                        p.w = fmaf(w[k].w, xw[k].w, p.w);
                    }
                    const float4 go = gn[g];
                    gv = make_float4(go.x * silu_grad_f(p.x), go.y * silu_grad_f(p.y),
                                     go.z * silu_grad_f(p.z), go.w * silu_grad_f(p.w));
                    if (s < t1) {
                        dba.x += gv.x; dba.y += gv.y; dba.z += gv.z; dba.w += gv.w;
#pragma unroll
                        for (int k = 0; k < K; ++k) {
                            dwa[k].x = fmaf(gv.x, xw[k].x, dwa[k].x);
                            dwa[k].y = fmaf(gv.y, xw[k].y, dwa[k].y);
                            dwa[k].z = fmaf(gv.z, xw[k].z, dwa[k].z);
                            dwa[k].w = fmaf(gv.w, xw[k].w, dwa[k].w);
                        }
                    }
                }
                gw[0] = gv;
                const int r = s - (K - 1);   // dx[r] = sum_k w[k] dpre[r+k] is complete now
                if (r >= t0 && r < t1) {
                    float4 acc = z4;
#pragma unroll
                    for (int k = 0; k < K; ++k) {   // dpre[r + k] sits in gw[K - 1 - k]
                        const float4 gk = gw[K - 1 - k];
                        acc.x = fmaf(w[k].x, gk.x, acc.x);
                        acc.y = fmaf(w[k].y, gk.y, acc.y);
                        acc.z = fmaf(w[k].z, gk.z, acc.z);
                        acc.w = fmaf(w[k].w, gk.w, acc.w);
                    }
                    st4(dx + (row0 + r) * a.ld_dx + d0, acc);
                }
            }
        }
    }
    // partial dw | dbias of this run: ws[(b*runs + run)][d][K+1]
    float* wsr = a.ws + (static_cast<size_t>(b) * runs + run) * a.dinner * (K + 1);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float* dst = wsr + static_cast<size_t>(d0 + c) * (K + 1);
#pragma unroll
        for (int k = 0; k < K; ++k)
            dst[k] = c == 0 ? dwa[k].x : c == 1 ? dwa[k].y : c == 2 ? dwa[k].z : dwa[k].w;
        dst[K] = c == 0 ? dba.x : c == 1 ? dba.y : c == 2 ? dba.z : dba.w;
    }
}

// Sum of the per-run dw | dbias partials: a CTA owns 32 columns of
// [dinner][K+1]; its 8 warps each add every 8th partial (lane = column, so a
// warp's loads are 128 contiguous bytes), then warp 0 adds the 8 warp sums in
// a fixed order (the result does not depend on scheduling).
constexpr int kReduceSlices = 8;
__global__ void __launch_bounds__(32 * kReduceSlices)
conv1d_reduce_kernel(const ConvArgs a, int nparts) {
    __shared__ float part[kReduceSlices][32];
    const int K = a.kconv;
    const int total = a.dinner * (K + 1);
    const int lane = threadIdx.x & 31, sl = threadIdx.x >> 5;
    const int i = blockIdx.x * 32 + lane;
    float s = 0.0f;
    if (i < total) {
#pragma unroll 4
        for (int p = sl; p < nparts; p += kReduceSlices) s += a.ws[static_cast<size_t>(p) * total + i];
    }
    part[sl][lane] = s;
    __syncthreads();
    if (sl == 0 && i < total) {
        float t = part[0][lane];
#pragma unroll
        for (int w = 1; w < kReduceSlices; ++w) t += part[w][lane];
        const int d = i / (K + 1), k = i % (K + 1);
        if (k < K) a.dw[d * K + k] = t;
        else if (a.dbias) a.dbias[d] = t;
    }
}

static unsigned blocks_for(long long n) {
    return static_cast<unsigned>((n + kConvThreads - 1) / kConvThreads);
}

template <template <int> class Sel>
static cudaError_t dispatch_k(int k, const ConvArgs& a, unsigned blocks, cudaStream_t st) {
    switch (k) {
        case 1: Sel<1>::run(a, blocks, st); break;
        case 2: Sel<2>::run(a, blocks, st); break;
        case 3: Sel<3>::run(a, blocks, st); break;
        case 4: Sel<4>::run(a, blocks, st); break;
        case 5: Sel<5>::run(a, blocks, st); break;
        case 6: Sel<6>::run(a, blocks, st); break;
        case 7: Sel<7>::run(a, blocks, st); break;
        case 8: Sel<8>::run(a, blocks, st); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}
template <int K> struct FwdSel {
    static void run(const ConvArgs& a, unsigned bl, cudaStream_t st) {
        conv1d_silu_fwd_kernel<K><<<bl, kConvThreads, 0, st>>>(a);
    }
};
template <int K> struct BwdSel {
    static void run(const ConvArgs& a, unsigned bl, cudaStream_t st) {
        conv1d_silu_bwd_kernel<K><<<bl, kConvThreads, 0, st>>>(a);
    }
};

cudaError_t launch_conv1d_fwd(const ConvArgs& a, cudaStream_t st) {
    const long long runs = (a.seqlen + kConvRun - 1) / kConvRun;
    const long long total = static_cast<long long>(a.dinner / 4) * runs * a.batch;
    if (total == 0) return cudaSuccess;
    return dispatch_k<FwdSel>(a.kconv, a, blocks_for(total), st);
}

cudaError_t launch_conv1d_bwd(const ConvArgs& a, cudaStream_t st) {
    const long long runs = (a.seqlen + kConvRun - 1) / kConvRun;
    const long long total = static_cast<long long>(a.dinner / 4) * runs * a.batch;
    if (total > 0) {
        cudaError_t e = dispatch_k<BwdSel>(a.kconv, a, blocks_for(total), st);
        if (e != cudaSuccess) return e;
    }
    const int nparts = static_cast<int>(runs * a.batch);
    const int n = a.dinner * (a.kconv + 1);
    if (n == 0) return cudaSuccess;
    conv1d_reduce_kernel<<<(n + 31) / 32, 32 * kReduceSlices, 0, st>>>(a, nparts);
    return cudaGetLastError();
}

// Scratch for the allocation-free backward entry point: the per-run dw/dbias
// partial sums live in this file-scope array instead of a caller workspace.
// Every GPU that loads the library keeps these kConvNoAllocScratchFloats floats
// (8 MiB) until the process exits.
static __device__ __align__(256) float g_conv_bwd_scratch[kConvNoAllocScratchFloats];

// Identity of the calling thread's current CUDA context (cuCtxGetId: unique
// for the life of the process, so a context destroyed and created again --
// cudaDeviceReset, or the primary context released and retained anew -- gets
// a new one), or 0 when no context is current or the driver cannot say.
static unsigned long long current_context_id() {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_conv_bwd_scratch in the current device's context (the
// array's name is only a host-side stand-in; the kernel needs this address).
// It is looked up with cudaGetSymbolAddress once per device and context and
// kept keyed on the context's identity, so a call after a device reset (the
// module reloaded, perhaps at another address) looks it up again; if the
// context cannot be identified it is looked up at every call.  Returns the
// cudaGetSymbolAddress error, if any.
cudaError_t conv1d_noalloc_scratch(float** out) {
    struct Entry {
        unsigned long long ctx;
        float* addr;
    };
    static std::mutex mu;
    static Entry cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && cache[dev].ctx == ctx && cache[dev].addr) {
        *out = cache[dev].addr;
        return cudaSuccess;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_conv_bwd_scratch);   // also makes the primary context current
    if (e != cudaSuccess) return e;
    cache[dev].ctx = current_context_id();
    cache[dev].addr = static_cast<float*>(p);
    *out = cache[dev].addr;
    return cudaSuccess;
}

size_t conv1d_bwd_workspace_bytes(int batch, int seqlen, int dinner, int kconv) {
    const size_t runs = (static_cast<size_t>(seqlen) + kConvRun - 1) / kConvRun;
    return runs * batch * dinner * (kconv + 1) * sizeof(float);
}

}  // namespace ssm

// probe.cu -- throughput probes of three arithmetic pipes of the SM: the MUFU
// ex2 unit, scalar fp32 FFMA and packed f32x2 FFMA2.  The scan's roofline
// divides its exponential count by the ex2 rate and its fp32 lane-operation
// count by the FFMA rate; these kernels measure both on the device at hand
// (the benchmark times them with CUDA events and the sampled SM clock).
//
// Every thread runs 8 independent dependency chains (4 packed pairs for
// FFMA2), so with 8 warps per SMSP the pipe, not the chain latency, sets the
// rate.  The chains stay bounded (ex2: x <- 2^-x converges to ~0.64; FFMA:
// x <- a x + b with |a| < 1), and each thread's sum is stored so nothing is
// dead code.
#include <cuda_runtime.h>

#include "ssm_common.cuh"
#include "ssm_gb300.h"

namespace {

// Self-test of the bounded waits: arm an mbarrier for 16 bytes of a copy that
// is never issued and wait on it with at most `limit` polls.  The wait gives
// up, records kFaultSelftest in this file's fault word and the kernel returns
// (nothing is in flight, so the barrier can simply be abandoned).
__global__ void bounded_wait_selftest_kernel(uint32_t limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ssm::mbar_init(&bar, 1);
        ssm::fence_mbar_init();
        ssm::mbar_arrive_expect_tx(&bar, 16);
        ssm::mbar_wait(&bar, 0, ssm::kFaultSelftest, limit);
    }
}

__device__ __forceinline__ float ex2_neg(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(-x));
    return y;
}

constexpr int kProbeThreads = 256;

template <int KIND>
__global__ void __launch_bounds__(kProbeThreads) pipe_probe_kernel(int iters, float a, float b,
                                                                   float* sink) {
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    float x[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = 0.25f + 0.01f * c + 1e-6f * (tid & 255);
    if constexpr (KIND == 0) {
#pragma unroll 4
        for (int it = 0; it < iters; ++it)
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = ex2_neg(x[c]);
    } else if constexpr (KIND == 1) {
#pragma unroll 4
        for (int it = 0; it < iters; ++it)
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = fmaf(x[c], a, b);
    } else if constexpr (KIND == 2) {
        float2 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = make_float2(x[2 * c], x[2 * c + 1]);
        const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
#pragma unroll 4
        for (int it = 0; it < iters; ++it)
#pragma unroll
            for (int c = 0; c < 4; ++c) v[c] = __ffma2_rn(v[c], a2, b2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            x[2 * c] = v[c].x;
            x[2 * c + 1] = v[c].y;
        }
    } else {
        // 3: a packed FFMA2 whose multiplier is a scalar that changes every
        // step, broadcast to both halves; 4: the same multiplier kept as a
        // pair (updated with FFMA2).  Their instruction counts per step show
        // what a scalar-to-pair broadcast costs.
        float2 v[4], s2[4];
        float s1[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            v[c] = make_float2(x[2 * c], x[2 * c + 1]);
            s1[c] = 0.5f + 0.01f * c;
            s2[c] = make_float2(s1[c], s1[c]);
        }
        const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
#pragma unroll 1
        for (int it = 0; it < iters; ++it)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if constexpr (KIND == 3) {
                    s1[c] = fmaf(s1[c], a, b);
                    v[c] = __ffma2_rn(v[c], make_float2(s1[c], s1[c]), b2);
                } else {
                    s2[c] = __ffma2_rn(s2[c], a2, b2);
                    v[c] = __ffma2_rn(v[c], s2[c], b2);
                }
            }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            x[2 * c] = v[c].x + s1[c];
            x[2 * c + 1] = v[c].y + s2[c].y;
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) s += x[c];
    sink[tid] = s;
}

}  // namespace

extern "C" ssm_status ssm_probe_pipe(int32_t kind, int32_t blocks, int32_t iters, float* sink,
                                     cudaStream_t stream) {
    if (kind < 0 || kind > 4 || blocks <= 0 || iters <= 0) return SSM_ERR_SHAPE;
    if (!sink) return SSM_ERR_NULL;
    // the inner loop is unrolled by 8 chains; a and b keep the fma chains in (0, 1)
    const float a = 0.999f, b = 0.0005f;
    switch (kind) {
        case 0: pipe_probe_kernel<0><<<blocks, kProbeThreads, 0, stream>>>(iters, a, b, sink); break;
        case 1: pipe_probe_kernel<1><<<blocks, kProbeThreads, 0, stream>>>(iters, a, b, sink); break;
        case 2: pipe_probe_kernel<2><<<blocks, kProbeThreads, 0, stream>>>(iters, a, b, sink); break;
        case 3: pipe_probe_kernel<3><<<blocks, kProbeThreads, 0, stream>>>(iters, a, b, sink); break;
        default: pipe_probe_kernel<4><<<blocks, kProbeThreads, 0, stream>>>(iters, a, b, sink); break;
    }
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

extern "C" ssm_status ssm_selftest_bounded_wait(uint32_t poll_limit, cudaStream_t stream) {
    if (poll_limit == 0 || poll_limit > (1u << 20)) return SSM_ERR_SHAPE;
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(poll_limit);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

namespace ssm {
cudaError_t read_clear_fault_probe(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_ssm_fault, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_ssm_fault, &zero, sizeof(unsigned));
}
}  // namespace ssm

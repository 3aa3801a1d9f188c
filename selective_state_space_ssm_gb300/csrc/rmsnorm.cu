// rmsnorm.cu -- RMSNorm forward and backward of the Mamba-1 block
// (cpu_ops.ts rmsNormForward / rmsNormBackward).  One warp per row; the
// weight gradient is a fixed-order column reduction (no atomics), so repeated
// runs give identical bits.
#include <algorithm>

#include "gemm_args.cuh"

namespace ssm {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kRowsPerBlock = 8;   // one warp per row
constexpr int kDwRows = 512;       // rows per weight-gradient partial

}  // namespace

__global__ void rmsnorm_fwd_kernel(const float* __restrict__ x, const float* __restrict__ w, int rows,
                                   int dm, float eps, float* __restrict__ y, float* __restrict__ inv) {
    const int r = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float* xr = x + static_cast<size_t>(r) * dm;
    float sq = 0.0f;
    for (int i = lane; i < dm; i += 32) sq = fmaf(xr[i], xr[i], sq);
    sq = warp_sum(sq);
    const float iv = 1.0f / sqrtf(sq / static_cast<float>(dm) + eps);
    if (lane == 0) inv[r] = iv;
    float* yr = y + static_cast<size_t>(r) * dm;
    for (int i = lane; i < dm; i += 32) yr[i] = xr[i] * iv * w[i];
}

// dx = res + g inv - inv^3 / dm * (sum_j g_j x_j) x, g = dy w.
__global__ void rmsnorm_bwd_dx_kernel(const float* __restrict__ dy, const float* __restrict__ x,
                                      const float* __restrict__ w, const float* __restrict__ inv,
                                      const float* __restrict__ res, int rows, int dm,
                                      float* __restrict__ dx) {
    const int r = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const size_t off = static_cast<size_t>(r) * dm;
    float dot = 0.0f;
    for (int i = lane; i < dm; i += 32) dot = fmaf(dy[off + i] * w[i], x[off + i], dot);
    dot = warp_sum(dot);
    const float iv = inv[r];
    const float s = iv * iv * iv / static_cast<float>(dm) * dot;
    for (int i = lane; i < dm; i += 32) {
        const float g = dy[off + i] * w[i];
        float v = g * iv - s * x[off + i];
        if (res) v += res[off + i];
        dx[off + i] = v;
    }
}

// Partial column sums of dy * x * inv over kDwRows-row slabs.
__global__ void rmsnorm_dw_partial_kernel(const float* __restrict__ dy, const float* __restrict__ x,
                                          const float* __restrict__ inv, int rows, int dm,
                                          float* __restrict__ part) {
    __shared__ float red[8][33];
    const int c = blockIdx.x * 32 + (threadIdx.x & 31);
    const int g = threadIdx.x >> 5;
    const int r0 = blockIdx.y * kDwRows;
    const int r1 = min(rows, r0 + kDwRows);
    float s = 0.0f;
    if (c < dm)
        for (int r = r0 + g; r < r1; r += 8) {
            const size_t o = static_cast<size_t>(r) * dm + c;
            s = fmaf(dy[o] * x[o], inv[r], s);
        }
    red[g][threadIdx.x & 31] = s;
    __syncthreads();
    if (g == 0 && c < dm) {
        float t = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) t += red[k][threadIdx.x & 31];
        part[static_cast<size_t>(blockIdx.y) * dm + c] = t;
    }
}

__global__ void rmsnorm_dw_final_kernel(const float* __restrict__ part, int nparts, int dm,
                                        float* __restrict__ dw) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= dm) return;
    float s = 0.0f;
    for (int p = 0; p < nparts; ++p) s += part[static_cast<size_t>(p) * dm + c];
    dw[c] = s;
}

cudaError_t launch_rmsnorm_fwd(const float* x, const float* w, int rows, int dm, float eps, float* y,
                               float* inv, cudaStream_t st) {
    if (rows == 0 || dm == 0) return cudaSuccess;
    rmsnorm_fwd_kernel<<<(rows + kRowsPerBlock - 1) / kRowsPerBlock, 32 * kRowsPerBlock, 0, st>>>(
        x, w, rows, dm, eps, y, inv);
    return cudaGetLastError();
}

size_t rmsnorm_ws_floats(int rows, int dm) {
    return static_cast<size_t>((rows + kDwRows - 1) / kDwRows) * dm;
}

cudaError_t launch_rmsnorm_bwd(const float* dy, const float* x, const float* w, const float* inv,
                               const float* res, int rows, int dm, float* dx, float* dw, float* ws,
                               cudaStream_t st) {
    if (dm == 0) return cudaSuccess;
    if (rows > 0) {
        rmsnorm_bwd_dx_kernel<<<(rows + kRowsPerBlock - 1) / kRowsPerBlock, 32 * kRowsPerBlock, 0, st>>>(
            dy, x, w, inv, res, rows, dm, dx);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        dim3 grid((dm + 31) / 32, (rows + kDwRows - 1) / kDwRows);
        rmsnorm_dw_partial_kernel<<<grid, 256, 0, st>>>(dy, x, inv, rows, dm, ws);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    rmsnorm_dw_final_kernel<<<(dm + 255) / 256, 256, 0, st>>>(ws, (rows + kDwRows - 1) / kDwRows, dm, dw);
    return cudaGetLastError();
}

}  // namespace ssm

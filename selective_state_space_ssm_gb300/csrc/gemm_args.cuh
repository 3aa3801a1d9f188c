// gemm_args.cuh -- argument blocks of the fp32 linear-algebra kernels
// (gemm.cu, rmsnorm.cu) shared with the C-ABI layer (abi.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

// TN GEMM tile: 128 x 128 output, K in blocks of 32 fp32 (one 128-byte
// swizzle row); kGemmStages raw fp32 A|B stages in flight by TMA and
// kGemmLoBufs K-blocks split ahead of the MMAs (A hi/lo in tensor memory,
// B lo in shared memory).
constexpr int kGemmBM = 128;
constexpr int kGemmBN = 128;
constexpr int kGemmBK = 32;
constexpr int kGemmStages = 5;
constexpr int kGemmLoBufs = 3;
// 16 warps in four warpgroups; registers per thread after the split: the
// producer/MMA/B warpgroup kGemmRegsSmall, the two A warpgroups
// kGemmRegsConv, the epilogue kGemmRegsEpi.
constexpr int kGemmThreads = 512;
constexpr int kGemmRegsSmall = 96;
constexpr int kGemmRegsConv = 88;
constexpr int kGemmRegsEpi = 240;
// K-blocks accumulated by the tensor core before the partial sum is added into
// fp32 registers (bounds the tensor core's accumulation drift at 128 products).
constexpr int kGemmGroup = 4;

// C[m, n] = sum_k A[m, k] B[n, k] (+ bias[n]) (+ R[m, n]), fp32 in and out,
// computed as three TF32 tensor-core products of hi/lo splits
// (A_hi B_hi + A_hi B_lo + A_lo B_hi) accumulated in fp32 in tensor memory;
// the kernel forms the splits itself from the fp32 tiles.  A is (M, K) and B
// is (N, K), row-major, K-contiguous, each with a row stride whose byte size
// is a multiple of 16 and a 16-byte-aligned base (TMA).
struct GemmArgs {
    float* C;
    const float* bias;   // may be null
    const float* R;      // may be null; may alias C (accumulate)
    int M, N, K;
    int64_t ldc, ldr;
    int ksplit;          // K slices computed by separate CTAs (1: none)
    float* part;         // ksplit > 1: [ksplit][M][N] partial sums (workspace)
};
// Split-K for GEMMs whose output tiles leave SMs idle: returns the number of
// K slices (1 = none) given the partial-sum space available (floats).
inline int gemm_ksplit(int M, int N, int K, size_t part_floats) {
    const long long tiles = static_cast<long long>((M + kGemmBM - 1) / kGemmBM) * ((N + kGemmBN - 1) / kGemmBN);
    const int nk = (K + kGemmBK - 1) / kGemmBK;
    if (tiles >= 152 || nk < 16) return 1;
    long long ks = (2 * 152 + tiles - 1) / tiles;
    if (ks > nk / 8) ks = nk / 8;
    while (ks > 1 && static_cast<size_t>(ks) * M * N > part_floats) --ks;
    return ks < 1 ? 1 : static_cast<int>(ks);
}
struct GemmMaps {
    CUtensorMap a, b;
};

cudaError_t launch_gemm_tf32x3(const GemmMaps& maps, const GemmArgs& a, cudaStream_t st);

// Copy of a (rows, cols) fp32 matrix with row stride ldx into out with row
// stride ldo: as it is (transpose = 0) or transposed to (cols, rows)
// (transpose = 1) -- GEMM operands that are not K-major or not TMA-aligned.
cudaError_t launch_operand_copy(const float* x, int64_t ldx, int rows, int cols, int transpose,
                                float* out, int64_t ldo, cudaStream_t st);

// out[n] = sum_m x[m, n] (fixed-order partial sums, no atomics); ws must hold
// colsum_ws_floats(rows, cols) floats.
size_t colsum_ws_floats(int rows, int cols);
cudaError_t launch_colsum(const float* x, int64_t ldx, int rows, int cols, float* out, float* ws,
                          cudaStream_t st);
// The transposed operand copy of launch_operand_copy (transpose = 1) that also
// writes colsum[n] = sum_m x[m, n] (null: the copy only) from the same pass
// over x when the copy takes 16-byte accesses; ws as for launch_colsum.
cudaError_t launch_operand_copy_t_colsum(const float* x, int64_t ldx, int rows, int cols, float* out,
                                         int64_t ldo, float* colsum, float* ws, cudaStream_t st);

// RMSNorm of cpu_ops.ts: inv[r] = 1/sqrt(mean_i x[r,i]^2 + eps); y = x inv w.
cudaError_t launch_rmsnorm_fwd(const float* x, const float* w, int rows, int dm, float eps,
                               float* y, float* inv, cudaStream_t st);
// Backward: dx[r,i] = res[r,i] + g_i inv - inv^3/dm * (sum_j g_j x_j) x_i with
// g = dy w (res may be null); dw = sum_r dy x inv (written; ws must hold
// rmsnorm_ws_floats(rows, dm) floats).
size_t rmsnorm_ws_floats(int rows, int dm);
cudaError_t launch_rmsnorm_bwd(const float* dy, const float* x, const float* w, const float* inv,
                               const float* res, int rows, int dm, float* dx, float* dw, float* ws,
                               cudaStream_t st);

// Reads and clears the bounded-wait fault word of the GEMM kernel.
cudaError_t read_clear_fault_gemm(unsigned* out);

}  // namespace ssm

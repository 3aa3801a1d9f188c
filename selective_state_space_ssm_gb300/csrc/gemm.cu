// gemm.cu -- fp32-accurate tensor-core GEMM for the Mamba-1 block projections
// (cpu_ops.ts linearForward / linearBackward: Y = X W^T + b, dX = dY W,
// dW = dY^T X), plus operand copies (transposes) and deterministic column
// sums.
//
// sm_103a design: one CTA computes a 128 x 128 tile of C = A B^T with
// tcgen05.mma (kind::tf32, cta_group::1, M = 128, N = 128, K = 8 per
// instruction) accumulating in tensor memory, as three TF32 products
// A_hi B_hi + A_hi B_lo + A_lo B_hi (about fp32 accuracy).  The tensor core
// reads a tf32 operand from an fp32 word and ignores its low 13 mantissa
// bits, so the raw fp32 tiles serve as the "hi" operands: warp 0 streams
// 128 x 32 fp32 tiles of A and B with TMA (128-byte swizzle) through a
// three-stage mbarrier pipeline, and the four epilogue warps (2-5) write the
// "lo" tiles (x minus x with its low 13 mantissa bits cleared: exact) next to
// them in shared memory, at the same swizzled offsets; one thread of warp 1
// issues the MMAs.  Compared with splitting the operands into hi/lo arrays
// beforehand, half the operand bytes cross L2 and no split pass runs.  The
// tensor core's fp32 accumulation drifts in one direction (its error grows
// linearly with K), so the accumulator is double-buffered in tensor memory and
// read back into fp32 registers every kGemmGroup K-blocks by the same
// epilogue warps, one group behind the conversion.  Every mbarrier wait is
// bounded; tensor memory is always released.
#include <algorithm>

#include "gemm_args.cuh"
#include "ssm_common.cuh"

namespace ssm {

constexpr unsigned kFaultGemm = 8u;
constexpr uint32_t kTmemCols = 2 * kGemmBN;                     // two fp32 accumulators
constexpr uint32_t kOpTileBytes = kGemmBM * kGemmBK * 4;         // 16 KB (BM == BN)
constexpr uint32_t kPairBytes = 2 * kOpTileBytes;                // [A][B] of one K-block
// Shared memory: kGemmStages raw stages [A raw][B raw], then kGemmLoBufs
// buffers [A lo][B lo], 32 KB each.
constexpr int kTileFloats = kGemmBM * kGemmBK;
static_assert(kGemmBM == kGemmBN, "square tiles share one tile size");

// Shared-memory matrix descriptor of a K-major operand tile laid out by TMA
// with the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);          // start address
    d |= static_cast<uint64_t>(1) << 16;                         // leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // stride offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                         // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                         // 128-byte swizzle
    return d;
}

// Instruction descriptor: D fp32, A and B tf32, both K-major, M = 128, N = 128.
constexpr uint32_t kIdescTF32 = (1u << 4) | (2u << 7) | (2u << 10) |
                                (static_cast<uint32_t>(kGemmBN >> 3) << 17) |
                                (static_cast<uint32_t>(kGemmBM >> 4) << 24);

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdescTF32), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
#define SSM_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : SSM_R8(0), SSM_R8(8), SSM_R8(16), SSM_R8(24)
        : "r"(taddr)
        : "memory");
}
#undef SSM_R8
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(192, 1)
gemm_tf32x3_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    constexpr int S = kGemmStages;
    constexpr int NL = kGemmLoBufs;
    constexpr int G = kGemmGroup;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* lobuf = smem + S * kPairBytes;                                 // [NL][A lo][B lo]
    uint64_t* full = reinterpret_cast<uint64_t*>(lobuf + NL * kPairBytes);        // [S] raw tiles landed
    uint64_t* conv = full + S;           // [NL] the lo tiles are written (one arrival per epilogue warp)
    uint64_t* empty = conv + NL;         // [S] the MMAs of that K-block are done (stage and its lo buffer free)
    uint64_t* acc_full = empty + S;      // [2] a partial accumulator is complete
    uint64_t* acc_empty = acc_full + 2;  // [2] the epilogue has read it back
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kGemmBN, m0 = blockIdx.y * kGemmBM;
    // this CTA's K range (split-K: blockIdx.z of ksplit slices, partial sums to
    // a.part, added up by gemm_splitk_reduce_kernel)
    const int nk_all = (a.K + kGemmBK - 1) / kGemmBK;
    const int per = (nk_all + a.ksplit - 1) / a.ksplit;
    const int kb0 = blockIdx.z * per;
    const int nk = max(0, min(per, nk_all - kb0));
    const int ngroups = (nk + G - 1) / G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int l = 0; l < NL; ++l) mbar_init(&conv[l], 4);   // one arrival per epilogue warp
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);   // one arrival per epilogue warp
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {   // TMA producer: the raw fp32 tiles of A and B
            int kb = 0;
            for (; kb < nk; ++kb) {
                const int s = kb % S;
                if (kb >= S && !mbar_wait(&empty[s], ((kb / S) - 1) & 1, kFaultGemm)) break;
                unsigned char* st = smem + s * kPairBytes;
                mbar_arrive_expect_tx(&full[s], kPairBytes);
                const int kx = (kb0 + kb) * kGemmBK;
                tma_load_2d(st, &maps.a, &full[s], kx, m0);
                tma_load_2d(st + kOpTileBytes, &maps.b, &full[s], kx, n0);
            }
            // copies still in flight land before the CTA may exit (bounded)
            for (int j = std::max(0, kb - S); j < kb; ++j)
                mbar_wait(&full[j % S], (j / S) & 1, kFaultDrain);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            bool ok = true;
            for (int gi = 0; gi < ngroups && ok; ++gi) {
                const int buf = gi & 1;
                // the epilogue must have read this buffer's previous group
                if (gi >= 2 && !mbar_wait(&acc_empty[buf], ((gi >> 1) - 1) & 1, kFaultGemm)) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(buf * kGemmBN);
                const int kb1 = std::min(nk, (gi + 1) * G);
                for (int kb = gi * G; kb < kb1; ++kb) {
                    const int s = kb % S, l = kb % NL;
                    if (!mbar_wait(&conv[l], (kb / NL) & 1, kFaultGemm)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + s * kPairBytes);
                    const uint32_t lt = smem_u32(lobuf + l * kPairBytes);
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 8; ++kk) {
                        const uint32_t off = kk * 32;   // 8 tf32 = 32 bytes along K
                        const uint64_t ahi = umma_desc_sw128(st + off);
                        const uint64_t bhi = umma_desc_sw128(st + kOpTileBytes + off);
                        const uint64_t alo = umma_desc_sw128(lt + off);
                        const uint64_t blo = umma_desc_sw128(lt + kOpTileBytes + off);
                        umma_tf32(d, ahi, bhi, (kb != gi * G || kk != 0) ? 1u : 0u);
                        umma_tf32(d, ahi, blo, 1u);
                        umma_tf32(d, alo, bhi, 1u);
                    }
                    umma_commit(&empty[s]);   // stage s and lo buffer l are free once these MMAs finish
                }
                umma_commit(&acc_full[buf]);  // this group's partial sum is complete
            }
        }
    } else {   // warps 2..5: lo tiles, then the epilogue; TMEM lane quadrant = warp % 4
        const int q = warp & 3;
        const int et = threadIdx.x - 64;   // 0..127
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
        // Each group's partial sum (at most G K-blocks, accumulated by the tensor
        // core) is added into fp32 registers, so the tensor core's own
        // accumulation never spans more than G * kGemmBK products.
        float acc[kGemmBN];
#pragma unroll
        for (int j = 0; j < kGemmBN; ++j) acc[j] = 0.0f;
        bool got = true;
        int drained = 0;
        auto drain = [&](int gi) {
            const int buf = gi & 1;
            got = mbar_wait(&acc_full[buf], (gi >> 1) & 1, kFaultGemm) && got;
            __syncwarp();
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < kGemmBN; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_base + static_cast<uint32_t>(buf * kGemmBN + c0), r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[c0 + j] += __uint_as_float(r[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        };
        for (int kb = 0; kb < nk && got; ++kb) {
            const int s = kb % S, l = kb % NL;
            // lo = x - (x with its low 13 mantissa bits cleared), for both raw
            // tiles of the stage, at the same (swizzled) offsets in lo buffer l,
            // once the MMAs of block kb - NL have finished reading that buffer
            got = mbar_wait(&full[s], (kb / S) & 1, kFaultGemm) && got;
            if (kb >= NL)
                got = mbar_wait(&empty[(kb - NL) % S], ((kb - NL) / S) & 1, kFaultGemm) && got;
            if (got) {
                const float4* src = reinterpret_cast<const float4*>(smem + s * kPairBytes);
                float4* dst = reinterpret_cast<float4*>(lobuf + l * kPairBytes);
#pragma unroll
                for (int i0 = 0; i0 < 2 * kTileFloats / 4 / 128; i0 += 4) {
                    float4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) v[u] = src[et + 128 * (i0 + u)];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float4 w;
                        w.x = v[u].x - __uint_as_float(__float_as_uint(v[u].x) & 0xFFFFE000u);
                        w.y = v[u].y - __uint_as_float(__float_as_uint(v[u].y) & 0xFFFFE000u);
                        w.z = v[u].z - __uint_as_float(__float_as_uint(v[u].z) & 0xFFFFE000u);
                        w.w = v[u].w - __uint_as_float(__float_as_uint(v[u].w) & 0xFFFFE000u);
                        dst[et + 128 * (i0 + u)] = w;
                    }
                }
                fence_proxy_async_smem();   // the tensor core reads them through the async proxy
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&conv[l]);
            // read back the groups that are a full group behind the conversion
            while (got && drained < (kb + 1) / G - 1) drain(drained++);
        }
        while (got && drained < ngroups) drain(drained++);
        // The operand stages are idle once the last group is complete: each
        // warp turns its 32 x 32 sub-tiles around through a padded slice of
        // stage 0 so that global stores run along rows.
        float* tile = reinterpret_cast<float*>(smem) + q * (32 * 33);
#pragma unroll
        for (int c0 = 0; c0 < kGemmBN; c0 += 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j) tile[lane * 33 + j] = acc[c0 + j];
            __syncwarp();
            const int col = n0 + c0 + lane;
            const int rbase = m0 + 32 * q;
            const int rows = min(32, a.M - rbase);
            if (got && col < a.N && rows > 0) {
                if (a.ksplit > 1) {
                    float* P = a.part + static_cast<size_t>(blockIdx.z) * a.M * a.N;
#pragma unroll 8
                    for (int rr = 0; rr < 32; ++rr)
                        if (rr < rows) P[static_cast<size_t>(rbase + rr) * a.N + col] = tile[rr * 33 + lane];
                } else {
                    const float bv = a.bias ? a.bias[col] : 0.0f;
                    // residual rows fetched 8 at a time so their loads overlap
#pragma unroll
                    for (int r0 = 0; r0 < 32; r0 += 8) {
                        float res[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            res[u] = (a.R && r0 + u < rows)
                                         ? a.R[static_cast<size_t>(rbase + r0 + u) * a.ldr + col] : 0.0f;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (r0 + u < rows)
                                a.C[static_cast<size_t>(rbase + r0 + u) * a.ldc + col] =
                                    tile[(r0 + u) * 33 + lane] + bv + res[u];
                    }
                }
            }
            __syncwarp();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t read_clear_fault_gemm(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_ssm_fault, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_ssm_fault, &zero, sizeof(unsigned));
}

// C = sum_z part[z] (+ bias) (+ R): the split-K finish, fixed order.
__global__ void gemm_splitk_reduce_kernel(const GemmArgs a) {
    const size_t total = static_cast<size_t>(a.M) * a.N;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t m = i / a.N;
        const int n = static_cast<int>(i % a.N);
        float o = 0.0f;
        for (int z = 0; z < a.ksplit; ++z) o += a.part[static_cast<size_t>(z) * total + i];
        if (a.bias) o += a.bias[n];
        if (a.R) o += a.R[m * a.ldr + n];
        a.C[m * a.ldc + n] = o;
    }
}

cudaError_t launch_gemm_tf32x3(const GemmMaps& maps, const GemmArgs& a, cudaStream_t st) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    if (a.ksplit < 1 || (a.ksplit > 1 && !a.part)) return cudaErrorInvalidValue;
    const size_t smem = (kGemmStages + kGemmLoBufs) * kPairBytes +
                        (2 * kGemmStages + kGemmLoBufs + 4) * 8 + 16 + 1024;
    cudaError_t e = cudaFuncSetAttribute(gemm_tf32x3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid((a.N + kGemmBN - 1) / kGemmBN, (a.M + kGemmBM - 1) / kGemmBM, a.ksplit);
    gemm_tf32x3_kernel<<<grid, 192, smem, st>>>(maps, a);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.ksplit == 1) return e;
    const size_t total = static_cast<size_t>(a.M) * a.N;
    const unsigned blocks = static_cast<unsigned>(std::min<size_t>((total + 255) / 256, 152 * 8));
    gemm_splitk_reduce_kernel<<<blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- operand copies

__global__ void copy2d_kernel(const float* __restrict__ x, int64_t ldx, int rows, int cols,
                              float* __restrict__ out, int64_t ldo) {
    const int64_t total = static_cast<int64_t>(rows) * cols;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / cols, c = i % cols;
        out[r * ldo + c] = x[r * ldx + c];
    }
}

// Transpose through a 32 x 33 shared tile: out is (cols, rows).
__global__ void transpose_kernel(const float* __restrict__ x, int64_t ldx, int rows, int cols,
                                 float* __restrict__ out, int64_t ldo) {
    __shared__ float tile[32][33];
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
    for (int k = ty; k < 32; k += 8) {
        const int r = r0 + k, c = c0 + tx;
        tile[k][tx] = (r < rows && c < cols) ? x[static_cast<int64_t>(r) * ldx + c] : 0.0f;
    }
    __syncthreads();
    for (int k = ty; k < 32; k += 8) {
        const int c = c0 + k, r = r0 + tx;
        if (c < cols && r < rows) out[static_cast<int64_t>(c) * ldo + r] = tile[tx][k];
    }
}

cudaError_t launch_operand_copy(const float* x, int64_t ldx, int rows, int cols, int transpose,
                                float* out, int64_t ldo, cudaStream_t st) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    if (transpose) {
        dim3 grid((cols + 31) / 32, (rows + 31) / 32);
        transpose_kernel<<<grid, 256, 0, st>>>(x, ldx, rows, cols, out, ldo);
    } else {
        const int64_t total = static_cast<int64_t>(rows) * cols;
        const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((total + 255) / 256, 152 * 32));
        copy2d_kernel<<<blocks, 256, 0, st>>>(x, ldx, rows, cols, out, ldo);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- column sums

constexpr int kColsumRows = 512;   // rows per partial

__global__ void colsum_partial_kernel(const float* __restrict__ x, int64_t ldx, int rows, int cols,
                                      float* __restrict__ part) {
    __shared__ float red[8][33];
    const int c = blockIdx.x * 32 + (threadIdx.x & 31);
    const int g = threadIdx.x >> 5;   // 8 row groups
    const int r0 = blockIdx.y * kColsumRows;
    const int r1 = min(rows, r0 + kColsumRows);
    float s = 0.0f;
    if (c < cols)
        for (int r = r0 + g; r < r1; r += 8) s += x[static_cast<int64_t>(r) * ldx + c];
    red[g][threadIdx.x & 31] = s;
    __syncthreads();
    if (g == 0 && c < cols) {
        float t = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) t += red[k][threadIdx.x & 31];
        part[static_cast<int64_t>(blockIdx.y) * cols + c] = t;
    }
}

__global__ void colsum_final_kernel(const float* __restrict__ part, int nparts, int cols,
                                    float* __restrict__ out) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    float s = 0.0f;
    for (int p = 0; p < nparts; ++p) s += part[static_cast<int64_t>(p) * cols + c];
    out[c] = s;
}

size_t colsum_ws_floats(int rows, int cols) {
    return static_cast<size_t>((rows + kColsumRows - 1) / kColsumRows) * cols;
}

cudaError_t launch_colsum(const float* x, int64_t ldx, int rows, int cols, float* out, float* ws,
                          cudaStream_t st) {
    if (cols == 0) return cudaSuccess;
    const int nparts = (rows + kColsumRows - 1) / kColsumRows;
    if (nparts > 0) {
        dim3 grid((cols + 31) / 32, nparts);
        colsum_partial_kernel<<<grid, 256, 0, st>>>(x, ldx, rows, cols, ws);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    colsum_final_kernel<<<(cols + 255) / 256, 256, 0, st>>>(ws, nparts, cols, out);
    return cudaGetLastError();
}

}  // namespace ssm

// gemm.cu -- fp32-accurate tensor-core GEMM for the Mamba-1 block projections
// (cpu_ops.ts linearForward / linearBackward: Y = X W^T + b, dX = dY W,
// dW = dY^T X), plus operand copies (transposes) and deterministic column
// sums.
//
// sm_103a design: a persistent, warp-specialized kernel (one CTA per SM walks
// 128 x 128 tiles of C = A B^T) on tcgen05.mma (kind::tf32, cta_group::1,
// M = 128, N = 128, K = 8 per instruction) accumulating in tensor memory, as
// three TF32 products A_hi B_hi + A_hi B_lo + A_lo B_hi (about fp32 accuracy;
// hi = x with its low 13 mantissa bits cleared, lo = x - hi, exact).  A TMA
// producer streams raw 128 x 32 fp32 tiles of A and B (128-byte swizzle);
// converter warps write A's hi and lo parts into tensor memory (tcgen05.st,
// one row per thread; the MMAs read A from there) and B's lo part into a
// shared-memory tile at the raw tile's swizzled offsets, while the raw B tile
// itself serves as B_hi (the tensor core reads a tf32 operand from an fp32
// word and ignores its low 13 mantissa bits); one thread issues the MMAs; an
// epilogue warpgroup reads the accumulator back.  The tensor core's fp32
// accumulation drifts in one direction (its error grows linearly with K), so
// the accumulator is double-buffered in tensor memory and read back into
// fp32 registers every kGemmGroup K-blocks, and the tile is stored after its
// last group while the MMAs of the next tile run.  Every mbarrier wait is
// bounded; tensor memory is always released.
#include <algorithm>
#include <type_traits>

#include "gemm_args.cuh"
#include "ssm_common.cuh"

namespace ssm {

constexpr unsigned kFaultGemm = 8u;
constexpr uint32_t kOpTileBytes = kGemmBM * kGemmBK * 4;         // 16 KB (BM == BN)
constexpr uint32_t kPairBytes = 2 * kOpTileBytes;                // [A][B] of one K-block
// Tensor memory: two fp32 accumulators (columns [0, 2 BN)), then kGemmLoBufs
// A operand buffers of 2 BK columns each: [A_hi | A_lo] of one K-block.
constexpr uint32_t kAccCols = 2 * kGemmBN;
constexpr uint32_t kABufCols = 2 * kGemmBK;
constexpr uint32_t kTmemCols = 512;
static_assert(kAccCols + kGemmLoBufs * kABufCols <= kTmemCols, "tensor memory budget");
// Shared memory: kGemmStages raw stages [A raw][B raw] of 32 KB, then
// kGemmLoBufs B_lo tiles of 16 KB.
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
// The same with A read from tensor memory (128 lanes = rows, 8 columns = K).
__device__ __forceinline__ void umma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(kIdescTF32), "r"(acc)
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
// Sixteen consecutive 32-bit columns of this thread's tensor-memory lane (no
// memory clobber: it touches no memory that C++ code reads or writes).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
// A global store in the global state space (so that it is not ordered
// against later shared-memory loads as a generic store would be).
__device__ __forceinline__ void st_global_f32(float* p, float v) {
    asm volatile("st.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
// A global load in the global state space.  The epilogue issues a sub-tile's
// 32 residual loads back to back with these before adding any of them (as
// plain loads they were issued one after another, each waiting for the
// last: 30 us per tile).
__device__ __forceinline__ float ld_global_f32(const float* p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
// Register split between the warpgroups (see the kernel).
__device__ __forceinline__ void regs_shrink() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGemmRegsSmall)); }
__device__ __forceinline__ void regs_conv() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGemmRegsConv)); }
__device__ __forceinline__ void regs_grow() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGemmRegsEpi)); }
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One output tile of the persistent schedule: tile t of a GEMM has n-tile
// t % ntn, m-tile (t / ntn) % ntm and K slice t / (ntn ntm); its K-blocks are
// [kb0, kb0 + nk) of the full K range.
struct GemmTile {
    int m0, n0, z, kb0, nk;
};

// Warp roles (512 threads, persistent, one CTA per SM):
//   warp 0        TMA producer: raw fp32 A | B tiles into kGemmStages stages
//   warp 1        tensor-memory allocation; one thread issues the MMAs
//   warps 2-3     3/8 of each B lo tile into shared memory
//   warps 4-7     for even K-blocks: A hi | lo into tensor memory (warp w
//                 writes lanes 32 (w % 4) ..) and the rest of the B lo tile
//   warps 8-11    epilogue: every group's partial accumulator into fp32
//                 registers, then the tile's stores
//   warps 12-15   as warps 4-7, for odd K-blocks
// (one converter warp per K-block and quadrant could not keep up with the
// MMAs: its loads, conversion and tensor-memory stores form a chain longer
// than one K-block's MMAs).  The epilogue warpgroup holds a 128-float row of
// running sums per thread, so the other three warpgroups hand it registers
// (setmaxnreg): 128 x (kGemmRegsSmall + 2 x kGemmRegsConv + kGemmRegsEpi) must not exceed the
// 512 x (launch registers) the CTA starts with, which the launcher checks.
//
// RES: the launch adds a residual R (ksplit 1); its epilogue loads each
// sub-tile's residual one sub-tile ahead, so that the loads' latency overlaps
// the previous sub-tile's stores (GEMMs with a short K are bound by it).  The
// launches without a residual keep the plain epilogue.
template <bool RES>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_tf32x3_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    constexpr int S = kGemmStages;
    constexpr int NL = kGemmLoBufs;
    constexpr int G = kGemmGroup;
    static_assert(NL <= S, "a lo buffer is reused only after its stage's MMAs finished");
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* lobuf = smem + S * kPairBytes;                                 // [NL][B lo]
    float* ebuf = reinterpret_cast<float*>(lobuf + NL * kOpTileBytes);            // [4][32][33] epilogue
    uint64_t* full = reinterpret_cast<uint64_t*>(ebuf + 4 * 32 * 33);             // [S] raw tiles landed
    uint64_t* conv = full + S;           // [NL] A hi/lo and B lo written (one arrival per converter warp)
    uint64_t* empty = conv + NL;         // [S] the MMAs of that K-block are done (stage and its lo buffers free)
    uint64_t* acc_full = empty + S;      // [2] a partial accumulator is complete
    uint64_t* acc_empty = acc_full + 2;  // [2] the epilogue has read it back
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Persistent schedule: CTA i computes tiles i, i + gridDim.x, ...  Every
    // role walks the same sequence, and the barrier phases run on across
    // tiles (K-block counter j, accumulator-group counter gg).
    const int ntn = (a.N + kGemmBN - 1) / kGemmBN;
    const int ntm = (a.M + kGemmBM - 1) / kGemmBM;
    const int ntiles = ntn * ntm * a.ksplit;
    const int nk_all = (a.K + kGemmBK - 1) / kGemmBK;
    const int per = (nk_all + a.ksplit - 1) / a.ksplit;
    auto tile_of = [&](int t) {
        GemmTile x;
        const int r = t / ntn;
        x.n0 = (t % ntn) * kGemmBN;
        x.m0 = (r % ntm) * kGemmBM;
        x.z = r / ntm;
        x.kb0 = x.z * per;
        x.nk = max(0, min(per, nk_all - x.kb0));
        return x;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int l = 0; l < NL; ++l) mbar_init(&conv[l], 6);   // 2 B warps + 4 A warps of the K-block's parity
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

    // TMA producer (one thread): the raw fp32 tiles of A and B
    auto producer = [&]() {
        tma_prefetch_desc(&maps.a);
        tma_prefetch_desc(&maps.b);
        int j = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const GemmTile x = tile_of(t);
            for (int kb = 0; kb < x.nk; ++kb, ++j) {
                const int s = j % S;
                if (j >= S && !mbar_wait(&empty[s], ((j / S) - 1) & 1, kFaultGemm)) {
                    ok = false;
                    break;
                }
                unsigned char* st = smem + s * kPairBytes;
                mbar_arrive_expect_tx(&full[s], kPairBytes);
                const int kx = (x.kb0 + kb) * kGemmBK;
                tma_load_2d(st, &maps.a, &full[s], kx, x.m0);
                tma_load_2d(st + kOpTileBytes, &maps.b, &full[s], kx, x.n0);
            }
        }
        // copies still in flight land before the CTA may exit (bounded)
        for (int jj = max(0, j - S); jj < j; ++jj) mbar_wait(&full[jj % S], (jj / S) & 1, kFaultDrain);
    };

    // MMA issuer (one thread)
    auto mma_issuer = [&]() {
        int j = 0, gg = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const GemmTile x = tile_of(t);
            const int ng = (x.nk + G - 1) / G;
            for (int gi = 0; gi < ng && ok; ++gi, ++gg) {
                const int buf = gg & 1;
                // the epilogue must have read this buffer's previous group
                if (gg >= 2 && !mbar_wait(&acc_empty[buf], ((gg >> 1) - 1) & 1, kFaultGemm)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(buf * kGemmBN);
                const int kb1 = min(x.nk, (gi + 1) * G);
                for (int kb = gi * G; kb < kb1; ++kb, ++j) {
                    const int s = j % S, l = j % NL;
                    if (!mbar_wait(&conv[l], (j / NL) & 1, kFaultGemm)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + s * kPairBytes);
                    const uint32_t lt = smem_u32(lobuf + l * kOpTileBytes);
                    const uint32_t at = tmem + kAccCols + static_cast<uint32_t>(l) * kABufCols;
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 8; ++kk) {
                        const uint32_t off = kk * 32;   // 8 tf32 = 32 bytes along K
                        const uint32_t ahi = at + kk * 8, alo = at + kGemmBK + kk * 8;
                        const uint64_t bhi = umma_desc_sw128(st + kOpTileBytes + off);
                        const uint64_t blo = umma_desc_sw128(lt + off);
                        umma_tf32_ta(d, ahi, bhi, (kb != gi * G || kk != 0) ? 1u : 0u);
                        umma_tf32_ta(d, ahi, blo, 1u);
                        umma_tf32_ta(d, alo, bhi, 1u);
                    }
                    umma_commit(&empty[s]);   // stage s and lo buffers l are free once these MMAs finish
                }
                if (!ok) break;
                umma_commit(&acc_full[buf]);  // this group's partial sum is complete
            }
        }
        // every MMA has finished before tensor memory is released
        if (j > 0) mbar_wait(&empty[(j - 1) % S], ((j - 1) / S) & 1, kFaultDrain);
    };

    // K-block j's lo parts go to lo buffer j % NL once the MMAs of block
    // j - NL have finished reading it: A hi | lo into tensor memory by the
    // A warpgroup of j's parity (warps 4-7 even j, 12-15 odd j), B lo into
    // shared memory at the raw tile's (swizzled) offsets, its first 3/8 by
    // warps 2-3 (6 float4 per thread), the rest by that A warpgroup (5 float4
    // per thread).
    auto converters = [&](bool is_a, int parity) {
        const int q = warp & 3;                        // A: TMEM lane quadrant
        const int ar = 32 * q + lane;                  // A: this thread's row (= its TMEM lane)
        const uint32_t a_lane = tmem + (static_cast<uint32_t>(32 * q) << 16) + kAccCols;
        constexpr int kF4 = kTileFloats / 4;           // float4 per B tile
        constexpr int kBwarpsF4 = 3 * kF4 / 8;         // B lo float4 of warps 2-3
        const int bf0 = is_a ? kBwarpsF4 + ar : threadIdx.x - 64;
        const int bstep = is_a ? 128 : 64;
        bool got = true;
        int j = 0;
        for (int t = blockIdx.x; t < ntiles && got; t += gridDim.x) {
            const int nk = tile_of(t).nk;
            for (int kb = 0; kb < nk && got; ++kb, ++j) {
                if (is_a && (j & 1) != parity) continue;
                const int s = j % S, l = j % NL;
                got = mbar_wait(&full[s], (j / S) & 1, kFaultGemm) && got;
                if (j >= NL)
                    got = mbar_wait(&empty[(j - NL) % S], ((j - NL) / S) & 1, kFaultGemm) && got;
                got = __all_sync(0xffffffffu, got);
                if (got) {
                    const float4* src =
                        reinterpret_cast<const float4*>(smem + s * kPairBytes + kOpTileBytes);
                    float4* dst = reinterpret_cast<float4*>(lobuf + l * kOpTileBytes);
                    auto b_lo = [&](auto nv) {
                        constexpr int NV = decltype(nv)::value;
                        float4 v[NV];
#pragma unroll
                        for (int u = 0; u < NV; ++u) v[u] = src[bf0 + bstep * u];
#pragma unroll
                        for (int u = 0; u < NV; ++u) {
                            float4 w;
                            w.x = v[u].x - __uint_as_float(__float_as_uint(v[u].x) & 0xFFFFE000u);
                            w.y = v[u].y - __uint_as_float(__float_as_uint(v[u].y) & 0xFFFFE000u);
                            w.z = v[u].z - __uint_as_float(__float_as_uint(v[u].z) & 0xFFFFE000u);
                            w.w = v[u].w - __uint_as_float(__float_as_uint(v[u].w) & 0xFFFFE000u);
                            dst[bf0 + bstep * u] = w;
                        }
                        fence_proxy_async_smem();   // the tensor core reads B lo through the async proxy
                    };
                    if (!is_a) {
                        b_lo(std::integral_constant<int, kBwarpsF4 / 64>{});
                    } else {
                        // row ar: hi | lo into columns of tensor-memory buffer l
                        tc_fence_after();
                        const unsigned char* arow = smem + s * kPairBytes + ar * 128;
                        const uint32_t adst = a_lane + static_cast<uint32_t>(l) * kABufCols;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // 16-byte chunks 4h .. 4h + 3 of the row (128-byte
                            // swizzle: chunk index xor row mod 8)
                            float4 v4[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                v4[c] = *reinterpret_cast<const float4*>(arow + (((4 * h + c) ^ (ar & 7)) << 4));
                            uint32_t hi[16], lo[16];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const float xv[4] = {v4[c].x, v4[c].y, v4[c].z, v4[c].w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    hi[4 * c + e] = __float_as_uint(xv[e]) & 0xFFFFE000u;
                                    lo[4 * c + e] = __float_as_uint(xv[e] - __uint_as_float(hi[4 * c + e]));
                                }
                            }
                            tmem_st16(adst + 16 * h, hi);
                            tmem_st16(adst + kGemmBK + 16 * h, lo);
                        }
                        b_lo(std::integral_constant<int, (kF4 - kBwarpsF4) / 128>{});
                        tmem_wait_st();
                        tc_fence_before();
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&conv[l]);
            }
        }
    };

    // Each group's partial sum (at most G K-blocks, accumulated by the tensor
    // core) is added into fp32 registers, so the tensor core's own
    // accumulation never spans more than G * kGemmBK products; after a tile's
    // last group its rows are stored.
    auto epilogue = [&]() {
        const int q = warp & 3;                        // TMEM lane quadrant
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
        float acc[kGemmBN];
#pragma unroll
        for (int c = 0; c < kGemmBN; ++c) acc[c] = 0.0f;
        bool got = true;
        float* tile = ebuf + q * (32 * 33);
        int gg = 0;
        for (int t = blockIdx.x; t < ntiles && got; t += gridDim.x) {
            const GemmTile x = tile_of(t);
            const int ng = (x.nk + G - 1) / G;
            // RES: the residual rows of the sub-tile stored next (column x.n0 +
            // c0 + lane, rows x.m0 + 32 q ..), loaded one sub-tile ahead
            const int rb = x.m0 + 32 * q;
            const int nrows = min(32, a.M - rb);
            float resn[RES ? 32 : 1];
            auto load_res = [&](int c0) {
                if constexpr (RES) {
                    const int col = x.n0 + c0 + lane;
                    const bool ld = col < a.N && nrows > 0;
                    const float* Rp = ld ? a.R + static_cast<size_t>(rb) * a.ldr + col : nullptr;
#pragma unroll
                    for (int rr = 0; rr < 32; ++rr)
                        resn[rr] = ld ? ld_global_f32(Rp + static_cast<size_t>(min(rr, nrows - 1)) * a.ldr) : 0.0f;
                }
            };
            for (int gi = 0; gi < ng && got; ++gi, ++gg) {
                const int buf = gg & 1;
                got = mbar_wait(&acc_full[buf], (gg >> 1) & 1, kFaultGemm) && got;
                got = __all_sync(0xffffffffu, got);
                if (got) {
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < kGemmBN; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(lane_base + static_cast<uint32_t>(buf * kGemmBN + c0), r);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) acc[c0 + c] += __uint_as_float(r[c]);
                    }
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
            }
            if (!got) break;
            load_res(0);
            // each warp turns its 32 x 32 sub-tiles around through its slice of
            // ebuf so that global stores run along rows
#pragma unroll
            for (int c0 = 0; c0 < kGemmBN; c0 += 32) {
#pragma unroll
                for (int c = 0; c < 32; ++c) tile[lane * 33 + c] = acc[c0 + c];
                __syncwarp();
                // the column of the sub-tile this lane stores, read whole
                // before any global store is issued
                float v[32];
#pragma unroll
                for (int rr = 0; rr < 32; ++rr) v[rr] = tile[rr * 33 + lane];
                __syncwarp();
                if constexpr (RES) {
#pragma unroll
                    for (int rr = 0; rr < 32; ++rr) v[rr] += resn[rr];
                    if (c0 + 32 < kGemmBN) load_res(c0 + 32);
                }
                const int col = x.n0 + c0 + lane;
                const int rbase = x.m0 + 32 * q;
                const int rows = min(32, a.M - rbase);
                if (col < a.N && rows > 0) {
                    if (a.ksplit > 1) {
                        float* P = a.part + static_cast<size_t>(x.z) * a.M * a.N +
                                   static_cast<size_t>(rbase) * a.N + col;
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr)
                            if (rr < rows) st_global_f32(P + static_cast<size_t>(rr) * a.N, v[rr]);
                    } else {
                        const float bv = a.bias ? a.bias[col] : 0.0f;
                        if (!RES && a.R) {
                            const float* Rp = a.R + static_cast<size_t>(rbase) * a.ldr + col;
                            float res[32];
#pragma unroll
                            for (int rr = 0; rr < 32; ++rr)
                                res[rr] = ld_global_f32(Rp + static_cast<size_t>(min(rr, rows - 1)) * a.ldr);
#pragma unroll
                            for (int rr = 0; rr < 32; ++rr) v[rr] += res[rr];
                        }
                        float* Cp = a.C + static_cast<size_t>(rbase) * a.ldc + col;
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr)
                            if (rr < rows) st_global_f32(Cp + static_cast<size_t>(rr) * a.ldc, v[rr] + bv);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < kGemmBN; ++c) acc[c] = 0.0f;
        }
    };

    // Roles by warpgroup; each warpgroup resizes its registers at one place.
    if (warp < 4) {
        regs_shrink();
        if (warp == 0) {
            if (lane == 0) producer();
        } else if (warp == 1) {
            if (lane == 0) mma_issuer();
        } else {
            converters(false, 0);
        }
    } else if (warp < 8) {
        regs_conv();
        converters(true, 0);
    } else if (warp < 12) {
        regs_grow();
        epilogue();
    } else {
        regs_conv();
        converters(true, 1);
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
    const size_t smem = kGemmStages * kPairBytes + kGemmLoBufs * kOpTileBytes + 4 * 32 * 33 * 4 +
                        (2 * kGemmStages + kGemmLoBufs + 4) * 8 + 16 + 1024;
    const bool res = a.R && a.ksplit == 1;
    auto kern = res ? gemm_tf32x3_kernel<true> : gemm_tf32x3_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // The warpgroups' register split must fit in what the CTA is launched
    // with (otherwise the epilogue's setmaxnreg.inc could never be granted).
    static int launch_regs[2] = {-1, -1};
    if (launch_regs[res] < 0) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        launch_regs[res] = fa.numRegs;
    }
    if (kGemmThreads * launch_regs[res] < 128 * (kGemmRegsSmall + 2 * kGemmRegsConv + kGemmRegsEpi))
        return cudaErrorInvalidConfiguration;
    // persistent: one CTA per SM (shared memory allows no more), each walking
    // its share of the output tiles
    const long long ntiles = static_cast<long long>((a.N + kGemmBN - 1) / kGemmBN) *
                             ((a.M + kGemmBM - 1) / kGemmBM) * a.ksplit;
    int dev = 0, nsm = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(std::min<long long>(ntiles, std::max(nsm, 1)));
    kern<<<grid, kGemmThreads, smem, st>>>(maps, a);
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

// Transpose of 64 x 64 tiles with 16-byte loads and stores (x, out 16-byte
// aligned, ldx and ldo multiples of 4); tiles cut by the matrix edge take
// single-element accesses.  256 threads, 4 float4 each way per thread.  With
// csum non-null the tile's column sums (over its 64 rows, in a fixed order)
// are also written to csum[blockIdx.y][column]: the column sums of x come out
// of the same pass over it.
__global__ void __launch_bounds__(256) transpose64_kernel(const float* __restrict__ x, int64_t ldx, int rows,
                                                          int cols, float* __restrict__ out, int64_t ldo,
                                                          float* __restrict__ csum) {
    __shared__ float tile[64][65];
    __shared__ float qsum[4][64];
    const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
    const int t = threadIdx.x;
    const bool full = r0 + 64 <= rows && c0 + 64 <= cols;
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = t + 256 * i, rr = idx >> 4, cc = (idx & 15) * 4;
        const float* src = x + static_cast<int64_t>(r0 + rr) * ldx + c0 + cc;
        if (full) {
            v[i] = *reinterpret_cast<const float4*>(src);
        } else {
            float e[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) e[k] = (r0 + rr < rows && c0 + cc + k < cols) ? src[k] : 0.0f;
            v[i] = make_float4(e[0], e[1], e[2], e[3]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = t + 256 * i, rr = idx >> 4, cc = (idx & 15) * 4;
        tile[rr][cc] = v[i].x;
        tile[rr][cc + 1] = v[i].y;
        tile[rr][cc + 2] = v[i].z;
        tile[rr][cc + 3] = v[i].w;
    }
    __syncthreads();
    if (csum) {
        // column t % 64 over rows 16 (t / 64) .. + 15 (zeros past the edge)
        const int c = t & 63, q = t >> 6;
        float sacc = 0.0f;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) sacc += tile[16 * q + rr][c];
        qsum[q][c] = sacc;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = t + 256 * i, cr = idx >> 4, rc = (idx & 15) * 4;
        const float4 w = make_float4(tile[rc][cr], tile[rc + 1][cr], tile[rc + 2][cr], tile[rc + 3][cr]);
        float* dst = out + static_cast<int64_t>(c0 + cr) * ldo + r0 + rc;
        if (full) {
            *reinterpret_cast<float4*>(dst) = w;
        } else if (c0 + cr < cols) {
            const float e[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (r0 + rc + k < rows) dst[k] = e[k];
        }
    }
    if (csum) {
        __syncthreads();
        if (t < 64 && c0 + t < cols)
            csum[static_cast<int64_t>(blockIdx.y) * cols + c0 + t] =
                ((qsum[0][t] + qsum[1][t]) + qsum[2][t]) + qsum[3][t];
    }
}

cudaError_t launch_operand_copy(const float* x, int64_t ldx, int rows, int cols, int transpose,
                                float* out, int64_t ldo, cudaStream_t st) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0 &&
                     ldx % 4 == 0 && ldo % 4 == 0;
    if (transpose && vec) {
        dim3 grid((cols + 63) / 64, (rows + 63) / 64);
        transpose64_kernel<<<grid, 256, 0, st>>>(x, ldx, rows, cols, out, ldo, nullptr);
    } else if (transpose) {
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

// Sum of nparts partial rows of cols columns: a CTA per 32 columns, its 8
// warps each adding every 8th partial (lane = column), then the 8 warp sums
// in a fixed order.
__global__ void __launch_bounds__(256) colsum_final8_kernel(const float* __restrict__ part, int nparts,
                                                            int cols, float* __restrict__ out) {
    __shared__ float red[8][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float s = 0.0f;
    if (c < cols)
        for (int p = w; p < nparts; p += 8) s += part[static_cast<int64_t>(p) * cols + c];
    red[w][lane] = s;
    __syncthreads();
    if (w == 0 && c < cols) {
        float t = red[0][lane];
#pragma unroll
        for (int k = 1; k < 8; ++k) t += red[k][lane];
        out[c] = t;
    }
}

// Partials of the 64-row tiles of the transposing copy, or of kColsumRows-row
// slabs: the larger count.
size_t colsum_ws_floats(int rows, int cols) {
    return static_cast<size_t>((rows + 63) / 64) * cols;
}

cudaError_t launch_operand_copy_t_colsum(const float* x, int64_t ldx, int rows, int cols, float* out,
                                         int64_t ldo, float* colsum, float* ws, cudaStream_t st) {
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0 &&
                     ldx % 4 == 0 && ldo % 4 == 0;
    if (!colsum || !vec) {
        cudaError_t e = launch_operand_copy(x, ldx, rows, cols, 1, out, ldo, st);
        if (e != cudaSuccess || !colsum) return e;
        return launch_colsum(x, ldx, rows, cols, colsum, ws, st);
    }
    if (cols == 0) return cudaSuccess;
    const int nparts = (rows + 63) / 64;
    if (nparts > 0) {
        dim3 grid((cols + 63) / 64, nparts);
        transpose64_kernel<<<grid, 256, 0, st>>>(x, ldx, rows, cols, out, ldo, ws);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    colsum_final8_kernel<<<(cols + 31) / 32, 256, 0, st>>>(ws, nparts, cols, colsum);
    return cudaGetLastError();
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

// scan_fwd.cu -- selective-scan forward for sm_103a.
//
// Computes mamba1_cpu.ts mamba1CpuForward steps 8-9 (page "@seanhogg/builderforce-
// memory-engine 2026.7.12 -> 2026.9.27"):
//   delta = softplus(delta_raw); A = -exp(clamp(A_log, -10, 5));
//   h_t = exp(delta_t A) h_{t-1} + beta_t u_t;  y_t = C_t . h_t + D u_t;
//   out_t = y_t * silu(z_t)
// with beta = delta*B (Euler) or expm1(delta A)/A * B (ZOH).
//
// Design (GB300): one thread owns one (batch row, channel) chain and keeps all
// dstate states of it in registers for the whole sequence, so every element
// costs one ex2 and four fp32 ops (two packed f32x2 instructions per state
// pair) and nothing crosses threads.  A warp-sized CTA streams u / delta_raw /
// z tiles of kFwdTile steps x 32 channels and the B/C tiles of the same steps
// (shared by the 32 channels) with TMA, 4 tiles in flight.  Every kChunk
// steps the state is written to the context buffer for the backward.
#include "scan_args.cuh"
#include "ssm_common.cuh"

namespace ssm {

// One step of the recurrence for the NL states this lane owns:
// h = exp(dt A) h + beta u; returns sum_n C_n h_n over those states.
// Bt/Ct point at the lane's first state in the fp32 B|C tile row.
// bs = dt*u (Euler) or u (ZOH).
template <int NL, int DISC>
__device__ __forceinline__ float fwd_step(float2 (&h)[NL / 2], const float2 (&A2)[NL / 2],
                                          const float2 (&Anat)[NL / 2], const float2 (&invA)[NL / 2],
                                          const float* Bt, const float* Ct, float dt, float bs) {
    const float2 dt2 = f2(dt);
    const float2 bs2 = f2(bs);
    float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
    for (int q4 = 0; q4 < NL / 4; ++q4) {
        const float4 B4 = *reinterpret_cast<const float4*>(Bt + 4 * q4);
        const float4 C4 = *reinterpret_cast<const float4*>(Ct + 4 * q4);
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            const int q = 2 * q4 + hq;
            const float2 Bq = hq ? make_float2(B4.z, B4.w) : make_float2(B4.x, B4.y);
            const float2 Cq = hq ? make_float2(C4.z, C4.w) : make_float2(C4.x, C4.y);
            const float2 x = mul2(dt2, A2[q]);
            const float2 av = make_float2(ex2(x.x), ex2(x.y));
            float2 bu;
            if (DISC == 0) {
                bu = mul2(bs2, Bq);                  // delta * u * B
            } else {
                // beta/B = expm1(delta A)/A = delta * phi1(delta A), stably
                const float2 xn = mul2(dt2, Anat[q]);
                const float c0f = fabsf(xn.x) < 0.5f ? dt * phi1_series(xn.x) : (av.x - 1.0f) * invA[q].x;
                const float c1f = fabsf(xn.y) < 0.5f ? dt * phi1_series(xn.y) : (av.y - 1.0f) * invA[q].y;
                bu = mul2(mul2(make_float2(c0f, c1f), bs2), Bq);
            }
            h[q] = fma2(av, h[q], bu);
            acc[hq] = fma2(Cq, h[q], acc[hq]);
        }
    }
    const float2 s = add2(acc[0], acc[1]);
    return s.x + s.y;
}

// fp32 B and C of one tile, [TS][NT] each (states past dstate and steps past
// seqlen read 0).  fp32 TMA tiles are used in place; bf16 TMA tiles are
// widened into bcs 8 values per lane; B/C that are not TMA-aligned are read
// straight from global memory into bcs.  Returns the B pointer (C follows
// TS*NT floats later).
template <typename T, int NT, int TS>
__device__ __forceinline__ const float* fwd_stage_bc(float* bcs, const T* Bs, bool from_tma,
                                                     const T* Bp, const T* Cp, int64_t ldB,
                                                     int64_t ldC, size_t row0, int k, int L, int N,
                                                     int lane) {
    constexpr int BCT = TS * NT;
    if (from_tma && sizeof(T) == 4) return reinterpret_cast<const float*>(Bs);
    if (from_tma) {
        for (int g8 = lane; g8 < 2 * BCT / 8; g8 += 32) {
            const uint4 v = *reinterpret_cast<const uint4*>(Bs + 8 * g8);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            float f[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                f[2 * q] = __uint_as_float(w[q] << 16);
                f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
            }
            *reinterpret_cast<float4*>(bcs + 8 * g8) = make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4*>(bcs + 8 * g8 + 4) = make_float4(f[4], f[5], f[6], f[7]);
        }
        return bcs;
    }
    for (int e = lane; e < 2 * BCT; e += 32) {
        const int isC = e >= BCT, j = (e % BCT) / NT, n = e % NT, t = k * TS + j;
        float v = 0.0f;
        if (t < L && n < N) {
            const size_t r = row0 + t;
            v = isC ? Act<T>::load(Cp + r * ldC + n) : Act<T>::load(Bp + r * ldB + n);
        }
        bcs[e] = v;
    }
    return bcs;
}

// Segment pass of the time-parallel forward: for segment g of batch row b,
// run the recurrence from h = 0 and keep only the end state and the sum of
// delta over the segment.  Since exp(delta_t A) multiplies across steps into
// exp(A sum_t delta_t), the true state entering segment g+1 is
//   h_start(g+1) = exp(A sum_g delta) h_start(g) + h_end_from_zero(g),
// evaluated by scan_fwd_combine_kernel (segments in separate CTAs) or inside
// the CTA (segments as its warps).  One warp; smem holds the stages and the
// barriers of the pass.  Returns false if a bounded wait gave up.
template <typename T, int NT, int DISC>
__device__ __forceinline__ bool fwd_segsum_run(const FwdMaps& maps, const ScanFwdArgs& a, unsigned char* smem,
                                               int c0, int b, int g, int lane, float2 (&h)[NT / 2],
                                               float& dsum) {
    constexpr int CW = kFwdChannels;
    constexpr int TS = kFwdTile;
    constexpr int S = kFwdStages;
    constexpr int NQ = NT / 2;
    constexpr int TILE = TS * CW;
    constexpr int BCT = TS * NT;
    constexpr int STAGE = 2 * TILE + BCT;               // u, delta_raw, B
    constexpr uint32_t kActBytes = 2 * TILE * sizeof(T);
    constexpr uint32_t kBBytes = BCT * sizeof(T);
    static_assert((STAGE * sizeof(T)) % 128 == 0, "stages stay 128-byte aligned");

    T* tiles = reinterpret_cast<T*>(smem);                                   // [S][STAGE]
    float* bsm = reinterpret_cast<float*>(smem + S * STAGE * sizeof(T));    // [TS][NT] fp32 B
    uint64_t* full = reinterpret_cast<uint64_t*>(bsm + BCT);                 // [S]

    const int d = c0 + lane;
    const bool active = d < a.dinner;
    const int L = a.seqlen, N = a.dstate;
    const size_t row0 = static_cast<size_t>(b) * L;
    const bool bc_tma = a.bc_tma != 0;
    const int kb = g * a.seg_tiles, ke = kb + a.seg_tiles;   // a full segment (never the last)

    float2 A2[NQ], Anat[NQ], invA[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        float v[2], w[2], r[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = 2 * q + e;
            const bool ok = active && n < N;
            const float A = ok ? a_from_alog(a.A_log[static_cast<size_t>(d) * N + n]) : -1.0f;
            v[e] = ok ? A * kLog2e : 0.0f;
            w[e] = A;
            r[e] = 1.0f / A;
        }
        A2[q] = make_float2(v[0], v[1]);
        Anat[q] = make_float2(w[0], w[1]);
        invA[q] = make_float2(r[0], r[1]);
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) h[q] = make_float2(0.0f, 0.0f);
    dsum = 0.0f;

    const T* Bp = static_cast<const T*>(a.B);
    auto issue = [&](int k) {
        const int s = (k - kb) % S;
        T* dst = tiles + s * STAGE;
        mbar_arrive_expect_tx(&full[s], kActBytes + (bc_tma ? kBBytes : 0u));
        tma_load_3d(dst, &maps.u, &full[s], c0, k * TS, b);
        tma_load_3d(dst + TILE, &maps.dr, &full[s], c0, k * TS, b);
        if (bc_tma) tma_load_3d(dst + 2 * TILE, &maps.B, &full[s], 0, k * TS, b);
    };
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0)
        for (int k = kb; k < kb + S && k < ke; ++k) issue(k);

    int k = kb;
    for (; k < ke; ++k) {
        const int s = (k - kb) % S;
        bool ok = mbar_wait(&full[s], ((k - kb) / S) & 1, kFaultFwdWait);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const T* tu = tiles + s * STAGE;
        const T* tr = tu + TILE;
        const T* tb = tu + 2 * TILE;
        // fp32 B of this tile ([TS][NT]; past dstate 0)
        const float* Bf;
        if (bc_tma && sizeof(T) == 4) {
            Bf = reinterpret_cast<const float*>(tb);
        } else {
            for (int e = lane; e < BCT; e += 32) {
                float v;
                if (bc_tma) {
                    v = Act<T>::to_f(tb[e]);
                } else {
                    const int j = e / NT, n = e % NT;
                    v = n < N ? Act<T>::load(Bp + (row0 + static_cast<size_t>(k) * TS + j) * a.ld_B + n)
                              : 0.0f;
                }
                bsm[e] = v;
            }
            Bf = bsm;
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < TS; ++j) {
            const float uv = Act<T>::to_f(tu[j * CW + lane]);
            const float xr = Act<T>::to_f(tr[j * CW + lane]);
            float e;
            const float dt = softplus_e(xr, e);
            dsum += dt;
            const float bs = DISC == 0 ? dt * uv : uv;
            const float2 dt2 = f2(dt), bs2 = f2(bs);
#pragma unroll
            for (int q4 = 0; q4 < NT / 4; ++q4) {
                const float4 B4 = *reinterpret_cast<const float4*>(Bf + j * NT + 4 * q4);
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    const int q = 2 * q4 + hq;
                    const float2 Bq = hq ? make_float2(B4.z, B4.w) : make_float2(B4.x, B4.y);
                    const float2 x = mul2(dt2, A2[q]);
                    const float2 av = make_float2(ex2(x.x), ex2(x.y));
                    float2 bu;
                    if (DISC == 0) {
                        bu = mul2(bs2, Bq);
                    } else {
                        const float2 xn = mul2(dt2, Anat[q]);
                        const float c0f = fabsf(xn.x) < 0.5f ? dt * phi1_series(xn.x) : (av.x - 1.0f) * invA[q].x;
                        const float c1f = fabsf(xn.y) < 0.5f ? dt * phi1_series(xn.y) : (av.y - 1.0f) * invA[q].y;
                        bu = mul2(mul2(make_float2(c0f, c1f), bs2), Bq);
                    }
                    h[q] = fma2(av, h[q], bu);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && k + S < ke) issue(k + S);
    }
    if (k < ke && lane == 0) {
        for (int kk = k; kk < ke && kk < k + S; ++kk)
            mbar_wait(&full[(kk - kb) % S], ((kk - kb) / S) & 1, kFaultDrain);
    }
    return k == ke;
}

// Shared memory of fwd_segsum_run: stages of u, delta_raw, B, the fp32 B tile
// and the barriers.
template <typename T, int NT>
constexpr size_t fwd_segsum_smem_bytes() {
    return kFwdStages * (2 * kFwdTile * kFwdChannels + kFwdTile * NT) * sizeof(T) + kFwdTile * NT * sizeof(float) +
           kFwdStages * sizeof(uint64_t);
}

template <typename T, int NT, int DISC>
__global__ void __launch_bounds__(32, 1)
scan_fwd_segsum_kernel(const __grid_constant__ FwdMaps maps, const ScanFwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int NQ = NT / 2;
    const int lane = threadIdx.x;
    const int c0 = blockIdx.x * kFwdChannels, b = blockIdx.y, g = blockIdx.z;
    const int d = c0 + lane;
    float2 h[NQ];
    float dsum;
    const bool done = fwd_segsum_run<T, NT, DISC>(maps, a, smem, c0, b, g, lane, h, dsum);
    if (d < a.dinner && done) {
        float* hp = a.seg_h + (static_cast<size_t>(b) * a.nseg + g) * NT * a.dinner + d;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            hp[static_cast<size_t>(2 * q) * a.dinner] = h[q].x;
            hp[static_cast<size_t>(2 * q + 1) * a.dinner] = h[q].y;
        }
        a.seg_ds[(static_cast<size_t>(b) * a.nseg + g) * a.dinner + d] = dsum;
    }
}

// Lane layout: a warp-sized CTA owns 32 channels of one batch row, one
// channel per lane with all NT states of it in registers, so nothing per step
// is computed twice and no value crosses lanes.
//
// CHUNKED: the a.nseg time segments of one 32-channel tile are the warps of
// one CTA (the sequence split into chunks scanned in parallel).  Each warp but
// the last first runs its segment from h = 0 (fwd_segsum_run) and leaves the
// end state and the sum of delta in shared memory; after a CTA barrier each
// warp combines the segments before it into its start state,
//   h_start(g+1) = exp(A sum_g delta) h_start(g) + h_end_from_zero(g),
// then scans its segment as below.  Each warp has its own shared-memory
// region of fwd_warp_smem_bytes.
template <typename T, int NT, int DISC, bool GATE>
constexpr size_t fwd_warp_smem_bytes() {
    constexpr int NTEN = GATE ? 3 : 2;
    constexpr int TILE = kFwdTile * kFwdChannels;
    constexpr int STAGE = NTEN * TILE + 2 * kFwdTile * NT;
    constexpr size_t bytes = kFwdStages * STAGE * sizeof(T) + 2 * kFwdTile * NT * sizeof(float) +
                             2 * (kFwdTile / kChunk) * NT * kFwdChannels * sizeof(float) +
                             2 * 2 * TILE * sizeof(T) + kFwdStages * sizeof(uint64_t);
    return (bytes + 127) / 128 * 128;
}
template <int NT>
constexpr size_t fwd_chunk_xchg_bytes(int nseg) {
    return static_cast<size_t>(nseg) * (NT + 1) * kFwdChannels * sizeof(float);
}

template <typename T, int NT, int DISC, bool GATE, bool CHUNKED>
__global__ void __launch_bounds__(CHUNKED ? 32 * kFwdChunkWarps : 32, 1)
scan_fwd_kernel(const __grid_constant__ FwdMaps maps, const ScanFwdArgs a) {
    constexpr int CW = kFwdChannels;                    // channels per CTA (32)
    constexpr int TS = kFwdTile;
    constexpr int S = kFwdStages;
    constexpr int NTEN = GATE ? 3 : 2;
    constexpr int NQ = NT / 2;                          // state pairs per lane
    constexpr int TILE = TS * CW;                       // elements per activation tile
    constexpr int BCT = TS * NT;                        // elements per B or C tile
    constexpr uint32_t kActBytes = NTEN * TILE * sizeof(T);
    constexpr uint32_t kBCBytes = 2 * BCT * sizeof(T);
    constexpr int STAGE = NTEN * TILE + 2 * BCT;        // elements per stage
    static_assert(TS % kChunk == 0, "tiles hold whole checkpoint chunks");
    static_assert((STAGE * sizeof(T)) % 128 == 0, "stages stay 128-byte aligned");

    constexpr int NCK = TS / kChunk;                    // chunk boundaries per tile
    extern __shared__ __align__(128) unsigned char smem_all[];
    const int wid = CHUNKED ? static_cast<int>(threadIdx.x >> 5) : 0;
    unsigned char* smem = smem_all + wid * fwd_warp_smem_bytes<T, NT, DISC, GATE>();
    T* tiles = reinterpret_cast<T*>(smem);                                   // [S][STAGE]
    float* bcs = reinterpret_cast<float*>(smem + S * STAGE * sizeof(T));    // [TS][NT] B | C
    float* ckst = bcs + 2 * BCT;                                             // [2][NCK][NT][CW]
    T* ost = reinterpret_cast<T*>(ckst + 2 * NCK * NT * CW);                // [2][2][TS][CW] out | y
    uint64_t* full = reinterpret_cast<uint64_t*>(ost + 2 * 2 * TILE);        // [S]

    const int lane = threadIdx.x & 31;
    const int c0 = blockIdx.x * CW;
    const int b = blockIdx.y;
    const int d = c0 + lane;
    const bool active = d < a.dinner;
    const int L = a.seqlen, N = a.dstate;
    const int ntiles = (L + TS - 1) / TS;
    const size_t row0 = static_cast<size_t>(b) * L;
    const bool bc_tma = a.bc_tma != 0;

    // Per-(channel, state) constants: A*log2(e) as the ex2 argument scale (0 on
    // padding states and inactive lanes, where B = C = 0 or u = 0 keeps h at 0).
    float2 A2[NQ], Anat[NQ], invA[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        float v[2], w[2], r[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = 2 * q + e;
            const bool ok = active && n < N;
            const float A = ok ? a_from_alog(a.A_log[static_cast<size_t>(d) * N + n]) : -1.0f;
            v[e] = ok ? A * kLog2e : 0.0f;
            w[e] = A;
            r[e] = 1.0f / A;
        }
        A2[q] = make_float2(v[0], v[1]);
        Anat[q] = make_float2(w[0], w[1]);
        invA[q] = make_float2(r[0], r[1]);
    }
    const float Dd = (active && a.D) ? a.D[d] : 0.0f;
    // This CTA's time segment: tiles [kb, ke).  A segment after the first starts
    // from the state the segment pass left in h0 (exact: see the combine).
    const int g = CHUNKED ? wid : static_cast<int>(blockIdx.z);
    const int kb = g * a.seg_tiles;
    const int ke = min(ntiles, kb + a.seg_tiles);
    float2 h[NQ];
    if constexpr (CHUNKED) {
        // segments before the last: end state from h = 0 and the sum of delta,
        // to shared memory ([nseg][NT][CW] states, then [nseg][CW] sums)
        float* xh = reinterpret_cast<float*>(smem_all + blockDim.x / 32 * fwd_warp_smem_bytes<T, NT, DISC, GATE>());
        float* xd = xh + static_cast<size_t>(a.nseg) * NT * CW;
        if (g + 1 < a.nseg) {
            float dsum;
            fwd_segsum_run<T, NT, DISC>(maps, a, smem, c0, b, g, lane, h, dsum);
            if (lane == 0)
                for (int s2 = 0; s2 < S; ++s2)
                    mbar_inval(reinterpret_cast<uint64_t*>(smem + fwd_segsum_smem_bytes<T, NT>() -
                                                           S * sizeof(uint64_t)) + s2);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                xh[(g * NT + 2 * q) * CW + lane] = h[q].x;
                xh[(g * NT + 2 * q + 1) * CW + lane] = h[q].y;
            }
            xd[g * CW + lane] = dsum;
        }
        fence_proxy_async_smem();   // the stages are TMA destinations again below
        __syncthreads();
        // start state: the caller's initial state (or 0), then the segments before g
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            h[q] = make_float2(0.0f, 0.0f);
            if (active && a.h_init) {
                const float* hp = a.h_init + (static_cast<size_t>(b) * N + 2 * q) * a.dinner + d;
                if (2 * q < N) h[q].x = hp[0];
                if (2 * q + 1 < N) h[q].y = hp[a.dinner];
            }
        }
        for (int gp = 0; gp < g; ++gp) {
            const float ds = xd[gp * CW + lane];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float2 P = make_float2(ex2(A2[q].x * ds), ex2(A2[q].y * ds));
                h[q] = make_float2(fmaf(P.x, h[q].x, xh[(gp * NT + 2 * q) * CW + lane]),
                                   fmaf(P.y, h[q].y, xh[(gp * NT + 2 * q + 1) * CW + lane]));
            }
        }
    } else {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        h[q] = make_float2(0.0f, 0.0f);
        if (g > 0 && active) {
            const float* hp = a.h0 + ((static_cast<size_t>(b) * a.nseg + g) * NT + 2 * q) * a.dinner + d;
            h[q] = make_float2(hp[0], hp[a.dinner]);
        } else if (g == 0 && active && a.h_init) {
            // caller's initial state [batch][dstate][dinner]
            const float* hp = a.h_init + (static_cast<size_t>(b) * N + 2 * q) * a.dinner + d;
            if (2 * q < N) h[q].x = hp[0];
            if (2 * q + 1 < N) h[q].y = hp[a.dinner];
        }
    }
    }

    const T* Bp = static_cast<const T*>(a.B);
    const T* Cp = static_cast<const T*>(a.C);
    auto issue = [&](int k) {
        const int s = (k - kb) % S;
        T* dst = tiles + s * STAGE;
        mbar_arrive_expect_tx(&full[s], kActBytes + (bc_tma ? kBCBytes : 0u));
        tma_load_3d(dst, &maps.u, &full[s], c0, k * TS, b);
        tma_load_3d(dst + TILE, &maps.dr, &full[s], c0, k * TS, b);
        if (GATE) tma_load_3d(dst + 2 * TILE, &maps.z, &full[s], c0, k * TS, b);
        if (bc_tma) {
            tma_load_3d(dst + NTEN * TILE, &maps.B, &full[s], 0, k * TS, b);
            tma_load_3d(dst + NTEN * TILE + BCT, &maps.C, &full[s], 0, k * TS, b);
        }
    };

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0)
        for (int k = kb; k < kb + S && k < ke; ++k) issue(k);

    const bool save_y = GATE && a.ysave != nullptr;
    const bool save_ck = a.ctx != nullptr && a.nck > 0;
    int k = kb;
    for (; k < ke; ++k) {
        const int s = (k - kb) % S;
        bool ok = mbar_wait(&full[s], ((k - kb) / S) & 1, kFaultFwdWait);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;

        const T* tu = tiles + s * STAGE;
        const T* tr = tu + TILE;
        const T* tz = tu + 2 * TILE;
        const float* Bf = fwd_stage_bc<T, NT, TS>(bcs, tu + NTEN * TILE, bc_tma, Bp, Cp, a.ld_B,
                                                  a.ld_C, row0, k, L, N, lane);
        __syncwarp();
        const int jmax = min(TS, L - k * TS);

        // Phase A: the per-step scalars of the whole tile (independent across
        // steps, so their dependency chains overlap), two steps at a time in
        // f32x2 arithmetic.
        float dtv[TS], bsv[TS], gzv[TS], duv[TS];
#pragma unroll
        for (int j = 0; j < TS; j += 2) {
            const float2 uv = make_float2(Act<T>::to_f(tu[j * CW + lane]), Act<T>::to_f(tu[(j + 1) * CW + lane]));
            const float2 xr = make_float2(Act<T>::to_f(tr[j * CW + lane]), Act<T>::to_f(tr[(j + 1) * CW + lane]));
            float2 dt, gz = f2(1.0f);
            if (GATE) {
                const float2 zv =
                    make_float2(Act<T>::to_f(tz[j * CW + lane]), Act<T>::to_f(tz[(j + 1) * CW + lane]));
                float2 sz;
                softplus_sigmoid2(xr, zv, dt, sz);
                gz = mul2(zv, sz);                              // silu(z)
            } else {
                dt = softplus2(xr);
            }
            const float2 bs = DISC == 0 ? mul2(dt, uv) : uv;    // Euler: delta*u; ZOH: u
            const float2 du = mul2(f2(Dd), uv);
            dtv[j] = dt.x;
            dtv[j + 1] = dt.y;
            bsv[j] = bs.x;
            bsv[j + 1] = bs.y;
            gzv[j] = gz.x;
            gzv[j + 1] = gz.y;
            duv[j] = du.x;
            duv[j + 1] = du.y;
        }
        if (a.h_last && jmax < TS) {
            // steps past seqlen: delta = 0 keeps the state exactly (a = 1,
            // beta u = 0), so it is the state after the last step at the end
#pragma unroll
            for (int j = 0; j < TS; ++j)
                if (j >= jmax) dtv[j] = bsv[j] = 0.0f;
        }

        // Phase B: the recurrence.  Every tile runs all TS steps: past seqlen
        // the TMA tiles and B|C are zero, so the extra steps only evolve a
        // state that is never stored (or, when the final state is asked for,
        // leave it unchanged: see above).  Outputs go to a staging tile in shared
        // memory (double-buffered) and leave by TMA store; the store of tile
        // k-2 must have finished reading its buffer first.
        if (lane == 0 && k - kb >= 2) bulk_wait_read_1();
        __syncwarp();
        T* so = ost + ((k - kb) & 1) * 2 * TILE;
        float* sc = ckst + ((k - kb) & 1) * NCK * NT * CW;
        // The recurrence first, the staging stores after it: a store could
        // alias the next step's B|C loads, which would then have to wait.
        float yv[TS];
        float2 hck[NCK][NQ];                            // states at the chunk ends
#pragma unroll
        for (int j = 0; j < TS; ++j) {
            yv[j] = fwd_step<NT, DISC>(h, A2, Anat, invA, Bf + j * NT, Bf + BCT + j * NT, dtv[j], bsv[j]) +
                    duv[j];
            if ((j + 1) % kChunk == 0) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) hck[j / kChunk][q] = h[q];
            }
        }
#pragma unroll
        for (int j = 0; j < TS; ++j) {
            so[j * CW + lane] = Act<T>::from_f(GATE ? yv[j] * gzv[j] : yv[j]);
            if (save_y) so[TILE + j * CW + lane] = Act<T>::from_f(yv[j]);
        }
        if (save_ck) {
            // state after the last step of a chunk = checkpoint of the next one
#pragma unroll
            for (int m = 0; m < NCK; ++m)
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    sc[(m * NT + 2 * q) * CW + lane] = hck[m][q].x;
                    sc[(m * NT + 2 * q + 1) * CW + lane] = hck[m][q].y;
                }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(&maps.out, so, c0, k * TS, b);
            if (save_y) tma_store_3d(&maps.y, so + TILE, c0, k * TS, b);
            if (save_ck) {
#pragma unroll
                for (int m = 0; m < NCK; ++m) {
                    const int t1 = k * TS + (m + 1) * kChunk;   // first step of the next chunk
                    if (t1 < L)
                        tma_store_2d(&maps.ck, sc + m * NT * CW, c0, (b * a.nck + t1 / kChunk - 1) * NT);
                }
            }
            bulk_commit();
            if (k + S < ke) issue(k + S);
        }
    }
    if (k < ke && lane == 0) {
        // A wait gave up: drain the copies still in flight (bounded) before exit.
        for (int kk = k; kk < ke && kk < k + S; ++kk)
            mbar_wait(&full[(kk - kb) % S], ((kk - kb) / S) & 1, kFaultDrain);
    }
    if (lane == 0) bulk_wait_all();   // the staged stores have left shared memory
    if (a.h_last && k == ke && ke == ntiles && active) {
        float* hp = a.h_last + static_cast<size_t>(b) * N * a.dinner + d;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            if (2 * q < N) hp[static_cast<size_t>(2 * q) * a.dinner] = h[q].x;
            if (2 * q + 1 < N) hp[static_cast<size_t>(2 * q + 1) * a.dinner] = h[q].y;
        }
    }
}

// Combine of the time segments: one thread per (batch row, state, channel)
// walks the segments in order, from the caller's initial state (or 0), and
// writes the state entering each segment.
template <int NT>
__global__ void scan_fwd_combine_kernel(const ScanFwdArgs a) {
    const size_t total = static_cast<size_t>(a.batch) * NT * a.dinner;
    const size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    if (i >= total) return;
    const int d = static_cast<int>(i % a.dinner);
    const int n = static_cast<int>((i / a.dinner) % NT);
    const int b = static_cast<int>(i / (static_cast<size_t>(a.dinner) * NT));
    const float A2 = n < a.dstate ? a2_from_alog(a.A_log[static_cast<size_t>(d) * a.dstate + n]) : 0.0f;
    float h = (a.h_init && n < a.dstate)
                  ? a.h_init[(static_cast<size_t>(b) * a.dstate + n) * a.dinner + d] : 0.0f;
    for (int g = 0; g + 1 < a.nseg; ++g) {
        const size_t sg = static_cast<size_t>(b) * a.nseg + g;
        const float P = ex2(A2 * a.seg_ds[sg * a.dinner + d]);   // product of a_t over segment g
        h = fmaf(P, h, a.seg_h[(sg * NT + n) * a.dinner + d]);
        a.h0[((sg + 1) * NT + n) * a.dinner + d] = h;
    }
}

template <typename T, int NT, int DISC, bool GATE>
static cudaError_t launch_fwd_t(const FwdMaps& m, const ScanFwdArgs& a, cudaStream_t st) {
    const size_t smem = fwd_warp_smem_bytes<T, NT, DISC, GATE>();
    const unsigned gx = (a.dinner + kFwdChannels - 1) / kFwdChannels;
    cudaError_t e;
    if (a.nseg > 1 && a.nseg <= kFwdChunkWarps) {
        // the segments as the warps of one CTA per (channel tile, batch row),
        // when those CTAs (one shared-memory region per warp) all fit at once;
        // otherwise separate CTAs per segment, which fit more per SM
        auto kc = scan_fwd_kernel<T, NT, DISC, GATE, true>;
        const size_t smc = a.nseg * smem + fwd_chunk_xchg_bytes<NT>(a.nseg);
        e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kFwdChunkWarps * smem + fwd_chunk_xchg_bytes<NT>(kFwdChunkWarps)));
        if (e != cudaSuccess) return e;
        int dev = 0, nsm = 0, per_sm = 0;
        e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kc, 32 * a.nseg, smc);
        if (e != cudaSuccess) return e;
        if (static_cast<long long>(gx) * a.batch <= static_cast<long long>(nsm) * per_sm) {
            kc<<<dim3(gx, a.batch, 1), 32 * a.nseg, smc, st>>>(m, a);
            return cudaGetLastError();
        }
    }
    auto kern = scan_fwd_kernel<T, NT, DISC, GATE, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (a.nseg > 1) {
        // segment pass (every segment but the last), then the combine
        constexpr int STG = 2 * kFwdTile * kFwdChannels + kFwdTile * NT;
        const size_t sm1 = kFwdStages * STG * sizeof(T) + kFwdTile * NT * sizeof(float) +
                           kFwdStages * sizeof(uint64_t);
        auto k1 = scan_fwd_segsum_kernel<T, NT, DISC>;
        e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm1));
        if (e != cudaSuccess) return e;
        k1<<<dim3(gx, a.batch, a.nseg - 1), 32, sm1, st>>>(m, a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const size_t total = static_cast<size_t>(a.batch) * NT * a.dinner;
        scan_fwd_combine_kernel<NT><<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    kern<<<dim3(gx, a.batch, a.nseg), 32, smem, st>>>(m, a);
    return cudaGetLastError();
}

template <typename T, int NT>
static cudaError_t launch_fwd_nt(int disc, bool gate, const FwdMaps& m, const ScanFwdArgs& a,
                                 cudaStream_t st) {
    if (disc == 0)
        return gate ? launch_fwd_t<T, NT, 0, true>(m, a, st) : launch_fwd_t<T, NT, 0, false>(m, a, st);
    return gate ? launch_fwd_t<T, NT, 1, true>(m, a, st) : launch_fwd_t<T, NT, 1, false>(m, a, st);
}

cudaError_t read_clear_fault_fwd(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_ssm_fault, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_ssm_fault, &zero, sizeof(unsigned));
}

cudaError_t launch_scan_fwd(int dtype, int nt, int disc, bool gate, const FwdMaps& maps,
                            const ScanFwdArgs& a, cudaStream_t stream) {
    if (dtype == 0)
        return nt == 8 ? launch_fwd_nt<float, 8>(disc, gate, maps, a, stream)
                       : launch_fwd_nt<float, 16>(disc, gate, maps, a, stream);
    return nt == 8 ? launch_fwd_nt<__nv_bfloat16, 8>(disc, gate, maps, a, stream)
                   : launch_fwd_nt<__nv_bfloat16, 16>(disc, gate, maps, a, stream);
}

}  // namespace ssm

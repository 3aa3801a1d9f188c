// scan_bwd.cu -- selective-scan backward for sm_103a.
//
// Computes mamba1_cpu.ts mamba1CpuBackward steps 9 (gate) and 8 (scan, walked
// backwards in time), page "@seanhogg/builderforce-memory-engine 2026.7.12 ->
// 2026.9.27":
//   g_t      = C_t dy_t + a_{t+1} g_{t+1}              (dL/dh_t; 0 after the last step)
//   du_t     = D dy_t + sum_n g_t beta_t/u_t           dz_t = dout_t y_t silu'(z_t)
//   ddelta_t = sum_n g_t (a_t h_{t-1} A + u_t B_t d(beta/B)/d delta)
//   dA       = sum_t g_t (a_t h_{t-1} delta_t + u_t B_t d(beta/B)/dA)
//   dB_t     = sum_d g_t u_t beta_t/B_t     dC_t = sum_d dy_t h_t     dD = sum dy u
//   dA_log   = dA * A inside (-10, 5), exactly 0 at or beyond the bounds
//   ddelta_raw = ddelta * sigmoid(delta_raw)
//
// Design (GB300): the forward saved h every kChunk (= 8) steps.  A warp-sized
// CTA owns 32 channels of one batch row and walks the chunks last to first.
// For each chunk it recomputes h forward from the checkpoint (pass B), keeping
// a_t h_{t-1} in registers, then runs the reverse recurrence for g over
// the chunk.  Each lane owns 4 channels x dstate/4 states (16 chains), so the
// sums over states (y, sum g B, sum g A a h) and over channels (dB, dC) are
// mostly register accumulations.  Per step, a lane's dB/dC partials (its 4
// channels) go to shared memory by channel group; once per chunk the warp
// adds the 8 groups with float4 loads and writes the rows of its own partial
// plane with plain vector stores (no inter-CTA synchronisation: an earlier
// cluster/DSMEM exchange cost a cluster-scope release fence per chunk, about
// 16% of the kernel); scan_reduce_kernel adds the planes and also finishes
// dA_log and dD.
#include <algorithm>

#include "scan_args.cuh"
#include "ssm_common.cuh"

namespace ssm {

// Loads CPL consecutive floats (CPL = 2 or 4) from shared memory.
template <int CPL>
__device__ __forceinline__ void ld_cpl(const float* p, float (&v)[CPL]) {
    if constexpr (CPL == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2*>(p);
        v[0] = t.x; v[1] = t.y;
    }
}
template <int CPL>
__device__ __forceinline__ void st_cpl(float* p, const float (&v)[CPL]) {
    if constexpr (CPL == 4)
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    else
        *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}

// Two adjacent activations (an even element index) as one 4- or 8-byte access.
template <typename T> struct ActPair;
template <> struct ActPair<float> {
    static __device__ __forceinline__ float2 load(const float* p) { return *reinterpret_cast<const float2*>(p); }
    static __device__ __forceinline__ void store(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
};
template <> struct ActPair<__nv_bfloat16> {
    static __device__ __forceinline__ float2 load(const __nv_bfloat16* p) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float2 v) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __float22bfloat162_rn(v);
    }
};

// Segment pass of the time-parallel backward: for segment sg >= 1 of batch
// row b, walk its steps last to first with g = 0 after its last step,
//   g_t = C_t dy_t + a_{t+1} g_{t+1},
// and keep g at its first step, the sum of delta over its steps after the
// first, and delta at its first step.  Because the product of a_s over steps
// t0+1 .. t1+1 is exp(A (that sum + delta at t1+1)), the true g at the first
// step of a segment is its zero-carry value plus that product times the true
// g at the first step of the next segment (scan_bwd_combine_kernel).  A lane
// owns NT * CW / 32 states of one channel: lane = (channel lane % CW, half
// lane / CW of the states).  One warp; smem holds the stages and barriers of
// the pass.  Returns false if a bounded wait gave up.
template <typename T, int NT, bool GATE, int CW>
__device__ __forceinline__ bool bwd_segsum_run(const BwdMaps& maps, const ScanBwdArgs& a, unsigned char* smem,
                                               int c0, int b, int sg, int lane, float2 (&gl)[NT * CW / 64],
                                               float& dsum, float& dfirst) {

    constexpr int TC = kChunk;
    constexpr int S = kBwdStages;
    constexpr int SPL = 32 / CW;                 // lanes per channel
    constexpr int NL = NT / SPL;                 // states per lane
    constexpr int NQ = NL / 2;
    constexpr int TILE = TC * CW;
    constexpr int BCT = TC * NT;
    constexpr int NTEN = GATE ? 3 : 2;           // delta_raw, dout, [z]
    constexpr int STAGE = NTEN * TILE + BCT;     // + C
    constexpr uint32_t kActBytes = NTEN * TILE * sizeof(T);
    constexpr uint32_t kCBytes = BCT * sizeof(T);
    static_assert((STAGE * sizeof(T)) % 128 == 0, "stages stay 128-byte aligned");

    T* tiles = reinterpret_cast<T*>(smem);                                   // [S][STAGE]
    float* csm = reinterpret_cast<float*>(smem + S * STAGE * sizeof(T));    // [TC][NT] fp32 C
    uint64_t* full = reinterpret_cast<uint64_t*>(csm + BCT);                 // [S]

    const int c = lane % CW, half = lane / CW;
    const int nbase = half * NL;
    const int d = c0 + c;
    const bool active = d < a.dinner;
    const int L = a.seqlen, N = a.dstate;
    const int nchunks = (L + TC - 1) / TC;
    const int kcb = sg * a.seg_chunks;
    const int kce = min(nchunks, kcb + a.seg_chunks);
    const int nit = kce - kcb;
    const size_t row0 = static_cast<size_t>(b) * L;
    const bool bc_tma = a.bc_tma != 0;

    float2 A2[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = nbase + 2 * q + e;
            const bool ok = active && n < N;
            v[e] = ok ? a2_from_alog(a.A_log[static_cast<size_t>(d) * N + n]) : 0.0f;
        }
        A2[q] = make_float2(v[0], v[1]);
    }
    float2 an[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) gl[q] = an[q] = make_float2(0.0f, 0.0f);
    dsum = 0.0f;
    dfirst = 0.0f;

    const T* Cp = static_cast<const T*>(a.C);
    auto issue = [&](int it) {
        const int kc = kce - 1 - it;
        const int s = it % S;
        T* dst = tiles + s * STAGE;
        mbar_arrive_expect_tx(&full[s], kActBytes + (bc_tma ? kCBytes : 0u));
        tma_load_3d(dst, &maps.dr, &full[s], c0, kc * TC, b);
        tma_load_3d(dst + TILE, &maps.dout, &full[s], c0, kc * TC, b);
        if (GATE) tma_load_3d(dst + 2 * TILE, &maps.z, &full[s], c0, kc * TC, b);
        if (bc_tma) tma_load_3d(dst + NTEN * TILE, &maps.C, &full[s], 0, kc * TC, b);
    };
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0)
        for (int it = 0; it < S && it < nit; ++it) issue(it);

    int it = 0;
    for (; it < nit; ++it) {
        const int kc = kce - 1 - it;
        const int s = it % S;
        bool ok = mbar_wait(&full[s], (it / S) & 1, kFaultBwdWait);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const T* tr = tiles + s * STAGE;
        const T* tg = tr + TILE;
        const T* tz = tr + 2 * TILE;
        const T* tc = tr + NTEN * TILE;
        const float* Cf;
        if (bc_tma && sizeof(T) == 4) {
            Cf = reinterpret_cast<const float*>(tc);
        } else {
            for (int e = lane; e < BCT; e += 32) {
                float v;
                if (bc_tma) {
                    v = Act<T>::to_f(tc[e]);
                } else {
                    const int j = e / NT, n = e % NT, t = kc * TC + j;
                    v = (n < N && t < L) ? Act<T>::load(Cp + (row0 + t) * a.ld_C + n) : 0.0f;
                }
                csm[e] = v;
            }
            Cf = csm;
        }
        __syncwarp();
#pragma unroll
        for (int j = TC - 1; j >= 0; --j) {
            const int t = kc * TC + j;
            const float xr = Act<T>::to_f(tr[j * CW + c]);
            const float go = Act<T>::to_f(tg[j * CW + c]);
            float dt, dy = go;
            if (GATE) {
                const float zv = Act<T>::to_f(tz[j * CW + c]);
                float sz;
                softplus_sigmoid(xr, zv, dt, sz);
                dy = go * zv * sz;
            } else {
                float e;
                dt = softplus_e(xr, e);
            }
            // past seqlen the tiles are zero: dy = 0 keeps g at 0 there
            const float2 dy2 = f2(dy), dt2 = f2(dt);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float2 Cq = *reinterpret_cast<const float2*>(Cf + j * NT + nbase + 2 * q);
                gl[q] = fma2(an[q], gl[q], mul2(Cq, dy2));
                const float2 x = mul2(dt2, A2[q]);
                an[q] = make_float2(ex2(x.x), ex2(x.y));
            }
            if (t < L) {
                if (t == kcb * TC) dfirst = dt;
                else dsum += dt;
            }
        }
        __syncwarp();
        if (lane == 0 && it + S < nit) issue(it + S);
    }
    if (it < nit && lane == 0) {
        for (int k2 = it; k2 < nit && k2 < it + S; ++k2)
            mbar_wait(&full[k2 % S], (k2 / S) & 1, kFaultDrain);
    }
    return it == nit;
}

// Shared memory of bwd_segsum_run.
template <typename T, int NT, bool GATE, int CW>
constexpr size_t bwd_segsum_smem_bytes() {
    return kBwdStages * ((GATE ? 3 : 2) * kChunk * CW + kChunk * NT) * sizeof(T) + kChunk * NT * sizeof(float) +
           kBwdStages * sizeof(uint64_t);
}

template <typename T, int NT, bool GATE, int CW>
__global__ void __launch_bounds__(32, 1)
scan_bwd_segsum_kernel(const __grid_constant__ BwdMaps maps, const ScanBwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int NL = NT * CW / 32, NQ = NL / 2;
    const int lane = threadIdx.x;
    const int c = lane % CW, half = lane / CW, nbase = half * NL;
    const int c0 = blockIdx.x * CW, b = blockIdx.y, sg = blockIdx.z + 1;   // segments 1 .. nseg-1
    const int d = c0 + c;
    float2 gl[NQ];
    float dsum, dfirst;
    const bool done = bwd_segsum_run<T, NT, GATE, CW>(maps, a, smem, c0, b, sg, lane, gl, dsum, dfirst);
    if (d < a.dinner && done) {
        const size_t pb = static_cast<size_t>(b) * a.nseg + sg;
        float* gp = a.seg_g + (pb * NT + nbase) * a.dinner + d;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            gp[static_cast<size_t>(2 * q) * a.dinner] = gl[q].x;
            gp[static_cast<size_t>(2 * q + 1) * a.dinner] = gl[q].y;
        }
        if (half == 0) {
            a.seg_ds[pb * a.dinner + d] = dsum;
            a.seg_d0[pb * a.dinner + d] = dfirst;
        }
    }
}

// Shared memory of one backward warp: its stages, checkpoint tiles, per-step
// scalars, partial sums and barriers.
template <typename T, int NT, int DISC, bool GATE, int CW>
__host__ __device__ constexpr size_t bwd_smem_bytes() {
    constexpr int TC = kChunk;
    constexpr int NTEN = GATE ? 5 : 3;
    constexpr int NQN = DISC == 1 ? 3 : 2;
    return kBwdStages * (NTEN * TC * CW + 2 * TC * NT) * sizeof(T)   // activation, B, C tiles
           + kBwdStages * NT * CW * sizeof(float)      // checkpoint tiles
           + 2 * TC * NT * sizeof(float)               // fp32 B|C (bf16 or unaligned B/C)
           + 3 * TC * CW * sizeof(float)               // delta, delta*u, dy
           + TC * NQN * 4 * CW * sizeof(float)         // state-sum partials
           + (CW == 32 ? TC : 4) * 9 * NT * sizeof(float)   // dB or dC partials by channel group
           + 2 * TC * CW * sizeof(float)               // sigmoid(delta_raw), sigmoid(z)
           + kBwdStages * sizeof(uint64_t);
}

// CW = channels per CTA (one warp): 32 (each lane 4 channels) or 16 (each lane
// 2 channels: half the work per warp and fewer registers, so twice the warps
// when the problem has few channels).
//
// CHUNKED: the a.nseg time segments of one channel tile are the warps of one
// CTA.  Each warp but the first first walks its segment backwards from g = 0
// (bwd_segsum_run) and leaves g at its first step, the sum of delta over its
// later steps and delta at its first step in shared memory; after a CTA
// barrier each warp but the last combines the segments after its own into its
// carry (dL/dh and delta at the first step of the next segment), then runs its
// segment as below.  Each warp has its own shared-memory region of
// bwd_warp_bytes(); the exchange follows them.
template <typename T, int NT, int DISC, bool GATE, int CW, bool CHUNKED = false>
__global__ void __launch_bounds__(CHUNKED ? 32 * kBwdChunkWarps : 32,
                                  CHUNKED ? kBwdMinBlocks16 / kBwdChunkWarps : (CW == 16 ? kBwdMinBlocks16 : 1))
scan_bwd_kernel(const __grid_constant__ BwdMaps maps, const ScanBwdArgs a) {
    constexpr int TC = kChunk;
    constexpr int S = kBwdStages;
    constexpr int CPL = CW / 8;                 // channels per lane
    constexpr int NS = NT / 4;                  // states per lane
    constexpr int NTEN = GATE ? 5 : 3;          // u, delta_raw, dout, [z, y]
    constexpr int TILE = TC * CW;
    constexpr int BCT = TC * NT;                // elements per B or C tile
    constexpr int STAGE = NTEN * TILE + 2 * BCT;
    constexpr uint32_t kActBytes = NTEN * TILE * sizeof(T);
    constexpr uint32_t kBCBytes = 2 * BCT * sizeof(T);
    constexpr uint32_t kCkBytes = NT * CW * sizeof(float);
    constexpr int BCN = 2 * TC * NT;
    static_assert((STAGE * sizeof(T)) % 128 == 0, "stages stay 128-byte aligned");
    static_assert((CPL == 2 || CPL == 4) && TC == 8, "lane layout below");
    constexpr int SPL = 32 / CW;                // steps per lane-iteration of pro/epilogue
    constexpr bool ZOH = DISC == 1;
    constexpr int NQN = ZOH ? 3 : 2;            // state sums kept per (step, channel)
    constexpr int PR = CW == 32 ? TC : 4;       // steps per dB/dC flush
    constexpr int PJ = 9 * NT;                  // padded partial row: conflict-free float4 sums

    extern __shared__ __align__(128) unsigned char smem_all[];
    const int wid = CHUNKED ? static_cast<int>(threadIdx.x >> 5) : 0;
    constexpr size_t warp_bytes = CHUNKED ? (bwd_smem_bytes<T, NT, DISC, GATE, CW>() + 127) / 128 * 128 : 0;
    unsigned char* smem = smem_all + wid * warp_bytes;
    T* tiles = reinterpret_cast<T*>(smem);                               // [S][STAGE]
    float* cks = reinterpret_cast<float*>(smem + S * STAGE * sizeof(T)); // [S][NT][CW]
    float* bcs = cks + S * NT * CW;                                      // [TC][NT] B | [TC][NT] C
    float* Pd = bcs + BCN;                                               // [TC][CW] delta
    float* Pbs = Pd + TILE;                                              // [TC][CW] delta*u | u
    float* Pdy = Pbs + TILE;                                             // [TC][CW] dy
    float* part = Pdy + TILE;                                            // [TC][NQN][4][CW]
    float* pbuf = part + TC * NQN * 4 * CW;                              // [PR][PJ] dB or dC by channel group
    float* Psdr = pbuf + PR * PJ;                                        // [TC][CW] sigmoid(delta_raw)
    float* Psz = Psdr + TILE;                                            // [TC][CW] sigmoid(z)
    uint64_t* full = reinterpret_cast<uint64_t*>(Psz + TILE);            // [S]

    const int lane = threadIdx.x & 31;
    const int cg = lane >> 2, ng = lane & 3;     // channel group (CPL channels), state group (NS states)
    const int cbase = cg * CPL;
    const int c0 = blockIdx.x * CW;
    const int b = blockIdx.y;
    const int L = a.seqlen, N = a.dstate, Dn = a.dinner;
    const int nchunks = (L + TC - 1) / TC;
    // this CTA's (warp's) time segment: chunks [kcb, kce), walked last to first
    const int sg = CHUNKED ? wid : static_cast<int>(blockIdx.z);
    const int kcb = sg * a.seg_chunks;
    const int kce = min(nchunks, kcb + a.seg_chunks);
    const int nit = kce - kcb;
    const size_t plane_b = static_cast<size_t>(b) * a.nseg + sg;   // dA / dD plane
    const size_t row0 = static_cast<size_t>(b) * L;
    // prologue / epilogue layout: lane = (channel pc, step phase pj)
    const int pc = lane % CW, pj = lane / CW;
    const int dch = c0 + pc;
    const bool lane_ok = dch < Dn;
    // column of channel c in state-group row k of `part`: rotated (CW = 32) or
    // xor-swizzled (CW = 16) so that the per-step writes and the epilogue's
    // reads hit distinct banks
    auto part_col = [](int c, int k) {
        return CW == 32 ? ((c + 8 * k) & 31) : (c ^ (8 * (k >> 1)));
    };

    // per (channel, state) constants of this lane's chains: A log2(e) (0 on
    // padding states and channels) [and 1/A for ZOH]
    float2 A2r[CPL][NS / 2], iAr[CPL][NS / 2];
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
        for (int p = 0; p < NS / 2; ++p) {
            float v[2], w[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int d = c0 + cbase + i, n = ng * NS + 2 * p + e;
                const bool ok = d < Dn && n < N;
                const float A = ok ? a_from_alog(a.A_log[static_cast<size_t>(d) * N + n]) : -1.0f;
                v[e] = ok ? A * kLog2e : 0.0f;
                w[e] = 1.0f / A;
            }
            A2r[i][p] = make_float2(v[0], v[1]);
            iAr[i][p] = make_float2(w[0], w[1]);
        }
    const float Dd = (lane_ok && a.D) ? a.D[dch] : 0.0f;

    const T* Bp = static_cast<const T*>(a.B);
    const T* Cp = static_cast<const T*>(a.C);
    const bool bc_tma = a.bc_tma != 0;
    auto issue = [&](int it) {
        const int kc = kce - 1 - it;
        const int s = it % S;
        T* dst = tiles + s * STAGE;
        mbar_arrive_expect_tx(&full[s], kActBytes + (kc > 0 ? kCkBytes : 0u) +
                                            (bc_tma ? kBCBytes : 0u));
        if (bc_tma) {
            tma_load_3d(dst + NTEN * TILE, &maps.B, &full[s], 0, kc * TC, b);
            tma_load_3d(dst + NTEN * TILE + BCT, &maps.C, &full[s], 0, kc * TC, b);
        }
        tma_load_3d(dst, &maps.u, &full[s], c0, kc * TC, b);
        tma_load_3d(dst + TILE, &maps.dr, &full[s], c0, kc * TC, b);
        tma_load_3d(dst + 2 * TILE, &maps.dout, &full[s], c0, kc * TC, b);
        if (GATE) {
            tma_load_3d(dst + 3 * TILE, &maps.z, &full[s], c0, kc * TC, b);
            tma_load_3d(dst + 4 * TILE, &maps.y, &full[s], c0, kc * TC, b);
        }
        if (kc > 0)
            tma_load_2d(cks + s * NT * CW, &maps.ck, &full[s], c0, (b * a.nck + kc - 1) * NT);
    };
    // CHUNKED: the segment pass of the warps after the first, the exchange and
    // this warp's carry ([NT][CW] dL/dh, then [CW] delta) in shared memory
    float* xcarry = nullptr;
    if constexpr (CHUNKED) {
        constexpr int SNL = NT * CW / 32, SNQ = SNL / 2;
        const int nw = static_cast<int>(blockDim.x >> 5);
        float* xg = reinterpret_cast<float*>(smem_all + nw * warp_bytes);    // [nseg][NT][CW]
        float* xds = xg + nw * NT * CW;                                       // [nseg][CW]
        float* xd0 = xds + nw * CW;                                           // [nseg][CW]
        xcarry = xd0 + nw * CW + wid * (NT + 1) * CW;                         // [nseg][NT + 1][CW]
        const int sc = lane % CW, shalf = lane / CW, snb = shalf * SNL;
        if (sg >= 1) {
            float2 gl[SNQ];
            float dsum, dfirst;
            bwd_segsum_run<T, NT, GATE, CW>(maps, a, smem, c0, b, sg, lane, gl, dsum, dfirst);
            if (lane == 0)
                for (int s2 = 0; s2 < S; ++s2)
                    mbar_inval(reinterpret_cast<uint64_t*>(smem + bwd_segsum_smem_bytes<T, NT, GATE, CW>() -
                                                           S * sizeof(uint64_t)) + s2);
#pragma unroll
            for (int q = 0; q < SNQ; ++q) {
                xg[(sg * NT + snb + 2 * q) * CW + sc] = gl[q].x;
                xg[(sg * NT + snb + 2 * q + 1) * CW + sc] = gl[q].y;
            }
            if (shalf == 0) {
                xds[sg * CW + sc] = dsum;
                xd0[sg * CW + sc] = dfirst;
            }
        }
        fence_proxy_async_smem();   // the stages are TMA destinations again below
        __syncthreads();
        if (sg + 1 < a.nseg) {
            // carry = true g at the first step of segment sg + 1, walking the
            // segments last to first as the global combine does
            const int dd = c0 + sc;
#pragma unroll
            for (int q = 0; q < SNL; ++q) {
                const int n = snb + q;
                const float A2 = (dd < Dn && n < N) ? a2_from_alog(a.A_log[static_cast<size_t>(dd) * N + n]) : 0.0f;
                float carry = 0.0f;
                for (int s2 = a.nseg - 1; s2 > sg; --s2) {
                    float gstart = xg[(s2 * NT + n) * CW + sc];
                    if (s2 + 1 < a.nseg)
                        gstart = fmaf(ex2(A2 * (xds[s2 * CW + sc] + xd0[(s2 + 1) * CW + sc])), carry, gstart);
                    carry = gstart;
                }
                xcarry[n * CW + sc] = carry;
            }
            if (shalf == 0) xcarry[NT * CW + sc] = xd0[(sg + 1) * CW + sc];
        }
        __syncwarp();
    }

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0)
        for (int it = 0; it < S && it < nit; ++it) issue(it);
    __syncwarp();

    // The carries of the reverse recurrence (g) and the dA accumulators: with
    // ZOH B, and in 16-channel CTAs held to 128 registers, they live in
    // registers only during the reverse pass and epilogue and are parked in the
    // (then idle) state-sum buffer between chunks, so pass B can hold the
    // chunk's a h_{t-1} values in registers without spilling; otherwise they
    // stay in registers throughout (no shared-memory round trip per chunk).
    constexpr bool kPark = DISC == 1 || (CW == 16 && !CHUNKED);
    float* stash = part;
    static_assert(2 * CPL * NS * 32 <= TC * NQN * 4 * CW, "stash fits in the partials buffer");
    float2 dA[CPL][NS / 2], g[CPL][NS / 2];
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
        for (int p = 0; p < NS / 2; ++p) dA[i][p] = g[i][p] = make_float2(0.f, 0.f);
    auto park = [&]() {
        if constexpr (!kPark) return;
#pragma unroll
        for (int i = 0; i < CPL; ++i)
#pragma unroll
            for (int p = 0; p < NS / 2; ++p) {
                reinterpret_cast<float2*>(stash)[(i * NS / 2 + p) * 32 + lane] = g[i][p];
                reinterpret_cast<float2*>(stash)[((CPL + i) * NS / 2 + p) * 32 + lane] = dA[i][p];
            }
    };
    auto unpark = [&]() {
        if constexpr (!kPark) return;
#pragma unroll
        for (int i = 0; i < CPL; ++i)
#pragma unroll
            for (int p = 0; p < NS / 2; ++p) {
                g[i][p] = reinterpret_cast<const float2*>(stash)[(i * NS / 2 + p) * 32 + lane];
                dA[i][p] = reinterpret_cast<const float2*>(stash)[((CPL + i) * NS / 2 + p) * 32 + lane];
            }
    };
    float dl_next[CPL];                         // delta of the step after this chunk
#pragma unroll
    for (int i = 0; i < CPL; ++i) dl_next[i] = 0.0f;
    if (sg + 1 < a.nseg) {
        // dL/dh and delta at the first step of the next segment
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int d = c0 + cbase + i;
            if (d < Dn && CHUNKED) {
                dl_next[i] = xcarry[NT * CW + cbase + i];
#pragma unroll
                for (int p = 0; p < NS / 2; ++p)
                    g[i][p] = make_float2(xcarry[(ng * NS + 2 * p) * CW + cbase + i],
                                          xcarry[(ng * NS + 2 * p + 1) * CW + cbase + i]);
            } else if (d < Dn) {
                dl_next[i] = a.carry_dl[plane_b * Dn + d];
#pragma unroll
                for (int p = 0; p < NS / 2; ++p) {
                    const float* cp = a.carry_g + (plane_b * NT + ng * NS + 2 * p) * Dn + d;
                    g[i][p] = make_float2(cp[0], cp[Dn]);
                }
            }
        }
    }
    park();
    float dD_acc = 0.0f;
    // 32-channel epilogue: lane = (step parity ep, channel pair 2 ecp, 2 ecp + 1)
    const int ep = lane >> 4, ec = c0 + 2 * (lane & 15);
    const bool eok0 = ec < Dn, eok1 = ec + 1 < Dn;
    const float2 eD = make_float2(eok0 && a.D ? a.D[ec] : 0.0f, eok1 && a.D ? a.D[ec + 1] : 0.0f);
    float2 eDD = make_float2(0.0f, 0.0f);

    T* dup = static_cast<T*>(a.du);
    T* ddp = static_cast<T*>(a.ddelta);
    T* dzp = static_cast<T*>(a.dz);
    // outputs written as channel pairs when every pair is aligned for it
    const bool pair_st = eok1 &&
        ((reinterpret_cast<uintptr_t>(dup) | reinterpret_cast<uintptr_t>(ddp) |
          (GATE ? reinterpret_cast<uintptr_t>(dzp) : 0)) % (2 * sizeof(T))) == 0 &&
        a.ld_du % 2 == 0 && a.ld_ddelta % 2 == 0 && (!GATE || a.ld_dz % 2 == 0);
    bool ok = true;
    int waited = 0;

    // this CTA's partial plane of dB|dC: [batch][seqlen][2][NT]
    float* plane = a.ws_bc + static_cast<size_t>(blockIdx.x) * a.batch * L * 2 * NT;
    // dB or dC partials of one step, summed over this lane's CPL channels, go
    // to pbuf by channel group; flush() adds the 8 groups (the CTA's channels)
    // for PR steps and writes those rows of the plane, float4 per lane.
    auto store_partial = [&](int j, const float2 (&v)[NS / 2]) {
        float* pp = pbuf + (j % PR) * PJ + cg * NT + ng * NS;
        if constexpr (NS == 4)
            *reinterpret_cast<float4*>(pp) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
        else
            *reinterpret_cast<float2*>(pp) = v[0];
    };
    auto flush = [&](int coff, int tf, int nrows) {
        constexpr int NM = NT / 4;
        __syncwarp();
        if (lane < PR * NM) {
            const int j = lane / NM, m = lane % NM;
            float4 acc = *reinterpret_cast<const float4*>(pbuf + j * PJ + 4 * m);
#pragma unroll
            for (int c = 1; c < 8; ++c) {
                const float4 v = *reinterpret_cast<const float4*>(pbuf + j * PJ + c * NT + 4 * m);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            if (j < nrows)
                *reinterpret_cast<float4*>(plane + (static_cast<size_t>(b) * L + tf + j) * 2 * NT + coff +
                                           4 * m) = acc;
        }
        __syncwarp();
    };

    for (int it = 0; it < nit; ++it) {
        const int kc = kce - 1 - it;
        const int t0 = kc * TC;
        const int jmax = min(TC, L - t0);
        const int s = it % S;

        if (ok) ok = mbar_wait(&full[s], (it / S) & 1, kFaultBwdWait);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) waited = it + 1;

        const T* tu = tiles + s * STAGE;
        const T* tr = tu + TILE;
        const T* tg = tu + 2 * TILE;
        const T* tz = tu + 3 * TILE;
        const T* ty = tu + 4 * TILE;
        const float* ck = cks + s * NT * CW;
        if (ok) {
            // fp32 B and C of this chunk: [TC][NT] each.  fp32 TMA tiles are used
            // in place; bf16 tiles are widened into bcs, 8 values per lane.
            const float* Bf;
            const float* Cf;
            {
                const T* Bs = tu + NTEN * TILE;
                if (bc_tma && sizeof(T) == 4) {
                    Bf = reinterpret_cast<const float*>(Bs);
                } else if (bc_tma) {
                    for (int g8 = lane; g8 < BCN / 8; g8 += 32) {
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
                    Bf = bcs;
                } else {
                    for (int e = lane; e < BCN; e += 32) {
                        const int isC = e >= BCT, j = (e % BCT) / NT, n = e % NT, t = t0 + j;
                        float v = 0.0f;
                        if (t < L && n < N) {
                            const size_t r = row0 + t;
                            v = isC ? Act<T>::load(Cp + r * a.ld_C + n) : Act<T>::load(Bp + r * a.ld_B + n);
                        }
                        bcs[e] = v;
                    }
                    Bf = bcs;
                }
                Cf = Bf + BCT;
            }

            // ---- prologue: delta, delta*u (or u), dy, sigmoid(delta_raw),
            //      sigmoid(z).  All TC steps run: past seqlen the tiles, B and
            //      C are zero, so dy = 0 and the extra steps add nothing.
            //      32-channel CTAs: lane = (step parity, channel pair) as in
            //      the epilogue; 16-channel CTAs: lane = (channel, step parity).
            if constexpr (CW == 32) {
                const int ce = ec - c0;
                float2 uv[TC / 2], xr[TC / 2], go[TC / 2], zv[TC / 2];
#pragma unroll
                for (int jj = 0; jj < TC / 2; ++jj) {
                    const int e = (2 * jj + ep) * CW + ce;
                    uv[jj] = ActPair<T>::load(tu + e);
                    xr[jj] = ActPair<T>::load(tr + e);
                    go[jj] = ActPair<T>::load(tg + e);
                    zv[jj] = GATE ? ActPair<T>::load(tz + e) : f2(0.0f);
                }
                float2 sxv[TC / 2];
#pragma unroll
                for (int jj = 0; jj < TC / 2; ++jj) {
                    float2 dt, sx, dy = go[jj];
                    if (GATE) {
                        float2 sz;
                        softplus_sig_xz2(xr[jj], zv[jj], dt, sx, sz);
                        dy = mul2(mul2(go[jj], zv[jj]), sz);
                        zv[jj] = sz;                            // reuse: sigmoid(z)
                    } else {
                        softplus_sig_x2(xr[jj], dt, sx);
                    }
                    sxv[jj] = sx;
                    xr[jj] = dt;                                // reuse: delta
                    go[jj] = dy;                                // reuse: dy
                    uv[jj] = ZOH ? uv[jj] : mul2(dt, uv[jj]);   // reuse: delta*u | u
                }
#pragma unroll
                for (int jj = 0; jj < TC / 2; ++jj) {
                    const int e = (2 * jj + ep) * CW + ce;
                    *reinterpret_cast<float2*>(Pd + e) = xr[jj];
                    *reinterpret_cast<float2*>(Pbs + e) = uv[jj];
                    *reinterpret_cast<float2*>(Pdy + e) = go[jj];
                    *reinterpret_cast<float2*>(Psdr + e) = sxv[jj];
                    if (GATE) *reinterpret_cast<float2*>(Psz + e) = zv[jj];
                }
            } else {
                // loads, math and stores in separate passes, so that the steps'
                // independent chains overlap (stores could alias later loads)
                constexpr int NJ = TC / SPL;
                float uvA[NJ], xrA[NJ], goA[NJ], zvA[NJ];
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const int j = SPL * jj + pj;
                    uvA[jj] = Act<T>::to_f(tu[j * CW + pc]);
                    xrA[jj] = Act<T>::to_f(tr[j * CW + pc]);
                    goA[jj] = Act<T>::to_f(tg[j * CW + pc]);
                    zvA[jj] = GATE ? Act<T>::to_f(tz[j * CW + pc]) : 0.0f;
                }
                float sxA[NJ];
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    float dt, sx, dy = goA[jj];
                    if (GATE) {
                        float sz;
                        softplus_sig_xz(xrA[jj], zvA[jj], dt, sx, sz);
                        dy = goA[jj] * zvA[jj] * sz;
                        zvA[jj] = sz;                           // reuse: sigmoid(z)
                    } else {
                        softplus_sig_x(xrA[jj], dt, sx);
                    }
                    sxA[jj] = sx;
                    xrA[jj] = dt;                               // reuse: delta
                    goA[jj] = dy;                               // reuse: dy
                    uvA[jj] = ZOH ? uvA[jj] : dt * uvA[jj];     // reuse: delta*u | u
                }
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const int j = SPL * jj + pj;
                    Pd[j * CW + pc] = xrA[jj];
                    Pbs[j * CW + pc] = uvA[jj];
                    Pdy[j * CW + pc] = goA[jj];
                    Psdr[j * CW + pc] = sxA[jj];
                    if (GATE) Psz[j * CW + pc] = zvA[jj];
                }
            }
            __syncwarp();

            // ---- pass B: h from the checkpoint, a_t h_{t-1} kept in registers;
            //      dC partials (over this lane's channels) to pbuf.
            float2 ah[TC][CPL][NS / 2];
            {
                float2 h[CPL][NS / 2];
#pragma unroll
                for (int i = 0; i < CPL; ++i)
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p)
                        h[i][p] = kc > 0 ? make_float2(ck[(ng * NS + 2 * p) * CW + cbase + i],
                                                       ck[(ng * NS + 2 * p + 1) * CW + cbase + i])
                                         : make_float2(0.f, 0.f);
                // a step's inputs are loaded one step ahead: a partial-sum store
                // could alias them, so they could not move above it otherwise
                float dlN[CPL], bsN[CPL], dyN[CPL];
                float2 BN[NS / 2];
                auto load_b = [&](int j) {
                    ld_cpl<CPL>(Pd + j * CW + cbase, dlN);
                    ld_cpl<CPL>(Pbs + j * CW + cbase, bsN);
                    ld_cpl<CPL>(Pdy + j * CW + cbase, dyN);
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p)
                        BN[p] = *reinterpret_cast<const float2*>(Bf + j * NT + ng * NS + 2 * p);
                };
                load_b(0);
#pragma unroll
                for (int j = 0; j < TC; ++j) {
                    float dlA[CPL], bsA[CPL], dyA[CPL];
                    float2 Bv[NS / 2];
#pragma unroll
                    for (int i = 0; i < CPL; ++i) {
                        dlA[i] = dlN[i];
                        bsA[i] = bsN[i];
                        dyA[i] = dyN[i];
                    }
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p) Bv[p] = BN[p];
                    if (j + 1 < TC) load_b(j + 1);
                    float2 dC[NS / 2];
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p) dC[p] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < CPL; ++i) {
#pragma unroll
                        for (int p = 0; p < NS / 2; ++p) {
                            const float2 x = mul2(f2(dlA[i]), A2r[i][p]);
                            const float2 av = make_float2(ex2(x.x), ex2(x.y));
                            const float2 ahv = mul2(av, h[i][p]);
                            float2 bu = f2(bsA[i]);
                            if (!ZOH) {
                                h[i][p] = fma2(bu, Bv[p], ahv);
                            } else {
                                const float xn0 = x.x * kLn2, xn1 = x.y * kLn2;
                                const float cf0 = fabsf(xn0) < 0.5f ? dlA[i] * phi1_series(xn0)
                                                                    : (av.x - 1.0f) * iAr[i][p].x;
                                const float cf1 = fabsf(xn1) < 0.5f ? dlA[i] * phi1_series(xn1)
                                                                    : (av.y - 1.0f) * iAr[i][p].y;
                                bu = mul2(mul2(make_float2(cf0, cf1), f2(bsA[i])), Bv[p]);
                                h[i][p] = add2(ahv, bu);
                            }
                            ah[j][i][p] = ahv;
                            dC[p] = fma2(f2(dyA[i]), h[i][p], dC[p]);
                        }
                    }
                    store_partial(j, dC);
                    if (j % PR == PR - 1) flush(NT, t0 + j + 1 - PR, jmax - (j + 1 - PR));
                }
            }

            // ---- reverse pass: g_t = C_t dy_t + a_{t+1} g_{t+1}; state sums to
            //      shared partials, dB partials to pbuf.
            unpark();
            __syncwarp();
            {
                float2 an[CPL][NS / 2];
#pragma unroll
                for (int i = 0; i < CPL; ++i)
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p) {
                        const float2 x = mul2(f2(dl_next[i]), A2r[i][p]);
                        an[i][p] = make_float2(ex2(x.x), ex2(x.y));
                    }
                // inputs one step ahead (see pass B)
                float dlN[CPL], bsN[CPL], dyN[CPL];
                float2 BN[NS / 2], CN[NS / 2];
                auto load_r = [&](int j) {
                    ld_cpl<CPL>(Pd + j * CW + cbase, dlN);
                    ld_cpl<CPL>(Pbs + j * CW + cbase, bsN);
                    ld_cpl<CPL>(Pdy + j * CW + cbase, dyN);
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p) {
                        BN[p] = *reinterpret_cast<const float2*>(Bf + j * NT + ng * NS + 2 * p);
                        CN[p] = *reinterpret_cast<const float2*>(Cf + j * NT + ng * NS + 2 * p);
                    }
                };
                load_r(TC - 1);
#pragma unroll
                for (int j = TC - 1; j >= 0; --j) {
                    float dlA[CPL], bsA[CPL], dyA[CPL];
                    float2 Bv[NS / 2], Cv[NS / 2];
#pragma unroll
                    for (int i = 0; i < CPL; ++i) {
                        dlA[i] = dlN[i];
                        bsA[i] = bsN[i];
                        dyA[i] = dyN[i];
                    }
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p) {
                        Bv[p] = BN[p];
                        Cv[p] = CN[p];
                    }
                    if (j > 0) load_r(j - 1);
                    float2 dB[NS / 2];
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p) dB[p] = make_float2(0.f, 0.f);
                    float sums[NQN][CPL];
#pragma unroll
                    for (int i = 0; i < CPL; ++i) {
                        float2 Sg = make_float2(0.f, 0.f), Eg = make_float2(0.f, 0.f);
                        float2 Sa = make_float2(0.f, 0.f);
#pragma unroll
                        for (int p = 0; p < NS / 2; ++p) {
                            const float2 A2p = A2r[i][p];
                            // g_t = C_t dy_t + a_{t+1} g_{t+1}
                            const float2 gv = fma2(an[i][p], g[i][p], mul2(Cv[p], f2(dyA[i])));
                            g[i][p] = gv;
                            const float2 q = mul2(gv, ah[j][i][p]);        // g a_t h_{t-1}
                            Eg = fma2(A2p, q, Eg);
                            const float2 x = mul2(f2(dlA[i]), A2p);
                            const float2 av = make_float2(ex2(x.x), ex2(x.y));   // a_t
                            float2 dAv = dA[i][p];
                            if (!ZOH) {
                                dAv = fma2(f2(dlA[i]), q, dAv);
                                Sg = fma2(gv, Bv[p], Sg);
                                dB[p] = fma2(f2(bsA[i]), gv, dB[p]);
                            } else {
                                const float dt = dlA[i], uv = bsA[i];
                                float cf[2], dcf[2];
#pragma unroll
                                for (int ee = 0; ee < 2; ++ee) {
                                    const float xn = (ee ? x.y : x.x) * kLn2;
                                    const float ae = ee ? av.y : av.x;
                                    const float ia = ee ? iAr[i][p].y : iAr[i][p].x;
                                    const bool small = fabsf(xn) < 0.5f;
                                    cf[ee] = small ? dt * phi1_series(xn) : (ae - 1.0f) * ia;
                                    dcf[ee] = small ? dt * dt * phi2_series(xn)
                                                    : (xn * ae - (ae - 1.0f)) * ia * ia;
                                }
                                const float2 gB = mul2(gv, Bv[p]);
                                dAv = fma2(f2(dt), q, fma2(mul2(gB, f2(uv)), make_float2(dcf[0], dcf[1]), dAv));
                                Sg = fma2(gB, make_float2(cf[0], cf[1]), Sg);
                                Sa = fma2(gB, av, Sa);
                                dB[p] = fma2(mul2(f2(uv), make_float2(cf[0], cf[1])), gv, dB[p]);
                            }
                            dA[i][p] = dAv;
                            an[i][p] = av;
                        }
                        sums[0][i] = Sg.x + Sg.y;
                        sums[1][i] = Eg.x + Eg.y;
                        if (ZOH) sums[NQN - 1][i] = Sa.x + Sa.y;
                    }
#pragma unroll
                    for (int qn = 0; qn < NQN; ++qn)
                        st_cpl<CPL>(part + ((j * NQN + qn) * 4 + ng) * CW + part_col(cbase, ng), sums[qn]);
                    store_partial(j, dB);
                    if (j % PR == 0) flush(0, t0 + j, jmax - j);
                }
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < CPL; ++i) dl_next[i] = Pd[cbase + i];   // delta of step t0
        }
        __syncwarp();

        if (ok) {
            // ---- epilogue: finish du, ddelta_raw, dz, dD.  32-channel CTAs:
            //      lane = (step parity, channel pair), paired loads and
            //      stores and f32x2 arithmetic; 16-channel CTAs: lane =
            //      (channel, step parity).
            if constexpr (CW == 32) {
#pragma unroll 1
                for (int jb = 0; jb < TC / 2; jb += 2) {
                    float2 Sg[2], Eg[2], Sa[2], uv[2], sx[2], dt[2], dy[2], sz[2], zv[2], go[2], yv[2];
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int j = 2 * (jb + jj) + ep;
                        float2 sm[NQN];
#pragma unroll
                        for (int qn = 0; qn < NQN; ++qn) {
                            // the 4 state groups' sums of both channels (a
                            // pair never wraps around the rotated row)
                            const float* pp = part + (j * NQN + qn) * 4 * CW;
                            float2 v[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                v[k] = *reinterpret_cast<const float2*>(pp + k * CW + part_col(ec - c0, k));
                            sm[qn] = add2(add2(v[0], v[1]), add2(v[2], v[3]));
                        }
                        Sg[jj] = sm[0];
                        Eg[jj] = mul2(sm[1], f2(kLn2));
                        Sa[jj] = sm[NQN - 1];
                        const int e = j * CW + (ec - c0);
                        uv[jj] = ActPair<T>::load(tu + e);
                        sx[jj] = *reinterpret_cast<const float2*>(Psdr + e);
                        dt[jj] = *reinterpret_cast<const float2*>(Pd + e);
                        dy[jj] = *reinterpret_cast<const float2*>(Pdy + e);
                        if (GATE) {
                            sz[jj] = *reinterpret_cast<const float2*>(Psz + e);
                            zv[jj] = ActPair<T>::load(tz + e);
                            go[jj] = ActPair<T>::load(tg + e);
                            yv[jj] = ActPair<T>::load(ty + e);
                        }
                    }
                    float2 duO[2], ddO[2], dzO[2];
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int j = 2 * (jb + jj) + ep;
                        duO[jj] = ZOH ? fma2(eD, dy[jj], Sg[jj]) : fma2(dt[jj], Sg[jj], mul2(eD, dy[jj]));
                        ddO[jj] = mul2(fma2(uv[jj], ZOH ? Sa[jj] : Sg[jj], Eg[jj]), sx[jj]);
                        if (j < jmax) eDD = fma2(dy[jj], uv[jj], eDD);
                        if (GATE) {
                            // dout y sigmoid(z) (1 + z (1 - sigmoid(z)))
                            const float2 om = fma2(sz[jj], f2(-1.0f), f2(1.0f));
                            dzO[jj] = mul2(mul2(mul2(go[jj], yv[jj]), sz[jj]), fma2(zv[jj], om, f2(1.0f)));
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int j = 2 * (jb + jj) + ep;
                        if (j < jmax && eok0) {
                            const size_t r = row0 + t0 + j;
                            if (pair_st) {
                                ActPair<T>::store(dup + r * a.ld_du + ec, duO[jj]);
                                ActPair<T>::store(ddp + r * a.ld_ddelta + ec, ddO[jj]);
                                if (GATE) ActPair<T>::store(dzp + r * a.ld_dz + ec, dzO[jj]);
                            } else {
                                dup[r * a.ld_du + ec] = Act<T>::from_f(duO[jj].x);
                                ddp[r * a.ld_ddelta + ec] = Act<T>::from_f(ddO[jj].x);
                                if (GATE) dzp[r * a.ld_dz + ec] = Act<T>::from_f(dzO[jj].x);
                                if (eok1) {
                                    dup[r * a.ld_du + ec + 1] = Act<T>::from_f(duO[jj].y);
                                    ddp[r * a.ld_ddelta + ec + 1] = Act<T>::from_f(ddO[jj].y);
                                    if (GATE) dzp[r * a.ld_dz + ec + 1] = Act<T>::from_f(dzO[jj].y);
                                }
                            }
                        }
                    }
                }
            } else if (lane_ok) {
                // loads, math and stores in separate passes (see the prologue),
                // two steps at a time for 32-channel CTAs (register pressure)
                constexpr int NJALL = TC / SPL;
                constexpr int NJ = (CW == 32) ? 2 : NJALL;   // steps per load/compute/store block
#pragma unroll 1
                for (int jb = 0; jb < NJALL; jb += NJ) {
                float Sg[NJ], Eg[NJ], Sa[NJ], uvA[NJ], sxA[NJ], dtA[NJ], dyA2[NJ], zvA[NJ], szA[NJ], goA[NJ],
                    yvA[NJ];
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const int j = SPL * (jb + jj) + pj;
                    float sm[NQN];
#pragma unroll
                    for (int qn = 0; qn < NQN; ++qn) {
                        // the 4 state groups' sums; a step-phase-1 lane reads
                        // them in the order 1,0,3,2 (other banks, same sum)
                        const float* pp = part + (j * NQN + qn) * 4 * CW;
                        float v[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int kk = k ^ pj;
                            v[k] = pp[kk * CW + part_col(pc, kk)];
                        }
                        sm[qn] = (v[0] + v[1]) + (v[2] + v[3]);
                    }
                    Sg[jj] = sm[0];
                    Eg[jj] = sm[1] * kLn2;
                    Sa[jj] = sm[NQN - 1];
                    uvA[jj] = Act<T>::to_f(tu[j * CW + pc]);
                    sxA[jj] = Psdr[j * CW + pc];
                    dtA[jj] = Pd[j * CW + pc];
                    dyA2[jj] = Pdy[j * CW + pc];
                    if (GATE) {
                        szA[jj] = Psz[j * CW + pc];
                        zvA[jj] = Act<T>::to_f(tz[j * CW + pc]);
                        goA[jj] = Act<T>::to_f(tg[j * CW + pc]);
                        yvA[jj] = Act<T>::to_f(ty[j * CW + pc]);
                    }
                }
                float duO[NJ], ddO[NJ], dzO[NJ];
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const int j = SPL * (jb + jj) + pj;
                    duO[jj] = ZOH ? fmaf(Dd, dyA2[jj], Sg[jj]) : fmaf(dtA[jj], Sg[jj], Dd * dyA2[jj]);
                    ddO[jj] = fmaf(uvA[jj], ZOH ? Sa[jj] : Sg[jj], Eg[jj]) * sxA[jj];
                    if (j < jmax) dD_acc = fmaf(dyA2[jj], uvA[jj], dD_acc);
                    if (GATE) {
                        const float sz = szA[jj];
                        dzO[jj] = goA[jj] * yvA[jj] * sz * (1.0f + zvA[jj] * (1.0f - sz));
                    }
                }
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const int j = SPL * (jb + jj) + pj;
                    if (j < jmax) {
                        const size_t r = row0 + t0 + j;
                        dup[r * a.ld_du + dch] = Act<T>::from_f(duO[jj]);
                        ddp[r * a.ld_ddelta + dch] = Act<T>::from_f(ddO[jj]);
                        if (GATE) dzp[r * a.ld_dz + dch] = Act<T>::from_f(dzO[jj]);
                    }
                }
            }
            }
            __syncwarp();
            park();
        }

        // ---- release this TMA stage
        __syncwarp();
        if (lane == 0 && ok && it + S < nit) issue(it + S);
    }

    if (lane == 0 && !ok) {
        for (int it = waited; it < nit && it < waited + S; ++it)
            mbar_wait(&full[it % S], (it / S) & 1, kFaultDrain);
    }
    __syncwarp();
    unpark();
    if (ok) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int d = c0 + cbase + i;
            if (d < Dn) {
#pragma unroll
                for (int p = 0; p < NS / 2; ++p) {
                    float* dst = a.ws_dA + (plane_b * Dn + d) * NT + ng * NS + 2 * p;
                    dst[0] = dA[i][p].x;
                    dst[1] = dA[i][p].y;
                }
            }
        }
        if constexpr (CW == 32) {
            // the two step-parity lanes of a channel pair each hold half of its dD sums
            const float ox = __shfl_xor_sync(0xffffffffu, eDD.x, 16);
            const float oy = __shfl_xor_sync(0xffffffffu, eDD.y, 16);
            if (ep == 0 && eok0) a.ws_dD[plane_b * Dn + ec] = eDD.x + ox;
            if (ep == 0 && eok1) a.ws_dD[plane_b * Dn + ec + 1] = eDD.y + oy;
        } else {
            // the two step-phase lanes of a channel each hold half of its dD sum
            const float dD_other = __shfl_xor_sync(0xffffffffu, dD_acc, 16);
            if (lane_ok && pj == 0) a.ws_dD[plane_b * Dn + dch] = dD_acc + dD_other;
        }
    }
}

// Combine of the backward's time segments: one thread per (batch row, state,
// channel) walks the segments last to first and writes the carry (true dL/dh
// and delta at the first step of the next segment) of every segment but the
// last.
template <int NT>
__global__ void scan_bwd_combine_kernel(const ScanBwdArgs a) {
    const size_t total = static_cast<size_t>(a.batch) * NT * a.dinner;
    const size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    if (i >= total) return;
    const int d = static_cast<int>(i % a.dinner);
    const int n = static_cast<int>((i / a.dinner) % NT);
    const int b = static_cast<int>(i / (static_cast<size_t>(a.dinner) * NT));
    const float A2 = n < a.dstate ? a2_from_alog(a.A_log[static_cast<size_t>(d) * a.dstate + n]) : 0.0f;
    float carry = 0.0f;
    for (int s = a.nseg - 1; s >= 1; --s) {
        const size_t pb = static_cast<size_t>(b) * a.nseg + s;
        float gstart = a.seg_g[(pb * NT + n) * a.dinner + d];
        if (s + 1 < a.nseg) {
            const float P = ex2(A2 * (a.seg_ds[pb * a.dinner + d] + a.seg_d0[(pb + 1) * a.dinner + d]));
            gstart = fmaf(P, carry, gstart);
        }
        a.carry_g[((pb - 1) * NT + n) * a.dinner + d] = gstart;
        if (n == 0) a.carry_dl[(pb - 1) * a.dinner + d] = a.seg_d0[pb * a.dinner + d];
        carry = gstart;
    }
}

// dB, dC: sum of the per-CTA-column planes; dA_log = A * sum_b dA inside the
// clamp (exactly 0 at or beyond it); dD = sum_b dD.
__global__ void scan_reduce_kernel(const ScanReduceArgs a) {
    const size_t M = static_cast<size_t>(a.batch) * a.seqlen;
    const size_t nBC = M * a.dstate;
    const size_t nA = static_cast<size_t>(a.dinner) * a.dstate;
    const size_t total = nBC + nA + (a.dD ? a.dinner : 0);
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        if (i < nBC) {
            const size_t r = i / a.dstate;
            const int n = static_cast<int>(i % a.dstate);
            float sb = 0.0f, sc = 0.0f;
            for (int p = 0; p < a.ncl; ++p) {
                const float* src = a.ws_bc + (static_cast<size_t>(p) * M + r) * 2 * a.nt;
                sb += src[n];
                sc += src[a.nt + n];
            }
            if (a.is_bf16) {
                static_cast<__nv_bfloat16*>(a.dB)[r * a.ld_dB + n] = __float2bfloat16_rn(sb);
                static_cast<__nv_bfloat16*>(a.dC)[r * a.ld_dC + n] = __float2bfloat16_rn(sc);
            } else {
                static_cast<float*>(a.dB)[r * a.ld_dB + n] = sb;
                static_cast<float*>(a.dC)[r * a.ld_dC + n] = sc;
            }
        } else if (i < nBC + nA) {
            const size_t k = i - nBC;
            const int d = static_cast<int>(k / a.dstate), n = static_cast<int>(k % a.dstate);
            const float al = a.A_log[k];
            float v = 0.0f;
            if (al > kALogLo && al < kALogHi) {
                float s = 0.0f;
                for (int bb = 0; bb < a.nb_sum; ++bb)
                    s += a.ws_dA[(static_cast<size_t>(bb) * a.dinner + d) * a.nt + n];
                v = s * -expf(al);
            }
            a.dA_log[k] = v;
        } else {
            const int d = static_cast<int>(i - nBC - nA);
            float s = 0.0f;
            for (int bb = 0; bb < a.nb_sum; ++bb) s += a.ws_dD[static_cast<size_t>(bb) * a.dinner + d];
            a.dD[d] = s;
        }
    }
}


template <typename T, int NT, int DISC, bool GATE, int CW>
static cudaError_t launch_bwd_cw(const BwdMaps& maps, const ScanBwdArgs& a, cudaStream_t st) {
    const size_t smem = bwd_smem_bytes<T, NT, DISC, GATE, CW>();
    cudaError_t e;
    if constexpr (CW == 16) {
        if (a.nseg > 1 && a.nseg <= kBwdChunkWarps) {
            // the segments as the warps of one CTA per (channel tile, batch row),
            // when those CTAs all fit at once
            auto kc = scan_bwd_kernel<T, NT, DISC, GATE, CW, true>;
            const size_t wb = (smem + 127) / 128 * 128;
            auto bytes = [&](int nw) {
                return nw * wb + static_cast<size_t>(nw) * (NT * CW + 2 * CW + (NT + 1) * CW) * sizeof(float);
            };
            e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(bytes(kBwdChunkWarps)));
            if (e != cudaSuccess) return e;
            int dev = 0, nsm = 0, per_sm = 0;
            e = cudaGetDevice(&dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kc, 32 * a.nseg, bytes(a.nseg));
            if (e != cudaSuccess) return e;
            if (static_cast<long long>(a.ncl) * a.batch <= static_cast<long long>(nsm) * per_sm) {
                kc<<<dim3(static_cast<unsigned>(a.ncl), static_cast<unsigned>(a.batch), 1), 32 * a.nseg,
                     bytes(a.nseg), st>>>(maps, a);
                return cudaGetLastError();
            }
        }
    }
    auto kern = scan_bwd_kernel<T, NT, DISC, GATE, CW>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (a.nseg > 1) {
        // segment pass (segments 1 .. nseg-1), then the combine of the carries
        constexpr int NTEN1 = GATE ? 3 : 2;
        const size_t sm1 = kBwdStages * (NTEN1 * kChunk * CW + kChunk * NT) * sizeof(T) +
                           kChunk * NT * sizeof(float) + kBwdStages * sizeof(uint64_t);
        auto k1 = scan_bwd_segsum_kernel<T, NT, GATE, CW>;
        e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm1));
        if (e != cudaSuccess) return e;
        k1<<<dim3(static_cast<unsigned>(a.ncl), static_cast<unsigned>(a.batch),
                  static_cast<unsigned>(a.nseg - 1)), 32, sm1, st>>>(maps, a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const size_t total = static_cast<size_t>(a.batch) * NT * a.dinner;
        scan_bwd_combine_kernel<NT><<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    kern<<<dim3(static_cast<unsigned>(a.ncl), static_cast<unsigned>(a.batch), static_cast<unsigned>(a.nseg)),
           32, smem, st>>>(maps, a);
    return cudaGetLastError();
}

template <typename T, int NT, int DISC, bool GATE>
static cudaError_t launch_bwd_t(const BwdMaps& maps, const ScanBwdArgs& a, cudaStream_t st) {
    return a.cw == 32 ? launch_bwd_cw<T, NT, DISC, GATE, 32>(maps, a, st)
                      : launch_bwd_cw<T, NT, DISC, GATE, 16>(maps, a, st);
}

template <typename T, int NT>
static cudaError_t launch_bwd_nt(int disc, bool gate, const BwdMaps& m, const ScanBwdArgs& a,
                                 cudaStream_t st) {
    if (disc == 0)
        return gate ? launch_bwd_t<T, NT, 0, true>(m, a, st) : launch_bwd_t<T, NT, 0, false>(m, a, st);
    return gate ? launch_bwd_t<T, NT, 1, true>(m, a, st) : launch_bwd_t<T, NT, 1, false>(m, a, st);
}

cudaError_t launch_scan_bwd(int dtype, int nt, int disc, bool gate, const BwdMaps& maps,
                            const ScanBwdArgs& a, cudaStream_t stream) {
    if (dtype == 0)
        return nt == 8 ? launch_bwd_nt<float, 8>(disc, gate, maps, a, stream)
                       : launch_bwd_nt<float, 16>(disc, gate, maps, a, stream);
    return nt == 8 ? launch_bwd_nt<__nv_bfloat16, 8>(disc, gate, maps, a, stream)
                   : launch_bwd_nt<__nv_bfloat16, 16>(disc, gate, maps, a, stream);
}

cudaError_t read_clear_fault_bwd(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_ssm_fault, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_ssm_fault, &zero, sizeof(unsigned));
}

cudaError_t launch_scan_reduce(const ScanReduceArgs& a, cudaStream_t stream) {
    const size_t M = static_cast<size_t>(a.batch) * a.seqlen;
    const size_t total = M * a.dstate + static_cast<size_t>(a.dinner) * a.dstate + a.dinner;
    if (total == 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>(std::min<size_t>((total + 255) / 256, 152 * 16));
    scan_reduce_kernel<<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ssm

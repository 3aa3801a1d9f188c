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
// Design (GB300): the forward saved h every kChunk (= 8) steps.  A CTA owns
// 32 channels of one batch row and walks the chunks last to first; its NT/8
// warps split the states, so the B8 x D4096 problem runs 2048 warps (about 13
// per SM) with 8 chains per lane.  For each chunk a prologue computes the
// per-(step, channel) scalars once for the CTA (delta, delta*u, dy and the two
// sigmoids, shared memory); pass B recomputes h forward from the checkpoint,
// keeping a_t h_{t-1} in registers; the reverse pass runs g over the chunk in
// two halves, each followed by the epilogue of its steps (du, ddelta_raw, dz,
// dD).  Sums over states leave as per-group partials through shared memory;
// sums over channels (dB, dC) as per-channel-pair partials that the warp adds
// into the CTA's partial plane (no inter-CTA synchronisation; an earlier
// cluster/DSMEM exchange paid a cluster-scope release fence per chunk).
// scan_reduce_kernel adds the planes and finishes dA_log and dD.
#include <algorithm>

#include "scan_args.cuh"
#include "ssm_common.cuh"

namespace ssm {

// Two adjacent activation elements as fp32 (loads from a TMA tile, stores to
// global memory): one 32-bit access for bf16, one 64-bit access for fp32.
template <typename T> struct Pair;
template <> struct Pair<float> {
    static __device__ __forceinline__ float2 ld(const float* p) {
        return *reinterpret_cast<const float2*>(p);
    }
    static __device__ __forceinline__ void st(float* p, float2 v) {
        *reinterpret_cast<float2*>(p) = v;
    }
};
template <> struct Pair<__nv_bfloat16> {
    static __device__ __forceinline__ float2 ld(const __nv_bfloat16* p) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, float2 v) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __float22bfloat162_rn(v);
    }
};

// delta = softplus(x) together with sigmoid(x) and sigmoid(z), from
// e = exp(-|x|), ez = exp(-z) and one reciprocal r = 1/((2+e)(1+ez)(1+e)):
// 1/(2+e) = r(1+ez)(1+e), sigmoid(z) = 1/(1+ez) = r(2+e)(1+e) and
// 1/(1+e) = r(2+e)(1+ez).  ez is capped at 2^100 (see softplus_sigmoid).
__device__ __forceinline__ void softplus_sig_xz(float x, float z, float& dt, float& sdr, float& sz) {
    const float e = ex2(-fabsf(x) * kLog2e);
    const float ez = ex2(fminf(-z * kLog2e, 100.0f));
    const float a = 2.0f + e, b = 1.0f + ez, c = 1.0f + e;
    const float ab = a * b;
    const float r = rcp(ab * c);
    const float inv_c = r * ab;
    sz = r * (a * c);
    dt = fmaxf(x, 0.0f) + log1p_unit(e, r * (b * c));
    sdr = x >= 0.0f ? inv_c : e * inv_c;
}
// The same without a gate: r = 1/((2+e)(1+e)).
__device__ __forceinline__ void softplus_sig_x(float x, float& dt, float& sdr) {
    const float e = ex2(-fabsf(x) * kLog2e);
    const float a = 2.0f + e, c = 1.0f + e;
    const float r = rcp(a * c);
    const float inv_c = r * a;
    dt = fmaxf(x, 0.0f) + log1p_unit(e, r * c);
    sdr = x >= 0.0f ? inv_c : e * inv_c;
}

// ZOH coefficient beta/B = (exp(delta A) - 1)/A = delta phi1(delta A) and its
// A-derivative delta^2 phi2(delta A), from x2 = delta A log2(e) and a = exp(delta A).
__device__ __forceinline__ float zoh_cf(float x2, float a, float dt, float inv_a) {
    const float xn = x2 * kLn2;
    return fabsf(xn) < 0.5f ? dt * phi1_series(xn) : (a - 1.0f) * inv_a;
}
__device__ __forceinline__ float zoh_dcf(float x2, float a, float dt, float inv_a) {
    const float xn = x2 * kLn2;
    return fabsf(xn) < 0.5f ? dt * dt * phi2_series(xn) : (xn * a - (a - 1.0f)) * inv_a * inv_a;
}

// A CTA owns 32 channels of one batch row for its time segment; its NT/8
// warps split the states (warp w: states 8w .. 8w+7).  Lane (pi, sq) of a
// warp owns channels 2pi, 2pi+1 and states 8w+4sq .. +3: 8 chains, held as
// state pairs in packed f32x2 registers.  The per-(step, channel) scalars
// (delta, delta*u, dy) are stored duplicated in shared memory, so one 16-byte
// load gives the broadcast pairs of both channels.  Sums over the states of a
// (step, channel) (sum g B, sum g A a h) leave as per-group partials (NT/4
// groups) that the epilogue adds; sums over the channels of a (step, state)
// (dB, dC) leave as per-channel-pair partials that the warp adds and writes to
// the CTA's partial plane.
template <typename T, int NT, int DISC, bool GATE>
__global__ void __launch_bounds__(4 * NT, DISC == 0 ? (NT == 16 ? 7 : 14) : (NT == 16 ? 6 : 12))
scan_bwd_kernel(const __grid_constant__ BwdMaps maps, const ScanBwdArgs a) {
    constexpr int TC = kChunk;
    constexpr int S = kBwdStages;
    constexpr int CW = kBwdChannels;
    constexpr int NW = NT / 8;                  // warps
    constexpr int NTH = 32 * NW;
    constexpr int NTEN = GATE ? 5 : 3;          // u, delta_raw, dout, [z, y]
    constexpr int TILE = TC * CW;
    constexpr int BCT = TC * NT;                // elements per B or C tile
    constexpr int STAGE = NTEN * TILE + 2 * BCT;
    constexpr uint32_t kActBytes = NTEN * TILE * sizeof(T);
    constexpr uint32_t kBCBytes = 2 * BCT * sizeof(T);
    constexpr uint32_t kCkBytes = NT * CW * sizeof(float);
    constexpr bool ZOH = DISC == 1;
    constexpr int HS = TC / 2;                  // steps per half chunk (flush / epilogue)
    constexpr int NG = 2 * NW;                  // state groups of a (step, channel)
    constexpr int NQ = ZOH ? 3 : 2;             // state sums per (step, channel)
    constexpr int PPJ = 16 * 8 + 8;             // padded partial row: 16 channel pairs x 8 states
    constexpr int PART = HS * NQ * NG * CW;     // floats of the state-sum partials
    constexpr int PBUF = NW * HS * PPJ;         // floats of one dB or dC partial buffer
    constexpr int PROW = PART > PBUF ? PART : PBUF;
    constexpr int PI = 128 / NTH;               // prologue pair-items per thread and chunk
    constexpr int EI = 64 / NTH;                // epilogue pair-items per thread and half
    constexpr int kSu = ZOH ? 2 : 0;            // the state sum that multiplies u in ddelta
    static_assert((STAGE * sizeof(T)) % 128 == 0, "stages stay 128-byte aligned");
    static_assert(TC == 8 && (NT == 8 || NT == 16), "lane layout below");

    extern __shared__ __align__(128) unsigned char smem[];
    T* tiles = reinterpret_cast<T*>(smem);                                   // [S][STAGE]
    float* cks = reinterpret_cast<float*>(smem + S * STAGE * sizeof(T));    // [S][NT][CW]
    float* bcs = cks + S * NT * CW;             // [TC][NT] B | [TC][NT] C (fp32)
    float* Pd = bcs + 2 * BCT;                  // [TC][CW][2] delta, each value twice
    float* Pbu = Pd + 2 * TILE;                 // [TC][CW][2] delta*u (Euler) | u (ZOH)
    float* Pdy = Pbu + 2 * TILE;                // [TC][CW][2] dy = dout * silu(z)
    float* Psdr = Pdy + 2 * TILE;               // [TC][CW] sigmoid(delta_raw)
    float* Psz = Psdr + TILE;                   // [TC][CW] sigmoid(z)
    float* part = Psz + TILE;                   // [HS][NQ][NG][CW] state sums; dC partials in pass B
    float* pbufB = part + PROW;                 // [NW][HS][PPJ] dB partials
    uint64_t* full = reinterpret_cast<uint64_t*>(pbufB + PBUF);   // [S]

    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    const int pi = lane & 15, sq = lane >> 4;
    const int cl = 2 * pi;                      // this lane's first channel (local)
    const int n0 = 8 * w + 4 * sq;              // this lane's first state
    const int grp = 2 * w + sq;                 // its state group
    const int cp = tid & 15;                    // channel pair of this thread's pro/epilogue items
    const int c0 = blockIdx.x * CW;
    const int b = blockIdx.y;
    const int L = a.seqlen, N = a.dstate, Dn = a.dinner;
    const int nchunks = (L + TC - 1) / TC;
    const int sg = blockIdx.z;                  // time segment: chunks [kcb, kce), last to first
    const int kcb = sg * a.seg_chunks;
    const int kce = min(nchunks, kcb + a.seg_chunks);
    const int nit = kce - kcb;
    const size_t plane_b = static_cast<size_t>(b) * a.nseg + sg;   // dA / dD plane
    const size_t row0 = static_cast<size_t>(b) * L;

    // per (channel, state pair) constants: A log2(e) (0 on padding) [and 1/A]
    float2 A2[2][2], iA[2][2];
#pragma unroll
    for (int ci = 0; ci < 2; ++ci)
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            float v[2], r[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int d = c0 + cl + ci, n = n0 + 2 * p + e;
                const bool ok = d < Dn && n < N;
                const float A = ok ? a_from_alog(a.A_log[static_cast<size_t>(d) * N + n]) : -1.0f;
                v[e] = ok ? A * kLog2e : 0.0f;
                r[e] = 1.0f / A;
            }
            A2[ci][p] = make_float2(v[0], v[1]);
            iA[ci][p] = make_float2(r[0], r[1]);
        }
    float2 Dp = make_float2(0.0f, 0.0f);   // D of the items' channel pair (D needs only 4-byte alignment)
    if (a.D && c0 + 2 * cp < Dn) Dp = make_float2(a.D[c0 + 2 * cp], a.D[c0 + 2 * cp + 1]);

    const T* Bp = static_cast<const T*>(a.B);
    const T* Cp = static_cast<const T*>(a.C);
    const bool bc_tma = a.bc_tma != 0;
    auto issue = [&](int it) {
        const int kc = kce - 1 - it;
        const int s = it % S;
        T* dst = tiles + s * STAGE;
        mbar_arrive_expect_tx(&full[s], kActBytes + (kc > 0 ? kCkBytes : 0u) + (bc_tma ? kBCBytes : 0u));
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
        if (kc > 0) tma_load_2d(cks + s * NT * CW, &maps.ck, &full[s], c0, (b * a.nck + kc - 1) * NT);
    };
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int it = 0; it < S && it < nit; ++it) issue(it);

    // carries of the reverse recurrence: g = dL/dh after this segment, delta of
    // the step after it
    float2 g[2][2], dA[2][2];
    float dl_next[2] = {0.0f, 0.0f};
#pragma unroll
    for (int ci = 0; ci < 2; ++ci)
#pragma unroll
        for (int p = 0; p < 2; ++p) g[ci][p] = dA[ci][p] = make_float2(0.0f, 0.0f);
    if (sg + 1 < a.nseg) {
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
            const int d = c0 + cl + ci;
            if (d < Dn) {
                dl_next[ci] = a.carry_dl[plane_b * Dn + d];
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const float* cq = a.carry_g + (plane_b * NT + n0 + 2 * p) * Dn + d;
                    g[ci][p] = make_float2(cq[0], cq[Dn]);
                }
            }
        }
    }
    float2 dDacc[EI];
#pragma unroll
    for (int m = 0; m < EI; ++m) dDacc[m] = make_float2(0.0f, 0.0f);

    T* dup = static_cast<T*>(a.du);
    T* ddp = static_cast<T*>(a.ddelta);
    T* dzp = static_cast<T*>(a.dz);
    float* plane = a.ws_bc + static_cast<size_t>(blockIdx.x) * a.batch * L * 2 * NT;

    // Adds the 16 channel-pair partials of every (step, state) of this warp's
    // rows [tf, tf + HS) and writes them to the plane (qoff 0: dB, NT: dC).
    // Lane -> (step jj, state pair sp, half hf of the channel pairs).
    auto flush = [&](const float* pb, int qoff, int tf, int nrows) {
        const int o = lane >> 1, hf = lane & 1;
        const int jj = o >> 2, sp = o & 3;
        const float* rp = pb + jj * PPJ + 2 * sp + 64 * hf;
        float2 acc = *reinterpret_cast<const float2*>(rp);
#pragma unroll
        for (int k = 1; k < 8; ++k) acc = add2(acc, *reinterpret_cast<const float2*>(rp + 8 * k));
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 1);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 1);
        if (hf == 0 && jj < nrows)
            *reinterpret_cast<float2*>(plane + (row0 + tf + jj) * 2 * NT + qoff + 8 * w + 2 * sp) = acc;
    };

    bool ok = true;
    int waited = 0;
    for (int it = 0; it < nit; ++it) {
        const int kc = kce - 1 - it;
        const int t0 = kc * TC;
        const int jmax = min(TC, L - t0);
        const int s = it % S;
        if (ok) ok = mbar_wait(&full[s], (it / S) & 1, kFaultBwdWait);
        ok = __syncthreads_and(ok) != 0;
        if (!ok) break;
        waited = it + 1;

        const T* tu = tiles + s * STAGE;
        const T* tr = tu + TILE;
        const T* tg = tu + 2 * TILE;
        const T* tz = tu + 3 * TILE;
        const T* ty = tu + 4 * TILE;
        const float* ck = cks + s * NT * CW;

        // fp32 B and C of the chunk, [TC][NT] each (states past dstate and
        // steps past seqlen are 0): fp32 TMA tiles in place, bf16 widened.
        const float* Bf;
        {
            const T* Bs = tu + NTEN * TILE;
            if (bc_tma && sizeof(T) == 4) {
                Bf = reinterpret_cast<const float*>(Bs);
            } else if (bc_tma) {
                for (int g8 = tid; g8 < 2 * BCT / 8; g8 += NTH) {
                    const uint4 v = *reinterpret_cast<const uint4*>(Bs + 8 * g8);
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                    float f[8];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        f[2 * q] = __uint_as_float(wv[q] << 16);
                        f[2 * q + 1] = __uint_as_float(wv[q] & 0xffff0000u);
                    }
                    *reinterpret_cast<float4*>(bcs + 8 * g8) = make_float4(f[0], f[1], f[2], f[3]);
                    *reinterpret_cast<float4*>(bcs + 8 * g8 + 4) = make_float4(f[4], f[5], f[6], f[7]);
                }
                Bf = bcs;
            } else {
                for (int e = tid; e < 2 * BCT; e += NTH) {
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
        }
        const float* Cf = Bf + BCT;

        // ---- prologue: per (step, channel pair) delta, delta*u | u, dy and the
        //      two sigmoids.  Past seqlen the tiles are zero: dy = 0 there.
#pragma unroll
        for (int m = 0; m < PI; ++m) {
            const int j = (tid >> 4) + (NTH / 16) * m;
            const int c = 2 * cp;
            const float2 u2 = Pair<T>::ld(tu + j * CW + c);
            const float2 x2 = Pair<T>::ld(tr + j * CW + c);
            const float2 o2 = Pair<T>::ld(tg + j * CW + c);
            float dt[2], sdr[2], sz[2] = {0.0f, 0.0f}, dy[2];
            if (GATE) {
                const float2 z2 = Pair<T>::ld(tz + j * CW + c);
                softplus_sig_xz(x2.x, z2.x, dt[0], sdr[0], sz[0]);
                softplus_sig_xz(x2.y, z2.y, dt[1], sdr[1], sz[1]);
                dy[0] = o2.x * z2.x * sz[0];
                dy[1] = o2.y * z2.y * sz[1];
            } else {
                softplus_sig_x(x2.x, dt[0], sdr[0]);
                softplus_sig_x(x2.y, dt[1], sdr[1]);
                dy[0] = o2.x;
                dy[1] = o2.y;
            }
            const float bu0 = ZOH ? u2.x : dt[0] * u2.x;
            const float bu1 = ZOH ? u2.y : dt[1] * u2.y;
            const int o = (j * CW + c) * 2;
            *reinterpret_cast<float4*>(Pd + o) = make_float4(dt[0], dt[0], dt[1], dt[1]);
            *reinterpret_cast<float4*>(Pbu + o) = make_float4(bu0, bu0, bu1, bu1);
            *reinterpret_cast<float4*>(Pdy + o) = make_float4(dy[0], dy[0], dy[1], dy[1]);
            *reinterpret_cast<float2*>(Psdr + j * CW + c) = make_float2(sdr[0], sdr[1]);
            if (GATE) *reinterpret_cast<float2*>(Psz + j * CW + c) = make_float2(sz[0], sz[1]);
        }
        __syncthreads();

        // ---- pass B: h from the chunk's checkpoint, a_t h_{t-1} kept in
        //      registers; dC partials (over this lane's two channels) flushed
        //      every HS steps through `part`.
        float2 ah[TC][2][2];
        {
            float2 h[2][2];
#pragma unroll
            for (int ci = 0; ci < 2; ++ci)
#pragma unroll
                for (int p = 0; p < 2; ++p)
                    h[ci][p] = kc > 0 ? make_float2(ck[(n0 + 2 * p) * CW + cl + ci],
                                                    ck[(n0 + 2 * p + 1) * CW + cl + ci])
                                      : make_float2(0.0f, 0.0f);
            float* pc = part + w * HS * PPJ;
#pragma unroll
            for (int j = 0; j < TC; ++j) {
                const float4 dl = *reinterpret_cast<const float4*>(Pd + (j * CW + cl) * 2);
                const float4 bu = *reinterpret_cast<const float4*>(Pbu + (j * CW + cl) * 2);
                const float4 dy = *reinterpret_cast<const float4*>(Pdy + (j * CW + cl) * 2);
                const float4 Bq = *reinterpret_cast<const float4*>(Bf + j * NT + n0);
                float2 dC[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
                for (int ci = 0; ci < 2; ++ci) {
                    const float2 dlc = ci ? make_float2(dl.z, dl.w) : make_float2(dl.x, dl.y);
                    const float2 buc = ci ? make_float2(bu.z, bu.w) : make_float2(bu.x, bu.y);
                    const float2 dyc = ci ? make_float2(dy.z, dy.w) : make_float2(dy.x, dy.y);
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const float2 Bv = p ? make_float2(Bq.z, Bq.w) : make_float2(Bq.x, Bq.y);
                        const float2 x = mul2(dlc, A2[ci][p]);
                        const float2 av = make_float2(ex2(x.x), ex2(x.y));
                        const float2 ahv = mul2(av, h[ci][p]);
                        if (!ZOH) {
                            h[ci][p] = fma2(buc, Bv, ahv);
                        } else {
                            const float2 cf = make_float2(zoh_cf(x.x, av.x, dlc.x, iA[ci][p].x),
                                                          zoh_cf(x.y, av.y, dlc.x, iA[ci][p].y));
                            h[ci][p] = fma2(mul2(cf, buc), Bv, ahv);
                        }
                        ah[j][ci][p] = ahv;
                        dC[p] = fma2(dyc, h[ci][p], dC[p]);
                    }
                }
                *reinterpret_cast<float4*>(pc + (j % HS) * PPJ + pi * 8 + 4 * sq) =
                    make_float4(dC[0].x, dC[0].y, dC[1].x, dC[1].y);
                if (j % HS == HS - 1) {
                    __syncwarp();
                    flush(pc, NT, t0 + j + 1 - HS, jmax - (j + 1 - HS));
                    __syncwarp();
                }
            }
        }
        __syncthreads();   // `part` changes role: state sums from here on

        // ---- reverse pass, in two halves (steps 7..4, then 3..0), each followed
        //      by the dB flush and the epilogue of its steps.
        float2 an[2][2];                        // a of the step after the current one
#pragma unroll
        for (int ci = 0; ci < 2; ++ci)
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const float2 x = mul2(f2(dl_next[ci]), A2[ci][p]);
                an[ci][p] = make_float2(ex2(x.x), ex2(x.y));
            }
#pragma unroll
        for (int hb = 1; hb >= 0; --hb) {
            const int jb = hb * HS;
#pragma unroll
            for (int jl = HS - 1; jl >= 0; --jl) {
                const int j = jb + jl;
                const float4 dl = *reinterpret_cast<const float4*>(Pd + (j * CW + cl) * 2);
                const float4 bu = *reinterpret_cast<const float4*>(Pbu + (j * CW + cl) * 2);
                const float4 dy = *reinterpret_cast<const float4*>(Pdy + (j * CW + cl) * 2);
                const float4 Bq = *reinterpret_cast<const float4*>(Bf + j * NT + n0);
                const float4 Cq = *reinterpret_cast<const float4*>(Cf + j * NT + n0);
                float2 dB[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
                float sums[NQ][2];
#pragma unroll
                for (int ci = 0; ci < 2; ++ci) {
                    const float2 dlc = ci ? make_float2(dl.z, dl.w) : make_float2(dl.x, dl.y);
                    const float2 buc = ci ? make_float2(bu.z, bu.w) : make_float2(bu.x, bu.y);
                    const float2 dyc = ci ? make_float2(dy.z, dy.w) : make_float2(dy.x, dy.y);
                    float2 Sg = make_float2(0.0f, 0.0f), Eg = Sg, Sa = Sg;
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const float2 Bv = p ? make_float2(Bq.z, Bq.w) : make_float2(Bq.x, Bq.y);
                        const float2 Cv = p ? make_float2(Cq.z, Cq.w) : make_float2(Cq.x, Cq.y);
                        // g_t = C_t dy_t + a_{t+1} g_{t+1}
                        const float2 gv = fma2(an[ci][p], g[ci][p], mul2(Cv, dyc));
                        g[ci][p] = gv;
                        const float2 q = mul2(gv, ah[j][ci][p]);      // g a_t h_{t-1}
                        Eg = fma2(A2[ci][p], q, Eg);
                        const float2 x = mul2(dlc, A2[ci][p]);
                        const float2 av = make_float2(ex2(x.x), ex2(x.y));   // a_t
                        if (!ZOH) {
                            dA[ci][p] = fma2(dlc, q, dA[ci][p]);
                            Sg = fma2(gv, Bv, Sg);
                            dB[p] = fma2(buc, gv, dB[p]);
                        } else {
                            const float2 cf = make_float2(zoh_cf(x.x, av.x, dlc.x, iA[ci][p].x),
                                                          zoh_cf(x.y, av.y, dlc.x, iA[ci][p].y));
                            const float2 dcf = make_float2(zoh_dcf(x.x, av.x, dlc.x, iA[ci][p].x),
                                                           zoh_dcf(x.y, av.y, dlc.x, iA[ci][p].y));
                            const float2 gB = mul2(gv, Bv);
                            dA[ci][p] = fma2(dlc, q, fma2(mul2(gB, buc), dcf, dA[ci][p]));
                            Sg = fma2(gB, cf, Sg);
                            Sa = fma2(gB, av, Sa);
                            dB[p] = fma2(mul2(buc, cf), gv, dB[p]);
                        }
                        an[ci][p] = av;
                    }
                    sums[0][ci] = Sg.x + Sg.y;
                    sums[1][ci] = Eg.x + Eg.y;
                    if (ZOH) sums[NQ - 1][ci] = Sa.x + Sa.y;
                }
                float* pp = part + (jl * NQ * NG + grp) * CW + cl;
#pragma unroll
                for (int qn = 0; qn < NQ; ++qn)
                    *reinterpret_cast<float2*>(pp + qn * NG * CW) = make_float2(sums[qn][0], sums[qn][1]);
                *reinterpret_cast<float4*>(pbufB + (w * HS + jl) * PPJ + pi * 8 + 4 * sq) =
                    make_float4(dB[0].x, dB[0].y, dB[1].x, dB[1].y);
            }
            __syncwarp();
            flush(pbufB + w * HS * PPJ, 0, t0 + jb, jmax - jb);
            __syncthreads();   // every warp's state sums of these steps are in `part`

            // ---- epilogue of steps jb .. jb+HS-1 (thread -> step, channel pair):
            //      du, ddelta_raw, dz, dD
#pragma unroll
            for (int m = 0; m < EI; ++m) {
                const int jl = (tid >> 4) + (NTH / 16) * m;
                const int j = jb + jl;
                const int c = 2 * cp;
                const float* pp = part + jl * NQ * NG * CW + c;
                float2 sm[NQ];
#pragma unroll
                for (int qn = 0; qn < NQ; ++qn) {
                    float2 v = *reinterpret_cast<const float2*>(pp + qn * NG * CW);
#pragma unroll
                    for (int gq = 1; gq < NG; ++gq)
                        v = add2(v, *reinterpret_cast<const float2*>(pp + (qn * NG + gq) * CW));
                    sm[qn] = v;
                }
                const float4 dl4 = *reinterpret_cast<const float4*>(Pd + (j * CW + c) * 2);
                const float4 dy4 = *reinterpret_cast<const float4*>(Pdy + (j * CW + c) * 2);
                const float2 dl2 = make_float2(dl4.x, dl4.z), dy2 = make_float2(dy4.x, dy4.z);
                const float2 sdr2 = *reinterpret_cast<const float2*>(Psdr + j * CW + c);
                const float2 u2 = Pair<T>::ld(tu + j * CW + c);
                const float2 du2 = ZOH ? fma2(Dp, dy2, sm[0]) : fma2(dl2, sm[0], mul2(Dp, dy2));
                const float2 dd2 = mul2(fma2(u2, sm[kSu], mul2(sm[1], f2(kLn2))), sdr2);
                float2 dz2 = make_float2(0.0f, 0.0f);
                if (GATE) {
                    const float2 sz2 = *reinterpret_cast<const float2*>(Psz + j * CW + c);
                    const float2 z2 = Pair<T>::ld(tz + j * CW + c);
                    const float2 o2 = Pair<T>::ld(tg + j * CW + c);
                    const float2 y2 = Pair<T>::ld(ty + j * CW + c);
                    const float2 one = f2(1.0f);
                    const float2 t1 = fma2(z2, add2(one, mul2(f2(-1.0f), sz2)), one);   // 1 + z (1 - sz)
                    dz2 = mul2(mul2(mul2(o2, y2), sz2), t1);
                }
                if (j < jmax) {
                    dDacc[m] = fma2(dy2, u2, dDacc[m]);
                    if (c0 + c < Dn) {
                        const size_t r = row0 + t0 + j;
                        Pair<T>::st(dup + r * a.ld_du + c0 + c, du2);
                        Pair<T>::st(ddp + r * a.ld_ddelta + c0 + c, dd2);
                        if (GATE) Pair<T>::st(dzp + r * a.ld_dz + c0 + c, dz2);
                    }
                }
            }
            __syncthreads();   // `part` and the dB rows are reused by the next half
        }
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) dl_next[ci] = Pd[(cl + ci) * 2];   // delta of step t0

        // ---- release this TMA stage
        if (tid == 0 && it + S < nit) issue(it + S);
    }

    if (!ok) {
        // a wait gave up: drain the copies still in flight (bounded) before exit
        if (tid == 0)
            for (int it = waited; it < nit && it < waited + S; ++it)
                mbar_wait(&full[it % S], (it / S) & 1, kFaultDrain);
        return;
    }
#pragma unroll
    for (int ci = 0; ci < 2; ++ci) {
        const int d = c0 + cl + ci;
        if (d < Dn)
            *reinterpret_cast<float4*>(a.ws_dA + (plane_b * Dn + d) * NT + n0) =
                make_float4(dA[ci][0].x, dA[ci][0].y, dA[ci][1].x, dA[ci][1].y);
    }
    // dD: the threads of a channel pair hold the sums over steps jl (mod 4)
    float* red = part;
#pragma unroll
    for (int m = 0; m < EI; ++m)
        *reinterpret_cast<float2*>(red + ((tid >> 4) + (NTH / 16) * m) * CW + 2 * cp) = dDacc[m];
    __syncthreads();
    if (tid < 16) {
        float2 v = *reinterpret_cast<const float2*>(red + 2 * cp);
#pragma unroll
        for (int k = 1; k < HS; ++k) v = add2(v, *reinterpret_cast<const float2*>(red + k * CW + 2 * cp));
        const int d = c0 + 2 * cp;
        if (d < Dn) *reinterpret_cast<float2*>(a.ws_dD + plane_b * Dn + d) = v;
    }
}

// Segment pass of the time-parallel backward: for segment sg >= 1 of batch
// row b, walk its steps last to first with g = 0 after its last step,
//   g_t = C_t dy_t + a_{t+1} g_{t+1},
// and keep g at its first step, the sum of delta over its steps after the
// first, and delta at its first step.  Because the product of a_s over steps
// t0+1 .. t1+1 is exp(A (that sum + delta at t1+1)), the true g at the first
// step of a segment is its zero-carry value plus that product times the true
// g at the first step of the next segment (scan_bwd_combine_kernel).  A lane
// owns NT * CW / 32 states of one channel.
template <typename T, int NT, bool GATE, int CW>
__global__ void __launch_bounds__(32, 1)
scan_bwd_segsum_kernel(const __grid_constant__ BwdMaps maps, const ScanBwdArgs a) {
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

    extern __shared__ __align__(128) unsigned char smem[];
    T* tiles = reinterpret_cast<T*>(smem);                                   // [S][STAGE]
    float* csm = reinterpret_cast<float*>(smem + S * STAGE * sizeof(T));    // [TC][NT] fp32 C
    uint64_t* full = reinterpret_cast<uint64_t*>(csm + BCT);                 // [S]

    const int lane = threadIdx.x;
    const int c = lane % CW, half = lane / CW;
    const int nbase = half * NL;
    const int c0 = blockIdx.x * CW;
    const int b = blockIdx.y;
    const int sg = blockIdx.z + 1;               // segments 1 .. nseg-1
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
    float2 gl[NQ], an[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) gl[q] = an[q] = make_float2(0.0f, 0.0f);
    float dsum = 0.0f, dfirst = 0.0f;

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
    if (active && it == nit) {
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

template <typename T, int NT, int DISC, bool GATE>
static size_t bwd_smem_bytes() {
    constexpr int TC = kChunk, CW = kBwdChannels, NW = NT / 8;
    constexpr int NTEN = GATE ? 5 : 3;
    constexpr int NQ = DISC == 1 ? 3 : 2;
    constexpr int HS = TC / 2, NG = 2 * NW, PPJ = 16 * 8 + 8;
    constexpr int PART = HS * NQ * NG * CW, PBUF = NW * HS * PPJ;
    return kBwdStages * (NTEN * TC * CW + 2 * TC * NT) * sizeof(T)   // activation, B, C tiles
           + kBwdStages * NT * CW * sizeof(float)      // checkpoint tiles
           + 2 * TC * NT * sizeof(float)               // fp32 B | C
           + 3 * 2 * TC * CW * sizeof(float)           // delta, delta*u | u, dy (duplicated)
           + 2 * TC * CW * sizeof(float)               // sigmoid(delta_raw), sigmoid(z)
           + (PART > PBUF ? PART : PBUF) * sizeof(float)   // state sums | dC partials
           + PBUF * sizeof(float)                      // dB partials
           + kBwdStages * sizeof(uint64_t);
}

template <typename T, int NT, int DISC, bool GATE>
static cudaError_t launch_bwd_t(const BwdMaps& maps, const ScanBwdArgs& a, cudaStream_t st) {
    const size_t smem = bwd_smem_bytes<T, NT, DISC, GATE>();
    auto kern = scan_bwd_kernel<T, NT, DISC, GATE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    constexpr int CW = kBwdChannels;
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
           4 * NT, smem, st>>>(maps, a);
    return cudaGetLastError();
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

// scan_args.cuh -- argument blocks and launch constants shared by the C-ABI
// layer (abi.cu) and the selective-scan kernels (scan_fwd.cu, scan_bwd.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

// Scan-state checkpoint spacing: the forward stores h every kChunk steps and
// the backward recomputes h inside each chunk of kChunk steps.
constexpr int kChunk = 8;

// Forward: one lane per channel (all states of it), one warp of 32 channels
// per CTA.
constexpr int kFwdChannels = 32;
constexpr int kFwdTile = 16;    // steps per TMA-staged tile
constexpr int kFwdStages = 4;   // tiles in flight
// Time segments up to this count run as the warps of one CTA, combined in
// shared memory; more segments run as separate CTAs combined in global memory.
constexpr int kFwdChunkWarps = 4;
// Time segments of the forward: one per batch row unless batch x ceil(dinner/32)
// warps leave the 152 SMs with fewer than 2 warps each (measured: at 2.5 warps
// per SM the segment pass costs more than it gains); then enough segments (of
// at least 256 steps) for about 6 warps per SM.
inline int fwd_segments(int batch, int dinner, int seqlen) {
    const long long warps = static_cast<long long>(batch) * ((dinner + 31) / 32);
    if (warps <= 0 || warps >= 152LL * 2) return 1;
    long long g = (152LL * 6 + warps - 1) / warps;
    const long long gmax = seqlen / 256;
    if (g > gmax) g = gmax;
    return g < 1 ? 1 : static_cast<int>(g);
}
// Tiles per segment for g segments, and the resulting segment count.
inline int fwd_seg_tiles(int seqlen, int g) {
    const int ntiles = (seqlen + kFwdTile - 1) / kFwdTile;
    return (ntiles + g - 1) / g;
}

// Backward: one warp per CTA covers 32 or 16 channels x all states (each lane
// owns 4 or 2 channels x dstate/4 states); every CTA writes its own dB/dC
// partial plane.  The 16-channel kernel is held to 128 registers so that 14
// CTAs fit an SM.
constexpr int kBwdStages = 2;
constexpr int kBwdMinBlocks16 = 14;
// Backward time segments up to this count run as the warps of one CTA
// (16-channel tiles), combined in shared memory.
constexpr int kBwdChunkWarps = 4;
// Channels per backward CTA: 32 when 32-channel CTAs already give at least 6
// warps per SM on the 152 SMs of a GB300, else 16 (twice the warps).
inline int bwd_channels(int batch, int dinner) {
    const long long ctas32 = static_cast<long long>(batch) * ((dinner + 31) / 32);
    return ctas32 >= 152LL * 6 ? 32 : 16;
}
// Time segments of the backward: one unless the CTAs of cw channels leave the
// SMs with fewer than 6 warps each; then enough segments (of at least 32
// chunks) for about 6 warps per SM (measured: B8 L2048 D1536 fp32, 768
// 16-channel warps, 0.720 -> 0.624 ms with 2 segments; unlike the forward,
// whose segment pass costs more than it gains above 2 warps per SM).
inline int bwd_segments(int batch, int dinner, int seqlen, int cw) {
    const long long warps = static_cast<long long>(batch) * ((dinner + cw - 1) / cw);
    if (warps <= 0 || warps >= 152LL * 6) return 1;
    long long g = (152LL * 6 + warps - 1) / warps;
    const long long gmax = ((seqlen + kChunk - 1) / kChunk) / 32;
    if (g > gmax) g = gmax;
    return g < 1 ? 1 : static_cast<int>(g);
}

struct ScanFwdArgs {
    const void* B;
    const void* C;
    const float* A_log;
    const float* D;      // may be null
    void* out;
    float* ctx;          // checkpoints [batch][nck][NT][dinner], may be null
    void* ysave;         // pre-gate y (M, dinner) packed, activation dtype; may be null
    int batch, seqlen, dinner, dstate;
    int64_t ld_B, ld_C, ld_out;
    int nck;             // checkpoints per batch row = ceil(seqlen / kChunk) - 1
    int bc_tma;          // 1: B and C arrive by TMA with the activation tiles
    // Time segments (scanned in parallel when the channels alone give too few
    // warps): nseg segments of seg_tiles tiles; segment g > 0 starts from
    // h0[b][g][NT][dinner].  seg_h / seg_ds: end state from a zero start and
    // sum of delta of each segment (segment pass output, combine input).
    int nseg, seg_tiles;
    float* h0;
    float* seg_h;
    float* seg_ds;
    // Carried state (inference): h_init is the state before the first step
    // (null = 0), h_last receives the state after the last step (may be null);
    // both [batch][dstate][dinner].
    const float* h_init;
    float* h_last;
};

struct ScanBwdArgs {
    const void* B;
    const void* C;
    const float* A_log;
    const float* D;      // may be null
    void* du;
    void* ddelta;
    void* dz;            // null when there is no gate
    float* ws_bc;        // [ncl][batch][seqlen][2][NT] dB | dC partial sums, one plane per CTA column
    float* ws_dA;        // [batch][dinner][NT] partial d/dA
    float* ws_dD;        // [batch][dinner] partial dD
    int batch, seqlen, dinner, dstate;
    int64_t ld_B, ld_C, ld_du, ld_ddelta, ld_dz;
    int nck;
    int ncl;             // CTA columns = ceil(dinner / cw) = dB/dC partial planes
    int cw;              // channels per CTA (bwd_channels)
    // Time segments (walked in parallel when the channels alone give too few
    // warps): nseg segments of seg_chunks chunks.  Segment sg < nseg-1 starts
    // its reverse walk from carry_g[b][sg][NT][dinner] (dL/dh at the first step
    // of segment sg+1) and carry_dl[b][sg][dinner] (delta there).  seg_g,
    // seg_ds, seg_d0: the segment pass's dL/dh at each segment's first step
    // from a zero carry, sum of delta over its steps after the first, and
    // delta at its first step.  ws_dA / ws_dD then hold batch*nseg planes.
    int nseg, seg_chunks;
    float* carry_g;
    float* carry_dl;
    float* seg_g;
    float* seg_ds;
    float* seg_d0;
    int bc_tma;          // 1: B and C arrive by TMA with the activation tiles
};

struct ScanReduceArgs {
    const float* ws_bc;
    const float* ws_dA;
    const float* ws_dD;
    const float* A_log;
    void* dB;
    void* dC;
    float* dA_log;
    float* dD;           // may be null
    int batch, seqlen, dinner, dstate, nt, ncl;
    int nb_sum;          // batch planes of ws_dA / ws_dD to add (0 if none were written)
    int64_t ld_dB, ld_dC;
    int is_bf16;
};

// Host launchers (scan_fwd.cu / scan_bwd.cu).  Return cudaSuccess or the launch error.
// Tensor maps of the forward: loads of u, delta_raw, z (32 channels x kFwdTile
// steps) and B, C (NT states x kFwdTile steps).
// Stores: out and the saved pre-gate y (32 channels x kFwdTile steps) and the
// checkpoints (32 channels x NT states of one chunk boundary).
struct FwdMaps {
    CUtensorMap u, dr, z, B, C, out, y, ck;
};
// With a.nseg > 1 this runs the segment pass, the combine and the segmented
// forward, in stream order.
cudaError_t launch_scan_fwd(int dtype, int nt, int disc, bool gate, const FwdMaps& maps,
                            const ScanFwdArgs& a, cudaStream_t stream);
// Tensor maps of the backward: u, delta_raw, z, dout, the saved pre-gate y
// (all cw channels x kChunk steps boxes) and the checkpoints (cw x NT box).
struct BwdMaps {
    CUtensorMap u, dr, z, dout, y, ck, B, C;
};
cudaError_t launch_scan_bwd(int dtype, int nt, int disc, bool gate, const BwdMaps& maps,
                            const ScanBwdArgs& a, cudaStream_t stream);
cudaError_t launch_scan_reduce(const ScanReduceArgs& a, cudaStream_t stream);

// Read and clear the fault word of the forward / backward translation unit.
cudaError_t read_clear_fault_fwd(unsigned* out);
cudaError_t read_clear_fault_bwd(unsigned* out);
// ... and of the probe / self-test translation unit.
cudaError_t read_clear_fault_probe(unsigned* out);

}  // namespace ssm

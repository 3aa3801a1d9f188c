// decode_args.cuh -- argument blocks of the single-token decode kernels
// (decode.cu), shared with the C-ABI layer (abi.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

// One step of the scan for every batch row.  Activations are rows of
// (batch, dinner) / (batch, dstate) views with the given row strides; the
// state h is [batch][dstate][dinner] fp32, read and overwritten.
struct ScanStepArgs {
    const void* u;
    const void* dr;        // delta_raw
    const void* z;         // may be null (no gate)
    const void* B;
    const void* C;
    const float* A_log;    // (dinner, dstate)
    const float* D;        // may be null
    float* h;
    void* out;
    int batch, dinner, dstate;
    int64_t ld_u, ld_dr, ld_z, ld_B, ld_C, ld_out;
};

// One step of the causal conv1d + SiLU; the kconv-1 previous inputs of batch
// row b sit in state [batch][kconv-1][dinner], slot j = the input kconv-1-j
// steps back (zeros before the sequence); the step shifts them by one.
struct ConvStepArgs {
    const float* x;
    const float* w;        // (dinner, kconv), tap 0 = current step
    const float* bias;     // may be null
    float* state;
    float* out;
    int batch, dinner, kconv;
    int64_t ld_x, ld_out;
};

// The conv state that continues a prompt of seqlen rows per batch row (x is
// (batch*seqlen, dinner) with row stride ld_x): slot j = the input at position
// seqlen-(kconv-1)+j, zero where that is before 0.
struct ConvStateFillArgs {
    const float* x;
    float* state;
    int batch, seqlen, dinner, kconv;
    int64_t ld_x;
};

cudaError_t launch_scan_step(int dtype, int nt, int disc, bool gate, const ScanStepArgs& a,
                             cudaStream_t st);
cudaError_t launch_conv_step(const ConvStepArgs& a, cudaStream_t st);
cudaError_t launch_conv_state_fill(const ConvStateFillArgs& a, cudaStream_t st);

}  // namespace ssm

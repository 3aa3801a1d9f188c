// conv_args.cuh -- argument block of the conv1d+SiLU kernels (conv1d.cu),
// shared with the C-ABI layer (abi.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

constexpr int kConvRun = 64;   // rows walked by one thread

struct ConvArgs {
    const float* x;
    const float* w;       // (dinner, kconv), tap 0 = current step
    const float* bias;    // may be null
    const float* dout;    // backward only
    float* out;           // forward only
    float* dx;            // backward only
    float* dw;
    float* dbias;         // may be null
    float* ws;            // backward partials [batch*runs][dinner][kconv+1]
    int batch, seqlen, dinner, kconv;
    int64_t ld_x, ld_out, ld_dout, ld_dx;
};

// Capacity, in floats, of the file-scope scratch used by the allocation-free
// backward entry point (8 MiB).
constexpr size_t kConvNoAllocScratchFloats = size_t(1) << 21;

cudaError_t launch_conv1d_fwd(const ConvArgs& a, cudaStream_t st);
cudaError_t conv1d_noalloc_scratch(float** out);
cudaError_t launch_conv1d_bwd(const ConvArgs& a, cudaStream_t st);
size_t conv1d_bwd_workspace_bytes(int batch, int seqlen, int dinner, int kconv);

}  // namespace ssm

// host_util.h -- host-side helpers shared by the C-ABI translation units
// (abi.cu, block.cu): device check, TMA encoder lookup, error bookkeeping.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdint>

#include "ssm_gb300.h"

namespace ssm_host {

// Records the CUDA error for ssm_last_cuda_error() and returns `s`.
ssm_status fail_cuda(cudaError_t e, ssm_status s = SSM_ERR_LAUNCH);
// SSM_OK when the current device is an sm_103 GPU (cached per device).
ssm_status check_device();
// cuTensorMapEncodeTiled through the runtime's driver entry point, or null.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
// The selective-scan forward with a saved context (ctx, may be null) and the
// carried states (h_init: state before the first step, null = 0; h_last:
// state after the last step, may be null), behind ssm_scan_fwd and
// ssm_scan_fwd_state (abi.cu); the block forward uses it for its prefill.
ssm_status scan_fwd_impl(const ssm_scan_desc* d, const void* u, const void* delta_raw,
                         const float* A_log, const void* B, const void* C, const float* D,
                         const void* z, void* out, void* ctx, size_t ctx_bytes, const float* h_init,
                         float* h_last, void* workspace, size_t workspace_bytes, cudaStream_t stream);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

}  // namespace ssm_host

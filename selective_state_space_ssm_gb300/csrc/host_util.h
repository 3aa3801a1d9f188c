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

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

}  // namespace ssm_host

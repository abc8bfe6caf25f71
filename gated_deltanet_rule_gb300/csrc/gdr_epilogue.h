// Internal declarations of the gated RMSNorm epilogue (not part of the ABI).
#pragma once

#include <cuda_runtime.h>

#include "gdr_internal.h"

namespace gdr {

constexpr int kKernEpilogue = kNumKernelIds;   // stage-timer id, after the path's own kernels

// Gated RMSNorm over `rows` rows of kD values: x, z, out bf16 [rows, kD]; w [kD] float32.
struct EpilogueArgs {
  const void* x;
  const void* z;
  const float* w;
  float eps;
  void* out;
  long long rows;
};
cudaError_t launch_gated_rmsnorm(const EpilogueArgs& a, cudaStream_t s);

}  // namespace gdr

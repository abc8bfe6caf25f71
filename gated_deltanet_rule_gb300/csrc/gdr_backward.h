// Internal declarations of the backward (not part of the ABI).
#pragma once

#include <cuda_runtime.h>

#include "gdr_epilogue.h"

namespace gdr {

// Stage-timer ids, after the epilogue's.
constexpr int kKernBackward = kKernEpilogue + 1;
constexpr int kKernBackwardReduce = kKernEpilogue + 2;

constexpr int kBwdSeg = 32;        // tokens per recomputed segment
constexpr int kBwdColBlocks = 8;   // CTAs per (row, value head), each owning D / 8 value columns

// Reverse mode through the token recurrence. q, k, v, dO share one element type (bf16 or f32);
// g, beta, S0, dS_T and every gradient are float32. S0 and dS_T may be NULL (zeros), dS0 may be
// NULL (not written). ws holds backward_workspace_bytes(B, L, Hk, Hv) bytes.
struct BackwardArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* S0;
  const void* dO;
  const float* dS_T;
  float* dq;
  float* dk;
  float* dv;
  float* dg;
  float* dbeta;
  float* dS0;
  void* ws;
  int B, L, Hk, Hv;
  bool bf16;
};
size_t backward_workspace_bytes(int B, int L, int Hk, int Hv);
cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s);

}  // namespace gdr

// Internal declarations of the backward (not part of the ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gdr_epilogue.h"

namespace gdr {

// Stage-timer ids, after the epilogue's.
constexpr int kKernBackward = kKernEpilogue + 1;
constexpr int kKernBackwardReduce = kKernEpilogue + 2;
// the chunked backward (bf16): the adjoint chain, the chunk-local gradients (with the key-head sums
// and the normalisations' backward)
constexpr int kKernChunkAdjoint = kKernEpilogue + 3;
constexpr int kKernChunkBwdLocal = kKernEpilogue + 4;

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

// The chunked backward's sequential passes over bf16 rows (any L >= 1): the forward's chunk factors
// (prep kernel, into ws), the chunk-entry states (state kernel, mode 1: S_save), and the adjoint
// chain with Nb = Q'^T dO formed on its output side (state kernel, mode 2: dS0 and, per chunk, the
// adjoint of its exiting state, dS_save). S_save and dS_save hold per (row, value head, chunk) four
// fp16 images of 8 KiB, one per 32-column slice (128 key rows of 64 bytes, 64-byte swizzle), each
// divided by its power of two in S_scale / dS_scale [B, Hv, NC, 4]; ws holds
// chunk_bwd_units_bytes(B, L, Hv) bytes. dS_T may be NULL (zeros), dS0 NULL (not written).
struct ChunkBwdChainLaunch {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* S0;
  const void* dO;
  const float* dS_T;
  float* dS0;
  __half* S_save;
  float* S_scale;
  __half* dS_save;
  float* dS_scale;
  float* unit_scale;   // [B, Hv, NC, 8]: dO's four slice powers of two, then v's
  void* ws;
  int B, L, Hk, Hv;
  int* err;
  bool saved = false;  // the factors, S_save, S_scale and v's scales are in place: adjoint chain only
};
size_t chunk_bwd_units_bytes(int B, int L, int Hv);
cudaError_t launch_chunk_bwd_chain(const ChunkBwdChainLaunch& p, cudaStream_t s);

// The forward (o, S_T, as the bf16 prefill computes them) that also leaves what the chunked
// backward's sequential passes would recompute: the chunk factors in ws, the chunk-entry states in
// S_save / S_scale and v's powers of two in unit_scale (word 4), in the layout of
// ChunkBwdChainLaunch (rows of one chunk included).
struct ChunkFwdSaveLaunch {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* S0;
  void* o;
  float* S_T;
  __half* S_save;
  float* S_scale;
  float* unit_scale;
  void* ws;
  int B, L, Hk, Hv;
  int* err;
};
cudaError_t launch_chunk_fwd_save(const ChunkFwdSaveLaunch& p, cudaStream_t s);

// The chunked backward of bf16 rows (q, k, v, dO bf16; g, beta, S0, dS_T and every gradient
// float32): the sequential passes above, then the chunk-local gradients, one CTA per (row, key head,
// chunk) taking the key head's value heads in turn and finishing dq, dk itself.
// ws holds chunk_bwd_workspace_bytes(B, L, Hk, Hv) bytes.
struct ChunkBackwardArgs {
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
  int* err;
  bool saved = false;  // ws holds what launch_chunk_forward_saving left: skip the forward passes
};
size_t chunk_bwd_workspace_bytes(int B, int L, int Hk, int Hv);
cudaError_t launch_chunk_backward(const ChunkBackwardArgs& p, cudaStream_t s);
// The bf16 prefill (o, S_T) leaving in ws (chunk_bwd_workspace_bytes) the forward passes'
// results for launch_chunk_backward with saved = true.
cudaError_t launch_chunk_forward_saving(const void* q, const void* k, const void* v, const float* g,
                                        const float* beta, const float* S0, void* o, float* S_T, void* ws,
                                        int B, int L, int Hk, int Hv, int* err, cudaStream_t s);

}  // namespace gdr

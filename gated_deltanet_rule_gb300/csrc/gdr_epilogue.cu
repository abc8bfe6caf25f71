// Gated RMSNorm epilogue: out = w * (x / sqrt(mean(x^2) + eps)) * silu(z) over each row of D values
// (DEG "model.py": _gated_rms, applied to the recurrence output o with the gate z per position and
// value head). A streaming kernel bound by HBM: sixteen threads per row, eight values (one 16-byte
// vector) each, the row's sum of squares reduced by shuffles; fp32 arithmetic from the bf16 inputs,
// one rounding to bf16 at the end.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdr_epilogue.h"

namespace gdr {
namespace {

constexpr int kEpiThreads = 256;   // 16 rows of 128 values per block

__global__ void __launch_bounds__(kEpiThreads) gated_rmsnorm_kernel(const EpilogueArgs a) {
  const long long row = ((long long)blockIdx.x * kEpiThreads + threadIdx.x) >> 4;
  const int part = threadIdx.x & 15;   // this thread's 8 values: columns 8 part .. 8 part + 7
  const bool live = row < a.rows;
  const long long off = (live ? row : 0) * (kD / 8) + part;
  float x[8], zf[8];
  {
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.x) + off);
    const uint4 zv = __ldg(reinterpret_cast<const uint4*>(a.z) + off);
    const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w}, zu[4] = {zv.x, zv.y, zv.z, zv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(xu[e] << 16);
      x[2 * e + 1] = __uint_as_float(xu[e] & 0xFFFF0000u);
      zf[2 * e] = __uint_as_float(zu[e] << 16);
      zf[2 * e + 1] = __uint_as_float(zu[e] & 0xFFFF0000u);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);   // the row's 16 threads
  const float r = rsqrtf(ss * (1.f / kD) + a.eps);
  const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.w) + 2 * part);
  const float4 w1 = __ldg(reinterpret_cast<const float4*>(a.w) + 2 * part + 1);
  const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  uint32_t ou[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float y[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float zz = zf[2 * e + u];
      y[u] = wv[2 * e + u] * (x[2 * e + u] * r) * __fdividef(zz, 1.f + __expf(-zz));
    }
    const __nv_bfloat162 h = __floats2bfloat162_rn(y[0], y[1]);
    ou[e] = *reinterpret_cast<const uint32_t*>(&h);
  }
  if (live) reinterpret_cast<uint4*>(a.out)[off] = make_uint4(ou[0], ou[1], ou[2], ou[3]);
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const EpilogueArgs& a, cudaStream_t s) {
  const int slot = stage_timer_begin(s, kKernEpilogue);
  const long long threads = a.rows * 16;
  gated_rmsnorm_kernel<<<(unsigned)((threads + kEpiThreads - 1) / kEpiThreads), kEpiThreads, 0, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  stage_timer_end(slot, s);
  return e;
}

}  // namespace gdr

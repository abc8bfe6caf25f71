// Token-by-token gated delta rule on CUDA cores, float32 state held in registers.
//
// Serves the float32 prefill path (where a 1e-4 relative bound rules out bf16 tensor-core
// operands), the fork batch and the L = 1 decode step (DEG "model.py": DecodeGraph, a CUDA-graph
// decode step over per-row states updated in place).
//
// Recurrence (Kev-4B-LiteRT "r15_kernel_test.py", truth_f64), rearranged so the state is read
// once per token:  with e = exp(g), kv = e S^T k^,  delta = beta (v - kv),
//   S' = e S + k^ delta^T,   o = S'^T q~ = e S^T q~ + (k^ . q~) delta.
// Columns of S are independent, so a CTA owns 32 value columns of one (row, value head) for all
// 128 key rows: thread t holds rows (t/8) + 16m, m = 0..7, and 4 adjacent columns 4(t%8)..+3
// (32 floats). The two column reductions over key rows (S^T k, S^T q) are warp shuffles plus a
// 4-warp exchange in shared memory; q, k norms and q.k are block reductions.
#include <cuda_bf16.h>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kCols = 32;       // value columns per CTA
constexpr int kThreads = 128;
constexpr float kScale = 0.08838834764831845f;   // 128^-0.5

__device__ __forceinline__ float ld_in(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_in(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(RecurrentArgs a) {
  const int cb = blockIdx.x & 3;      // which 32-column block of the 128 value columns
  const int b = blockIdx.x >> 2;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int cg = tid & 7;
  const int rg = tid >> 3;
  const int warp = tid >> 5, lane = tid & 31;
  const int hk = h / (a.Hv / a.Hk);
  // tokens of this row: L, or the row's length (later tokens are not run, their o is not written)
  int L = a.L;
  if (a.lengths) {
    L = a.lengths[b];
    if (L < 0 || L > a.L) {
      if (tid == 0) atomicCAS(a.err, 0, kErrDeviceIndex);
      return;   // this row's outputs stay untouched
    }
  }

  __shared__ float qs[2][kD], ks[2][kD], vs[2][kCols];
  __shared__ float nred[2][4][3];        // per-warp partials of q.q, k.k, q.k
  __shared__ float red[2][4][8][8];      // [buf][warp][cg][pk0..3, pq0..3]

  const float* S_in = nullptr;
  if (a.S_in != nullptr) {
    long long src = b;
    if (a.idx != nullptr) {
      src = a.idx[b];
      if (src < 0 || src >= a.n_in) {
        if (tid == 0) atomicCAS(a.err, 0, kErrDeviceIndex);
        return;   // this row's outputs stay untouched
      }
    }
    S_in = a.S_in + ((size_t)src * a.Hv + h) * kD * kD;
  }
  const int col0 = cb * kCols + 4 * cg;
  float S[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (S_in) x = __ldg(reinterpret_cast<const float4*>(S_in + (size_t)(rg + 16 * m) * kD + col0));
    S[m][0] = x.x; S[m][1] = x.y; S[m][2] = x.z; S[m][3] = x.w;
  }

  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  T* o = static_cast<T*>(a.o);
  const size_t row_tok = (size_t)b * a.L;

  float qn = 0.f, kn = 0.f, vn = 0.f, gn = 0.f, bn = 0.f;
  auto fetch = [&](int t) {
    const size_t qk_off = ((row_tok + t) * a.Hk + hk) * kD + tid;
    qn = ld_in(q + qk_off);
    kn = ld_in(k + qk_off);
    if (tid < kCols) vn = ld_in(v + ((row_tok + t) * a.Hv + h) * kD + cb * kCols + tid);
    gn = __ldg(a.g + (row_tok + t) * a.Hv + h);
    bn = __ldg(a.beta + (row_tok + t) * a.Hv + h);
  };
  if (L > 0) fetch(0);

  bool changed = false;
  for (int t = 0; t < L; ++t) {
    const int buf = t & 1;
    const float qv = qn, kv = kn, vv = vn, gt = gn, bt = bn;
    if (t + 1 < L) fetch(t + 1);
    changed |= (gt != 0.f) || (bt != 0.f);

    qs[buf][tid] = qv;
    ks[buf][tid] = kv;
    if (tid < kCols) vs[buf][tid] = vv;
    float s0 = qv * qv, s1 = kv * kv, s2 = qv * kv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
      s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    }
    if (lane == 0) { nred[buf][warp][0] = s0; nred[buf][warp][1] = s1; nred[buf][warp][2] = s2; }
    __syncthreads();

    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float kk = ks[buf][rg + 16 * m], qq = qs[buf][rg + 16 * m];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        pk[c] = fmaf(S[m][c], kk, pk[c]);
        pq[c] = fmaf(S[m][c], qq, pq[c]);
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      pk[c] += __shfl_xor_sync(0xffffffffu, pk[c], 8);
      pk[c] += __shfl_xor_sync(0xffffffffu, pk[c], 16);
      pq[c] += __shfl_xor_sync(0xffffffffu, pq[c], 8);
      pq[c] += __shfl_xor_sync(0xffffffffu, pq[c], 16);
    }
    if (lane < 8) {
#pragma unroll
      for (int c = 0; c < 4; ++c) { red[buf][warp][lane][c] = pk[c]; red[buf][warp][lane][4 + c] = pq[c]; }
    }
    __syncthreads();

    const float sqq = nred[buf][0][0] + nred[buf][1][0] + nred[buf][2][0] + nred[buf][3][0];
    const float skk = nred[buf][0][1] + nred[buf][1][1] + nred[buf][2][1] + nred[buf][3][1];
    const float sqk = nred[buf][0][2] + nred[buf][1][2] + nred[buf][2][2] + nred[buf][3][2];
    const float qinv = rsqrtf(sqq + 1e-6f), kinv = rsqrtf(skk + 1e-6f);
    const float e = expf(gt);
    const float ekinv = e * kinv, eqs = e * qinv * kScale, kq = kinv * qinv * kScale * sqk;
    float delta[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float fk = red[buf][0][cg][c] + red[buf][1][cg][c] + red[buf][2][cg][c] + red[buf][3][cg][c];
      delta[c] = bt * (vs[buf][4 * cg + c] - ekinv * fk);
    }
    if (rg == 0) {
      T* op = o + ((row_tok + t) * a.Hv + h) * kD + col0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float fq = red[buf][0][cg][4 + c] + red[buf][1][cg][4 + c] + red[buf][2][cg][4 + c] +
                         red[buf][3][cg][4 + c];
        st_out(op + c, eqs * fq + kq * delta[c]);
      }
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float kk = kinv * ks[buf][rg + 16 * m];
#pragma unroll
      for (int c = 0; c < 4; ++c) S[m][c] = fmaf(e, S[m][c], kk * delta[c]);
    }
  }

  if (a.S_out != nullptr) {
    // An in-place update whose tokens were all pads (beta = g = 0) leaves the state bit-identical.
    const bool untouched = !changed && a.idx == nullptr && a.S_out == a.S_in;
    if (!untouched) {
      float* S_out = a.S_out + ((size_t)b * a.Hv + h) * kD * kD;
#pragma unroll
      for (int m = 0; m < 8; ++m)
        *reinterpret_cast<float4*>(S_out + (size_t)(rg + 16 * m) * kD + col0) =
            make_float4(S[m][0], S[m][1], S[m][2], S[m][3]);
    }
  }
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentArgs& a, cudaStream_t s) {
  dim3 grid((unsigned)(4 * a.B), (unsigned)a.Hv);
  if (a.bf16)
    recurrent_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a);
  else
    recurrent_kernel<float><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace gdr

// GDN prologue: the causal depthwise convolution + SiLU that turns the q|k|v projection into the
// path's q, k, v, the gates beta and g, and the convolution carry for the next call.
// (DEG "model.py": _linear_layer, with _conv_silu over ext = [tail, mixed] and _dn_gates.)
//
// One streaming kernel, bound by HBM: every input element is read once and every output written
// once. A block takes a tile of 16 positions x 512 channels of one row: one warp copies the tile's
// ext rows (the 16 positions and the K - 1 before them, 1 KB each) into shared memory by bulk
// asynchronous copies completing on one mbarrier, so that many kilobytes per SM are in flight
// without registers; then each thread convolves 4 channels down the 16 positions with the last K
// inputs in registers (a sliding window), fp32 arithmetic and one rounding to bf16, a warp writing
// 256 contiguous bytes per position. Then every thread takes a grid-stride share of
//  - the gates: one (row, position, value head) per element, and
//  - the carry: 8 channels of one of the K-1 carried positions per element.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gdr_internal.h"
#include "ptx.cuh"

namespace gdr {
namespace {

using namespace ptx;

constexpr int kConvThreads = 128;                // threads per block (4 channels each)
constexpr int kConvRun = 16;                     // positions per tile
constexpr int kTileCh = 4 * kConvThreads;        // channels per tile
constexpr uint32_t kRowBytes = kTileCh * 2;      // shared-memory row: one ext position of the tile
constexpr long long kDrainBudget = 2000000000ll; // cycles (~1 s) a block that gave up waits for its copies
template <int K>
constexpr uint32_t conv_smem() { return (kConvRun + K - 1) * kRowBytes; }

__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ext position e of row b: the carried input tail[b][e] for e < K-1, else mixed[b][e - (K-1)]
__device__ __forceinline__ uint4 ext_load(const PrologueArgs& a, int b, int e, int c8, int K) {
  const size_t C = a.C;
  if (e < K - 1) {
    if (!a.tail) return make_uint4(0, 0, 0, 0);
    return __ldg(reinterpret_cast<const uint4*>(a.tail) + ((size_t)b * (K - 1) + e) * (C / 8) + c8);
  }
  return __ldg(reinterpret_cast<const uint4*>(a.mixed) + ((size_t)b * a.L + (e - (K - 1))) * (C / 8) + c8);
}

__device__ __forceinline__ void bf16x4_to_f32(uint2 w, float* x) {
  x[0] = __uint_as_float(w.x << 16);
  x[1] = __uint_as_float(w.x & 0xFFFF0000u);
  x[2] = __uint_as_float(w.y << 16);
  x[3] = __uint_as_float(w.y & 0xFFFF0000u);
}

__device__ __forceinline__ uint2 f32x4_to_bf16(const float* x) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(x[0], x[1]), h1 = __floats2bfloat162_rn(x[2], x[3]);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
}

// out[t] = sum_{j < K} w[c][j] ext[t + j]; y = out sigmoid(out), written to q, k or v by channel.
// The tile's ext rows t0 .. t0 + K + 14 land in stage (row i = ext position t0 + i, kRowBytes
// apart); rows past the last one that feeds an output (ext position >= L + K - 1) are not loaded.
template <int K>
__device__ __forceinline__ void conv_run(const PrologueArgs& a, uint8_t* stage, uint64_t* bar) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int c_base = blockIdx.x * kTileCh, b = blockIdx.z, t0 = blockIdx.y * kConvRun;
  const int nch = min(kTileCh, a.C - c_base);               // a multiple of 128
  const int rows = min(kConvRun + K - 1, a.L - t0 + K - 1);  // ext rows that feed this tile's outputs
  const uint32_t row_bytes = (uint32_t)nch * 2;
  if (!a.tail) {
    // carried positions without a carry read as zeros
    for (int i = 0; i < rows && t0 + i < K - 1; ++i)
      if (4 * tid < nch) *reinterpret_cast<uint2*>(stage + i * kRowBytes + tid * 8) = make_uint2(0, 0);
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid < 32) {
    const int first = a.tail ? 0 : max(0, K - 1 - t0);   // the rows before it are zeros, not copies
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(rows - first) * row_bytes);
    __syncwarp();
    for (int i = first + lane; i < rows; i += 32) {
      const int e = t0 + i;
      const uint8_t* src = e < K - 1
          ? static_cast<const uint8_t*>(a.tail) + (((size_t)b * (K - 1) + e) * a.C + c_base) * 2
          : static_cast<const uint8_t*>(a.mixed) + (((size_t)b * a.L + (e - (K - 1))) * a.C + c_base) * 2;
      bulk_load(stage + i * kRowBytes, src, row_bytes, bar);
    }
  }
  const int c4 = c_base / 4 + tid;   // this thread's 4-channel vector
  const bool mine = 4 * tid < nch;
  float w[K][4];   // this thread's 4 x K weights are 4 K contiguous floats (16-byte aligned: 16 K bytes)
  if (mine) {
    const float4* w4 = reinterpret_cast<const float4*>(a.conv_w + (size_t)c4 * 4 * K);
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const float4 f = __ldg(w4 + i);
      const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) w[(4 * i + u) % K][(4 * i + u) / K] = fv[u];
    }
  }
  // every thread waits for the copies (bounded); a block that gives up records the timeout and waits
  // once more for its copies before it leaves
  const bool ok = mbar_wait(bar, 0, a.wait_budget);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) {
      set_error(a.err, kErrTimeout);
      mbar_wait(bar, 0, kDrainBudget);
    }
    __syncthreads();
    return;
  }
  if (!mine) return;
  // destination: channels [0, HkD) -> q, [HkD, 2 HkD) -> k, the rest -> v (4-channel vectors never
  // straddle a boundary, since the boundaries are multiples of 128)
  const int HkD = a.Hk * kD, c0 = c4 * 4;
  uint2* dst;
  size_t stride4;   // vectors per position in the destination
  if (c0 < HkD) {
    dst = reinterpret_cast<uint2*>(a.q) + c0 / 4;
    stride4 = HkD / 4;
  } else if (c0 < 2 * HkD) {
    dst = reinterpret_cast<uint2*>(a.k) + (c0 - HkD) / 4;
    stride4 = HkD / 4;
  } else {
    dst = reinterpret_cast<uint2*>(a.v) + (c0 - 2 * HkD) / 4;
    stride4 = (size_t)a.Hv * kD / 4;
  }
  const uint8_t* col = stage + tid * 8;
  float win[K][4];   // ext positions t .. t + K - 1
#pragma unroll
  for (int j = 0; j < K - 1; ++j) bf16x4_to_f32(*reinterpret_cast<const uint2*>(col + j * kRowBytes), win[j]);
  const int n = min(kConvRun, a.L - t0);
#pragma unroll 4
  for (int u = 0; u < n; ++u) {
    bf16x4_to_f32(*reinterpret_cast<const uint2*>(col + (u + K - 1) * kRowBytes), win[K - 1]);
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float sacc = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j) sacc = fmaf(w[j][e], win[j][e], sacc);
      y[e] = __fdividef(sacc, 1.f + __expf(-sacc));   // one rounding to bf16 follows
    }
    dst[((size_t)b * a.L + t0 + u) * stride4] = f32x4_to_bf16(y);
#pragma unroll
    for (int j = 0; j < K - 1; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) win[j][e] = win[j + 1][e];
  }
}

// beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias) at valid positions, 0 at pads
__device__ __forceinline__ void gate_element(const PrologueArgs& a, long long i) {
  const int h = (int)(i % a.Hv);
  const long long bt = i / a.Hv;
  const int t = (int)(bt % a.L), b = (int)(bt / a.L);
  int len = a.L;
  if (a.lengths) {
    len = a.lengths[b];
    if (len < 0 || len > a.L) {
      if (t == 0 && h == 0) set_error(a.err, kErrDeviceIndex);
      return;   // the row's gates are left untouched
    }
  }
  float beta = 0.f, g = 0.f;
  if (t < len) {
    beta = 1.f / (1.f + expf(-a.proj_b[i]));
    const float x = a.proj_a[i] + a.dt_bias[h];
    const float sp = x > 20.f ? x : log1pf(expf(x));
    g = -expf(a.A_log[h]) * sp;
  }
  a.beta[i] = beta;
  a.g[i] = g;
}

// new_tail[b][j] = ext[b][len_b + j], j < K-1: the K-1 inputs ending at the row's last valid token
__device__ __forceinline__ void carry_element(const PrologueArgs& a, long long i, int K) {
  const int c8 = (int)(i % (a.C / 8));
  const int j = (int)((i / (a.C / 8)) % (K - 1)), b = (int)(i / ((long long)(a.C / 8) * (K - 1)));
  int len = a.L;
  if (a.lengths) {
    len = a.lengths[b];
    if (len < 0 || len > a.L) return;   // recorded with the gates; the row's carry is untouched
  }
  reinterpret_cast<uint4*>(a.new_tail)[((size_t)b * (K - 1) + j) * (a.C / 8) + c8] = ext_load(a, b, len + j, c8, K);
}

// One launch for the whole prologue: every thread runs its part of the convolution, then takes its
// share of the gates and of the carry (grid-stride over their elements).
template <int K>
__global__ void __launch_bounds__(kConvThreads) prologue_kernel(const PrologueArgs a) {
  extern __shared__ __align__(16) uint8_t stage[];
  __shared__ uint64_t bar;
  const long long nthreads = (long long)gridDim.x * gridDim.y * gridDim.z * kConvThreads;
  const long long gtid =
      (((long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * kConvThreads + threadIdx.x;
  conv_run<K>(a, stage, &bar);
  const long long ngates = (long long)a.B * a.L * a.Hv;
  for (long long i = gtid; i < ngates; i += nthreads) gate_element(a, i);
  if (K > 1 && a.new_tail) {
    const long long ncarry = (long long)a.B * (K - 1) * (a.C / 8);
    for (long long i = gtid; i < ncarry; i += nthreads) carry_element(a, i, K);
  }
}

template <int K>
cudaError_t launch_conv(const PrologueArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)((a.C + kTileCh - 1) / kTileCh), (unsigned)((a.L + kConvRun - 1) / kConvRun),
                  (unsigned)a.B);
  // (below the default 48 KB; the largest carveout lets ten or more blocks share an SM. Set once per
  // device ordinal: it is a hint, and a call per launch costs host time a 30 us kernel notices)
  static std::atomic<unsigned long long> set_on{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (!bit || !(set_on.load() & bit)) {
    e = cudaFuncSetAttribute(prologue_kernel<K>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    set_on.fetch_or(bit);
  }
  prologue_kernel<K><<<grid, kConvThreads, conv_smem<K>(), s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t s) {
  int slot = stage_timer_begin(s, kKernPrologue);
  cudaError_t e;
  switch (a.K) {
    case 1: e = launch_conv<1>(a, s); break;
    case 2: e = launch_conv<2>(a, s); break;
    case 3: e = launch_conv<3>(a, s); break;
    case 4: e = launch_conv<4>(a, s); break;
    case 5: e = launch_conv<5>(a, s); break;
    case 6: e = launch_conv<6>(a, s); break;
    case 7: e = launch_conv<7>(a, s); break;
    default: e = launch_conv<8>(a, s); break;
  }
  stage_timer_end(slot, s);
  return e;
}

}  // namespace gdr

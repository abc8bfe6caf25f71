// Chunked gated delta rule on tcgen05 tensor cores (bf16 operands, float32 accumulation).
//
// Chunk algebra (64-token chunks; the "R64" form named in Kev-4B-LiteRT "r15_kernel_test.py",
// with the pair decay computed directly, never as a ratio of cumulative decays). For a chunk with
// entering state S, gamma_i = sum_{j<=i} g_j, Gamma_i = exp(gamma_i), raw q/k rows and their
// inverse norms qi_i = (|q_i|^2 + 1e-6)^-1/2, ki_i likewise:
//
//   A_ij  = beta_i ki_i ki_j (k_i . k_j) exp(gamma_i - gamma_j),  j < i         (strictly lower)
//   T     = (I + A)^-1                                                          (unit lower)
//   W     = T diag(beta Gamma ki) K,     U = T diag(beta) V                     (WY factors)
//   P_ij  = qi_i ki_j D^-1/2 (q_i . k_j) exp(gamma_i - gamma_j),  j <= i
//   Vnew  = U - W S
//   O     = diag(Gamma qi D^-1/2) Q S + P Vnew
//   S'    = Gamma_C S + K^T diag(exp(gamma_C - gamma) ki) Vnew
//
// Kernel 1 (gdr_chunk_prep, one CTA per (row, key head, chunk), all chunks in parallel):
//   TMA loads the raw q, k tiles once per key head and the v tile of each of its r value heads;
//   one MMA gives [Q; K] K^T (both Gram matrices); CUDA cores build A and P, invert I + A by
//   16x16 blocks in fp32, and scale T's columns; one MMA pair gives W and U. W and P are written
//   to the workspace as 128B-swizzled shared-memory images (bulk-copied as they are by kernel 2),
//   U in 64-column slices, plus the per-position scales.
// Kernel 2 (gdr_chunk_state, one CTA per (row, value head, 64 value columns), sequential over
//   chunks): the float32 state slice stays in registers (one key row per thread); per chunk
//   MMA_A = [W; Q] S (both products in one M = 128 MMA), Vnew on CUDA cores, then MMA2 = K^T Vs
//   (state increment) and MMA3 = P Vnew (intra-chunk output), S update and the output stores.
//   The next chunk's tiles are loaded by TMA while the current chunk computes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "gdr_internal.h"
#include "ptx.cuh"

namespace gdr {

using namespace ptx;

namespace {

constexpr float kScale = 0.08838834764831845f;   // 128^-0.5
constexpr long long kWaitBudget = 2000000000ll;   // cycles (~1 s) before a wait gives up

// Workspace image sizes per (row, value head, chunk) unit.
// Precision: the operands an MMA takes from computed values are split into bf16 hi + lo pairs
// where a single bf16 rounding would cost accuracy (T's scaled columns, U, P, and the two Vnew
// operands); W and the state operand S stay single bf16. Measured against the float64 oracle, this
// keeps outputs at the floor set by rounding o itself to bf16.
constexpr uint32_t kWBytes = 16384;     // W: 64 x 128 bf16, two 64-column swizzled atoms
constexpr uint32_t kPBytes = 16384;     // P: hi and lo bf16 images, 64 x 64 each, swizzled
constexpr uint32_t kUBytes = 32768;     // U: two slices of 64 x 64 float32, 16-byte chunks swizzled
constexpr uint32_t kSBytes = 1024;      // scales: sq[64], sk[64], Gamma_C (129 floats used)
constexpr uint32_t kSCopy = 528;        // bytes of the scale block kernel 2 copies (16-byte multiple)
constexpr uint32_t kUnitP = kWBytes, kUnitU = kUnitP + kPBytes, kUnitS = kUnitU + kUBytes;
constexpr uint32_t kUnitBytes = kUnitS + kSBytes;

struct ChunkArgs {
  const float* g;
  const float* beta;
  const float* S0;
  __nv_bfloat16* o;
  float* S_T;
  uint8_t* ws;       // 1024-aligned
  int B, L, Hk, Hv, NC;
  int* err;
};

__device__ __forceinline__ uint8_t* unit_base(const ChunkArgs& a, int b, int h, int c) {
  return a.ws + ((size_t)((size_t)b * a.Hv + h) * a.NC + c) * kUnitBytes;
}

__device__ __forceinline__ void set_error(int* err, int code) { atomicCAS(err, 0, code); }

// -------------------------------------------------------------------------------------------
// Kernel 1: per-chunk WY factors
// -------------------------------------------------------------------------------------------
constexpr int kPrepThreads = 128;
constexpr uint32_t kOffQK0 = 0, kOffQK1 = 16384, kOffV = 32768, kOffAop = 49152;
constexpr uint32_t kOffAm = 65536, kOffTm = kOffAm + 64 * 65 * 4, kOffXs = kOffTm + 64 * 65 * 4;
constexpr uint32_t kOffVec = kOffXs + 3 * 16 * 17 * 4;
constexpr uint32_t kPrepSmem = kOffVec + 5 * 64 * 4 + 1024;   // + alignment slack

__global__ void __launch_bounds__(kPrepThreads, 2)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_qk, bar_v, bar_mma;
  __shared__ uint32_t tmem_base;

  const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = a.Hv / a.Hk;
  float* Am = reinterpret_cast<float*>(sm + kOffAm);      // [64][65]
  float* Tm = reinterpret_cast<float*>(sm + kOffTm);      // [64][65]
  float* Xs = reinterpret_cast<float*>(sm + kOffXs);      // [3][16][17]
  float* gam = reinterpret_cast<float*>(sm + kOffVec);
  float* Gam = gam + 64;
  float* bet = gam + 128;
  float* qinv = gam + 192;
  float* kinv = gam + 256;

  if (tid == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    mbar_init(&bar_qk, 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  bool ok = true;

  if (tid == 0) {
    mbar_arrive_expect_tx(&bar_qk, 32768);
    tma_load_4d(sm + kOffQK0, &tm_q, &bar_qk, 0, hk, c * 64, b);
    tma_load_4d(sm + kOffQK1, &tm_q, &bar_qk, 64, hk, c * 64, b);
    tma_load_4d(sm + kOffQK0 + 8192, &tm_k, &bar_qk, 0, hk, c * 64, b);
    tma_load_4d(sm + kOffQK1 + 8192, &tm_k, &bar_qk, 64, hk, c * 64, b);
    mbar_arrive_expect_tx(&bar_v, 16384);
    tma_load_4d(sm + kOffV, &tm_v, &bar_v, 0, hk * r, c * 64, b);
    tma_load_4d(sm + kOffV + 8192, &tm_v, &bar_v, 64, hk * r, c * 64, b);
  }

  ok = mbar_wait(&bar_qk, 0, kWaitBudget);
  if (!__syncthreads_and(ok)) goto fail;

  // Inverse norms: thread t < 64 reads q row t, t >= 64 reads k row t - 64 (order-free sum).
  {
    const int row = tid & 63;
    const uint8_t* base = sm + (tid < 64 ? 0 : 8192) + row * 128;
    float s = 0.f;
#pragma unroll
    for (int atom = 0; atom < 2; ++atom) {
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + atom * 16384 + ch * 16);
        const uint32_t ws4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(ws4[e] << 16), hi = __uint_as_float(ws4[e] & 0xFFFF0000u);
          s = fmaf(lo, lo, s);
          s = fmaf(hi, hi, s);
        }
      }
    }
    (tid < 64 ? qinv : kinv)[row] = rsqrtf(s + 1e-6f);
  }

  // Gram MMA: D[0:128, 0:64] = [Q; K] K^T  (A rows 0-63 = q, 64-127 = k; B = k rows)
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = idesc_bf16(128, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t atom = smem_u32(sm) + (kk >> 2) * 16384 + (kk & 3) * 32;
      mma_bf16(tb, smem_desc(atom, 16, 1024), smem_desc(atom + 8192, 16, 1024), idesc, kk > 0);
    }
    mma_commit(&bar_mma);
  }
  ok = mbar_wait(&bar_mma, 0, kWaitBudget);
  if (!__syncthreads_and(ok)) goto fail;
  tc_fence_after();

  {
    // This thread's Gram row: rows 0-63 = (Q K^T)_i,:, rows 64-127 = (K K^T)_i,:
    float G[64];
    tmem_ld32(tb + lane_base + 0, G);
    tmem_ld32(tb + lane_base + 32, G + 32);
    tc_fence_before();
    const int i = tid & 63;

    for (int j = 0; j < r; ++j) {
      const int h = hk * r + j;
      // gates of this value head; positions past L read as beta = g = 0
      if (tid < 64) {
        const int p = c * 64 + tid;
        const bool in = p < a.L;
        const float gg = in ? __ldg(a.g + ((size_t)b * a.L + p) * a.Hv + h) : 0.f;
        bet[tid] = in ? __ldg(a.beta + ((size_t)b * a.L + p) * a.Hv + h) : 0.f;
        // inclusive scan of g over the chunk (two warps)
        float x = gg;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, off);
          if ((tid & 31) >= off) x += y;
        }
        gam[tid] = x;
      }
      __syncthreads();
      if (tid >= 32 && tid < 64) gam[tid] += gam[31];
      __syncthreads();
      if (tid < 64) Gam[tid] = expf(gam[tid]);

      // A (threads 64..127, row i) and P (threads 0..63, row i)
      const float gi = gam[i];
      if (tid >= 64) {
        const float si = bet[i] * kinv[i];
#pragma unroll
        for (int jj = 0; jj < 64; ++jj)
          Am[i * 65 + jj] = (jj < i) ? si * kinv[jj] * G[jj] * expf(gi - gam[jj]) : 0.f;
      } else {
        const float si = qinv[i] * kScale;
        uint8_t* prow = unit_base(a, b, h, c) + kUnitP + i * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t hv[4], lv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
            const float p0 = (j0 <= i) ? si * kinv[j0] * G[j0] * expf(gi - gam[j0]) : 0.f;
            const float p1 = (j1 <= i) ? si * kinv[j1] * G[j1] * expf(gi - gam[j1]) : 0.f;
            split_bf16x2(p0, p1, hv[e], lv[e]);
          }
          const uint32_t off = (ch ^ (i & 7)) << 4;
          *reinterpret_cast<uint4*>(prow + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<uint4*>(prow + 8192 + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        }
      }
      __syncthreads();

      // T = (I + A)^-1 by 16x16 blocks. Diagonal blocks: forward substitution per column.
      if (tid < 64) {
        const int blk = tid >> 4, col = tid & 15, r0 = blk * 16;
        float x[16];
#pragma unroll
        for (int ii = 0; ii < 16; ++ii) {
          float acc = 0.f;
#pragma unroll
          for (int jj = 0; jj < ii; ++jj) acc = fmaf(Am[(r0 + ii) * 65 + r0 + jj], x[jj], acc);
          x[ii] = (ii == col) ? 1.f : ((ii < col) ? 0.f : -acc);
          Tm[(r0 + ii) * 65 + r0 + col] = x[ii];
        }
      } else {
        // zero the blocks above the diagonal
        for (int e = tid - 64; e < 64 * 64; e += 64) {
          const int rr = e >> 6, cc = e & 63;
          if ((cc >> 4) > (rr >> 4)) Tm[rr * 65 + cc] = 0.f;
        }
      }
      __syncthreads();
      for (int I = 1; I < 4; ++I) {
        // X_IJ = sum_{M=J}^{I-1} A_IM T_MJ for J < I
        for (int e = tid; e < I * 256; e += kPrepThreads) {
          const int J = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
          float acc = 0.f;
          for (int M = J; M < I; ++M) {
#pragma unroll
            for (int m = 0; m < 16; ++m)
              acc = fmaf(Am[(16 * I + rr) * 65 + 16 * M + m], Tm[(16 * M + m) * 65 + 16 * J + cc], acc);
          }
          Xs[(J * 16 + rr) * 17 + cc] = acc;
        }
        __syncthreads();
        // T_IJ = -T_II X_IJ  (T_II unit lower triangular)
        for (int e = tid; e < I * 256; e += kPrepThreads) {
          const int J = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
          float acc = Xs[(J * 16 + rr) * 17 + cc];
          for (int m = 0; m < rr; ++m)
            acc = fmaf(Tm[(16 * I + rr) * 65 + 16 * I + m], Xs[(J * 16 + m) * 17 + cc], acc);
          Tm[(16 * I + rr) * 65 + 16 * J + cc] = -acc;
        }
        __syncthreads();
      }

      // A operand [T diag(beta Gamma ki); T diag(beta)], K-major swizzled (K = 64 positions), as
      // a bf16 hi image and a bf16 lo image (the lo image reuses A's storage, dead by now)
      {
        const bool wrow = tid < 64;
        uint8_t* arow = sm + kOffAop + tid * 128;
        uint8_t* lrow = sm + kOffAm + tid * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t hv[4], lv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
            const float s0 = wrow ? bet[j0] * Gam[j0] * kinv[j0] : bet[j0];
            const float s1 = wrow ? bet[j1] * Gam[j1] * kinv[j1] : bet[j1];
            split_bf16x2(Tm[i * 65 + j0] * s0, Tm[i * 65 + j1] * s1, hv[e], lv[e]);
          }
          const uint32_t off = (ch ^ (tid & 7)) << 4;
          *reinterpret_cast<uint4*>(arow + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<uint4*>(lrow + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();

      ok = mbar_wait(&bar_v, j & 1, kWaitBudget);
      if (!__syncthreads_and(ok)) goto fail;
      if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, 128, false, true);
        const uint32_t aop[2] = {smem_u32(sm + kOffAop), smem_u32(sm + kOffAm)};   // hi, lo
        const uint32_t kt = smem_u32(sm + kOffQK0 + 8192);   // k atoms at +8192 and +24576
        const uint32_t vt = smem_u32(sm + kOffV);            // v atoms at +0 and +8192
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tb, smem_desc(aop[part] + kk * 32, 16, 1024), smem_desc(kt + kk * 2048, 16384, 1024), idesc,
                     part | kk);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tb + 128, smem_desc(aop[part] + kk * 32, 16, 1024), smem_desc(vt + kk * 2048, 8192, 1024),
                     idesc, part | kk);
        mma_commit(&bar_mma);
      }
      ok = mbar_wait(&bar_mma, (j + 1) & 1, kWaitBudget);
      if (!__syncthreads_and(ok)) goto fail;
      tc_fence_after();

      // next value head's v tile (the U MMA has consumed this one)
      if (tid == 0 && j + 1 < r) {
        mbar_arrive_expect_tx(&bar_v, 16384);
        tma_load_4d(sm + kOffV, &tm_v, &bar_v, 0, h + 1, c * 64, b);
        tma_load_4d(sm + kOffV + 8192, &tm_v, &bar_v, 64, h + 1, c * 64, b);
      }

      uint8_t* ub = unit_base(a, b, h, c);
      if (tid < 64) {
        // W row i (TMEM lanes 0-63, columns 0-127) -> swizzled image
#pragma unroll
        for (int part = 0; part < 4; ++part) {
          float w[32];
          tmem_ld32(tb + lane_base + part * 32, w);
#pragma unroll
          for (int ch4 = 0; ch4 < 4; ++ch4) {
            const int col = part * 32 + ch4 * 8;
            const int atom = col >> 6, ch = (col & 63) >> 3;
            uint4 pk = make_uint4(pack_bf16x2(w[ch4 * 8 + 0], w[ch4 * 8 + 1]), pack_bf16x2(w[ch4 * 8 + 2], w[ch4 * 8 + 3]),
                                  pack_bf16x2(w[ch4 * 8 + 4], w[ch4 * 8 + 5]), pack_bf16x2(w[ch4 * 8 + 6], w[ch4 * 8 + 7]));
            *reinterpret_cast<uint4*>(ub + atom * 8192 + i * 128 + ((ch ^ (i & 7)) << 4)) = pk;
          }
        }
        // per-position scales for kernel 2
        float* sc = reinterpret_cast<float*>(ub + kUnitS);
        sc[i] = Gam[i] * qinv[i] * kScale;
        sc[64 + i] = expf(gam[63] - gam[i]) * kinv[i];
        if (i == 0) sc[128] = Gam[63];
      } else {
        // U row i (TMEM lanes 64-127, columns 128-255) -> two 64-column float32 slices; the
        // 16-byte chunk c of row i is stored at chunk c ^ (i % 8) so that row reads do not collide
#pragma unroll
        for (int part = 0; part < 4; ++part) {
          float u[32];
          tmem_ld32(tb + lane_base + 128 + part * 32, u);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const int col = part * 32 + c4 * 4;
            const int sl = col >> 6, ch = (col & 63) >> 2;
            *reinterpret_cast<float4*>(ub + kUnitU + sl * 16384 + i * 256 + ((ch ^ (i & 7)) << 4)) =
                make_float4(u[c4 * 4 + 0], u[c4 * 4 + 1], u[c4 * 4 + 2], u[c4 * 4 + 3]);
          }
        }
      }
      tc_fence_before();
      __syncthreads();
    }
  }
  goto done;
fail:
  if (tid == 0) set_error(a.err, kErrTimeout);
done:
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 256);
  }
}

// -------------------------------------------------------------------------------------------
// Kernel 2: sequential state recurrence over chunks, 64 value columns per CTA
// -------------------------------------------------------------------------------------------
constexpr int kStateThreads = 128;
// Stage (one chunk's tiles, 1024-aligned). [W0|Q0] and [W1|Q1] form the two K-atoms of the
// M = 128 operand [W; Q]; the 8 KB before P_hi (Q1) and before P_lo (P_hi) are the unused top
// halves of the operands [. ; P_hi] and [. ; P_lo].
constexpr uint32_t kStW0 = 0, kStQ0 = 8192, kStW1 = 16384, kStQ1 = 24576, kStPh = 32768, kStPl = 40960;
constexpr uint32_t kStK0 = 49152, kStK1 = 57344, kStU = 65536, kStS = 81920;
constexpr uint32_t kStage = 82944;
constexpr uint32_t kStageTx = kWBytes + 16384 + kPBytes + 16384 + 16384 + kSCopy;
constexpr uint32_t kOffSb = 2 * kStage, kOffVsh = kOffSb + 16384, kOffVsl = kOffVsh + 8192;
constexpr uint32_t kOffVuh = kOffVsl + 8192, kOffVul = kOffVuh + 8192;
constexpr uint32_t kStateSmem = kOffVul + 8192 + 1024;

__global__ void __launch_bounds__(kStateThreads, 1)
chunk_state_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[2], bar_mma;
  __shared__ uint32_t tmem_base;

  const int sl = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int hk = h / (a.Hv / a.Hk);
  const int NC = a.NC;

  auto issue_loads = [&](int c) {
    uint8_t* st = sm + (c & 1) * kStage;
    const uint8_t* ub = unit_base(a, b, h, c);
    uint64_t* bar = &full[c & 1];
    mbar_arrive_expect_tx(bar, kStageTx);
    bulk_load(st + kStW0, ub, 8192, bar);
    bulk_load(st + kStW1, ub + 8192, 8192, bar);
    bulk_load(st + kStPh, ub + kUnitP, kPBytes, bar);
    bulk_load(st + kStU, ub + kUnitU + sl * 16384, 16384, bar);
    bulk_load(st + kStS, ub + kUnitS, kSCopy, bar);
    tma_load_4d(st + kStQ0, &tm_q, bar, 0, hk, c * 64, b);
    tma_load_4d(st + kStQ1, &tm_q, bar, 64, hk, c * 64, b);
    tma_load_4d(st + kStK0, &tm_k, bar, 0, hk, c * 64, b);
    tma_load_4d(st + kStK1, &tm_k, bar, 64, hk, c * 64, b);
  };

  if (tid == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (tid == 0) issue_loads(0);

  // State slice: thread kr owns key row kr, value columns [64 sl, 64 sl + 64), float32.
  const int kr = tid;
  float Sm[64];
  {
    const float* s0 = a.S0 ? a.S0 + (((size_t)b * a.Hv + h) * kD + kr) * kD + sl * 64 : nullptr;
#pragma unroll
    for (int n = 0; n < 64; n += 4) {
      float4 x = s0 ? __ldg(reinterpret_cast<const float4*>(s0 + n)) : make_float4(0.f, 0.f, 0.f, 0.f);
      Sm[n] = x.x; Sm[n + 1] = x.y; Sm[n + 2] = x.z; Sm[n + 3] = x.w;
    }
  }
  // bf16 state operand: MN-major (rows = key index, 64 value columns per 128-byte row)
  auto write_state_operand = [&]() {
    uint8_t* row = sm + kOffSb + kr * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint4 pk = make_uint4(pack_bf16x2(Sm[ch * 8 + 0], Sm[ch * 8 + 1]), pack_bf16x2(Sm[ch * 8 + 2], Sm[ch * 8 + 3]),
                            pack_bf16x2(Sm[ch * 8 + 4], Sm[ch * 8 + 5]), pack_bf16x2(Sm[ch * 8 + 6], Sm[ch * 8 + 7]));
      *reinterpret_cast<uint4*>(row + ((ch ^ (kr & 7)) << 4)) = pk;
    }
  };
  write_state_operand();
  fence_async_smem();
  __syncthreads();

  bool ok = true;
  const int i = tid & 63;   // chunk position for the row-per-position phases
  for (int c = 0; c < NC; ++c) {
    uint8_t* st = sm + (c & 1) * kStage;
    if (tid == 0 && c + 1 < NC) issue_loads(c + 1);
    ok = mbar_wait(&full[c & 1], (c >> 1) & 1, kWaitBudget);
    if (!__syncthreads_and(ok)) goto fail;

    // MMA_A: D[:, 0:64] = [W; Q] S   (rows 0-63 W S, rows 64-127 Q S)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, false, true);
      const uint32_t sb = smem_u32(sm + kOffSb);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aa = smem_u32(st) + (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tb, smem_desc(aa, 16, 1024), smem_desc(sb + kk * 2048, 8192, 1024), idesc, kk > 0);
      }
      mma_commit(&bar_mma);
    }
    ok = mbar_wait(&bar_mma, 0, kWaitBudget);
    if (!__syncthreads_and(ok)) goto fail;
    tc_fence_after();

    const float* sc = reinterpret_cast<const float*>(st + kStS);
    float qs[64];
    if (tid < 64) {
      // Vnew row i = U_i - (W S)_i ; Vs = sk_i Vnew (state operand), Vu = Vnew (output operand),
      // each as bf16 hi + lo rows of the MN-major B operands
      float ws_[64];
      tmem_ld32(tb + lane_base, ws_);
      tmem_ld32(tb + lane_base + 32, ws_ + 32);
      const float sk = sc[64 + i];
      const uint8_t* urow = st + kStU + i * 256;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const float4 u0 = *reinterpret_cast<const float4*>(urow + (((2 * ch) ^ (i & 7)) << 4));
        const float4 u1 = *reinterpret_cast<const float4*>(urow + (((2 * ch + 1) ^ (i & 7)) << 4));
        const float un[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        uint32_t vsh[4], vsl[4], vuh[4], vul[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v0 = un[2 * e] - ws_[ch * 8 + 2 * e];
          const float v1 = un[2 * e + 1] - ws_[ch * 8 + 2 * e + 1];
          split_bf16x2(sk * v0, sk * v1, vsh[e], vsl[e]);
          split_bf16x2(v0, v1, vuh[e], vul[e]);
        }
        const uint32_t off = i * 128 + ((ch ^ (i & 7)) << 4);
        *reinterpret_cast<uint4*>(sm + kOffVsh + off) = make_uint4(vsh[0], vsh[1], vsh[2], vsh[3]);
        *reinterpret_cast<uint4*>(sm + kOffVsl + off) = make_uint4(vsl[0], vsl[1], vsl[2], vsl[3]);
        *reinterpret_cast<uint4*>(sm + kOffVuh + off) = make_uint4(vuh[0], vuh[1], vuh[2], vuh[3]);
        *reinterpret_cast<uint4*>(sm + kOffVul + off) = make_uint4(vul[0], vul[1], vul[2], vul[3]);
      }
    } else {
      tmem_ld32(tb + lane_base, qs);
      tmem_ld32(tb + lane_base + 32, qs + 32);
      const float sq = sc[i];
#pragma unroll
      for (int n = 0; n < 64; ++n) qs[n] *= sq;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // MMA2: D[:, 64:128] = K^T (Vs_hi + Vs_lo)  (state increment)
    // MMA3: D[64:128, 128:192] = P_hi Vu_hi + P_hi Vu_lo + P_lo Vu_hi  (intra-chunk output)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id2 = idesc_bf16(128, 64, true, true);
      const uint32_t id3 = idesc_bf16(128, 64, false, true);
      const uint32_t kt = smem_u32(st + kStK0);
      const uint32_t vsh = smem_u32(sm + kOffVsh), vsl = smem_u32(sm + kOffVsl);
      const uint32_t vuh = smem_u32(sm + kOffVuh), vul = smem_u32(sm + kOffVul);
      const uint32_t ph = smem_u32(st + kStQ1), pl = smem_u32(st + kStPh);   // rows 64-127 = P_hi / P_lo
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tb + 64, smem_desc(kt + kk * 2048, 8192, 1024), smem_desc(vsh + kk * 2048, 8192, 1024), id2, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tb + 64, smem_desc(kt + kk * 2048, 8192, 1024), smem_desc(vsl + kk * 2048, 8192, 1024), id2, 1);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tb + 128, smem_desc(ph + kk * 32, 16, 1024), smem_desc(vuh + kk * 2048, 8192, 1024), id3, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tb + 128, smem_desc(ph + kk * 32, 16, 1024), smem_desc(vul + kk * 2048, 8192, 1024), id3, 1);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tb + 128, smem_desc(pl + kk * 32, 16, 1024), smem_desc(vuh + kk * 2048, 8192, 1024), id3, 1);
      mma_commit(&bar_mma);
    }
    ok = mbar_wait(&bar_mma, 1, kWaitBudget);
    if (!__syncthreads_and(ok)) goto fail;
    tc_fence_after();

    {
      // S = Gamma_C S + X (this thread's key row), then the bf16 operand for the next chunk
      const float gc = sc[128];
      float x[32];
      tmem_ld32(tb + lane_base + 64, x);
#pragma unroll
      for (int n = 0; n < 32; ++n) Sm[n] = fmaf(gc, Sm[n], x[n]);
      tmem_ld32(tb + lane_base + 96, x);
#pragma unroll
      for (int n = 0; n < 32; ++n) Sm[32 + n] = fmaf(gc, Sm[32 + n], x[n]);
      write_state_operand();
    }
    if (tid >= 64) {
      // o row i = sq_i (Q S)_i + (P Vnew)_i
      const int p = c * 64 + i;
      float pv[32];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        tmem_ld32(tb + lane_base + 128 + part * 32, pv);
        if (p < a.L) {
          __nv_bfloat16* orow = a.o + (((size_t)b * a.L + p) * a.Hv + h) * kD + sl * 64 + part * 32;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int n0 = part * 32 + ch * 8;
            uint4 pk = make_uint4(pack_bf16x2(qs[n0 + 0] + pv[ch * 8 + 0], qs[n0 + 1] + pv[ch * 8 + 1]),
                                  pack_bf16x2(qs[n0 + 2] + pv[ch * 8 + 2], qs[n0 + 3] + pv[ch * 8 + 3]),
                                  pack_bf16x2(qs[n0 + 4] + pv[ch * 8 + 4], qs[n0 + 5] + pv[ch * 8 + 5]),
                                  pack_bf16x2(qs[n0 + 6] + pv[ch * 8 + 6], qs[n0 + 7] + pv[ch * 8 + 7]));
            *reinterpret_cast<uint4*>(orow + ch * 8) = pk;
          }
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
  }

  if (a.S_T) {
    float* dst = a.S_T + (((size_t)b * a.Hv + h) * kD + kr) * kD + sl * 64;
#pragma unroll
    for (int n = 0; n < 64; n += 4)
      *reinterpret_cast<float4*>(dst + n) = make_float4(Sm[n], Sm[n + 1], Sm[n + 2], Sm[n + 3]);
  }
  goto done;
fail:
  if (tid == 0) set_error(a.err, kErrTimeout);
done:
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 256);
  }
}

// -------------------------------------------------------------------------------------------
// Host side
// -------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [B, L, H, 128] bf16 tensor, box {64 columns, 1 head, 64 positions, 1 row}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int B, int L, int H) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2, (cuuint64_t)L * H * kD * 2};
  cuuint32_t box[4] = {64, 1, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t chunk_workspace_bytes(int B, int L, int Hv) {
  const size_t NC = (size_t)(L + kChunk - 1) / kChunk;
  return (size_t)B * Hv * NC * kUnitBytes + 1024;
}

cudaError_t launch_chunk_bf16(const ChunkLaunch& p, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.B, p.L, p.Hk) || !make_map(&mk, p.k, p.B, p.L, p.Hk) ||
      !make_map(&mv, p.v, p.B, p.L, p.Hv))
    return cudaErrorInvalidValue;
  ChunkArgs a;
  a.g = p.g;
  a.beta = p.beta;
  a.S0 = p.S0;
  a.o = static_cast<__nv_bfloat16*>(p.o);
  a.S_T = p.S_T;
  a.ws = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p.ws) + 1023) & ~uintptr_t(1023));
  a.B = p.B;
  a.L = p.L;
  a.Hk = p.Hk;
  a.Hv = p.Hv;
  a.NC = (p.L + kChunk - 1) / kChunk;
  a.err = p.err;

  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
    cudaFuncSetAttribute(chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStateSmem);
    attr_set = true;
  }
  int slot = stage_timer_begin(s, kKernChunkPrep);
  chunk_prep_kernel<<<dim3(a.NC, p.Hk, p.B), kPrepThreads, kPrepSmem, s>>>(mq, mk, mv, a);
  stage_timer_end(slot, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  slot = stage_timer_begin(s, kKernChunkState);
  chunk_state_kernel<<<dim3(kD / 64, p.Hv, p.B), kStateThreads, kStateSmem, s>>>(mq, mk, a);
  stage_timer_end(slot, s);
  return cudaGetLastError();
}

}  // namespace gdr

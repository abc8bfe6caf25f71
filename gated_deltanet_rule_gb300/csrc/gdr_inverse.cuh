// The unit lower triangular inverse of the chunk algebra, T = (I + A)^-1 for 64 x 64 A, shared by
// the forward's prep kernel and the chunked backward.
#pragma once

#include "ptx.cuh"

namespace gdr {
namespace {
using namespace ptx;

// T = (I + A)^-1 for the strictly lower 64 x 64 A in AT (row stride 68, 1 on the diagonal), by
// recursive doubling: 16 x 16 diagonal blocks by forward substitution, then the merges
// T_BL = -T_BR (A_BL T_TL) for the 16-blocks (1,0), (3,2) and for the 32-block (1,0). T is written
// twice: transposed into AT's strictly upper part (T(i, j) = AT[j][i], a column of T is a row of
// AT) and row-major into Tm, whose diagonal is 1 and upper part 0 on entry. Entries of A are
// zeroed once consumed, so that a row of AT restricted to a finished diagonal block is exactly a
// column of T. Block products read rows of the left factor and columns of the right factor as
// contiguous float4 runs, and skip the blocks that are zero by triangularity. At least 256 threads
// (warps 8 and up only run side(tid) and the barriers); while warps 0 and 1 invert the diagonal
// blocks, the others run side(tid).
template <typename SideWork>
__device__ __forceinline__ void invert_unit_lower(float* AT, float* Tm, float* Xs, int tid, SideWork side) {
  const int warp = tid >> 5, lane = tid & 31;
  // 1. diagonal 16-blocks (warps 0, 1): thread = (block, column c), computing column c of the
  //    block's inverse in registers, left-looking: x_i = -sum_{j < i} A_ij x_j for rows i > c (x_c = 1,
  //    x_j = 0 above it). Each row of A is read as four float4 broadcasts; no shuffles.
  if (warp < 2) {
    const int r0 = (tid >> 4) * 16, c = tid & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      const float4* arow = reinterpret_cast<const float4*>(AT + (r0 + i) * 68 + r0);
      float av[16];
#pragma unroll
      for (int m4 = 0; m4 < 4; ++m4) {
        if (4 * m4 < i) {
          const float4 t = arow[m4];
          av[4 * m4] = t.x; av[4 * m4 + 1] = t.y; av[4 * m4 + 2] = t.z; av[4 * m4 + 3] = t.w;
        }
      }
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < i; ++j) {
        if (j & 1) s1 = fmaf(av[j], x[j], s1);
        else s0 = fmaf(av[j], x[j], s0);
      }
      x[i] = (i > c) ? -(s0 + s1) : x[i];
    }
    __syncwarp();   // every lane of the block has read A's rows before row c of AT is overwritten
    // column c of T: Tm rows below the diagonal (its diagonal 1 and upper zeros are in place), and
    // AT row c over the block's columns: 0 above the diagonal of T (the consumed A), 1 on it, T below
#pragma unroll
    for (int i = 1; i < 16; ++i)
      if (i > c) Tm[(r0 + i) * 68 + r0 + c] = x[i];
    float4* trow = reinterpret_cast<float4*>(AT + (r0 + c) * 68 + r0);
#pragma unroll
    for (int m4 = 0; m4 < 4; ++m4)
      trow[m4] = make_float4(x[4 * m4], x[4 * m4 + 1], x[4 * m4 + 2], x[4 * m4 + 3]);
  } else {
    side(tid);   // warps 2-7 meanwhile: the caller's work that does not touch AT, Tm or Xs
  }
  __syncthreads();
  // 2. 16-block merges p = 0, 1 (TL = [32p, 32p+16), BR = [32p+16, 32p+32)) with the same warp-level
  //    products: warp w < 4 forms the 16 x 8 tile (merge p = w >> 1, columns 8 (w & 1)) of
  //    X = A_BL T_TL (stored transposed, Xs[p][j][i]) and then of T_BL = -T_BR X (into Tm and AT).
  if (warp < 4) {
    const int g = lane >> 2, t = lane & 3, p = warp >> 1, n = warp & 1, base = 32 * p;
    float dh[4] = {0.f, 0.f, 0.f, 0.f}, dc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      if (kk < n) continue;
      const float* ar = AT + (base + 16 + g) * 68 + base + 8 * kk + t;   // A_BL(i, k)
      const float* br = AT + (base + 8 * n + g) * 68 + base + 8 * kk + t;   // T_TL(k, j) = AT[j][k]
      const float a4[4] = {ar[0], ar[8 * 68], ar[4], ar[8 * 68 + 4]};
      const float b2[2] = {br[0], br[4]};
      mma_3xtf32(dh, dc, a4, b2);
    }
    const int j0 = 8 * n + 2 * t;
    Xs[(p * 16 + j0) * 20 + g] = dh[0] + dc[0];
    Xs[(p * 16 + j0 + 1) * 20 + g] = dh[1] + dc[1];
    Xs[(p * 16 + j0) * 20 + g + 8] = dh[2] + dc[2];
    Xs[(p * 16 + j0 + 1) * 20 + g + 8] = dh[3] + dc[3];
  }
  __syncthreads();
  if (warp < 4) {
    {   // A_BL consumed: a row of AT restricted to a finished 32-block is then exactly a column of T
      const int p = lane >> 4, i = lane & 15, base = 32 * p;
      reinterpret_cast<float4*>(AT + (base + 16 + i) * 68 + base)[warp] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int g = lane >> 2, t = lane & 3, p = warp >> 1, n = warp & 1, base = 32 * p;
    float dh[4] = {0.f, 0.f, 0.f, 0.f}, dc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const float* ar = Tm + (base + 16 + g) * 68 + base + 16 + 8 * kk + t;   // T_BR(i, k), row-major
      const float* br = Xs + (p * 16 + 8 * n + g) * 20 + 8 * kk + t;         // X(k, j) = Xs[p][j][k]
      const float a4[4] = {ar[0], ar[8 * 68], ar[4], ar[8 * 68 + 4]};
      const float b2[2] = {br[0], br[4]};
      mma_3xtf32(dh, dc, a4, b2);
    }
    const int j0 = 8 * n + 2 * t;
    const float r[4] = {-(dh[0] + dc[0]), -(dh[1] + dc[1]), -(dh[2] + dc[2]), -(dh[3] + dc[3])};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = base + 16 + g + 8 * (e >> 1), j = base + j0 + (e & 1);
      Tm[i * 68 + j] = r[e];
      AT[j * 68 + i] = r[e];
    }
  }
  __syncthreads();
  // 3. 32-block merge on the tensor cores with warp-level products at fp32 accuracy (3xTF32): warp w
  //    forms the 16 x 8 tile (rows 16 (w & 1), columns 8 (w >> 1)) of X = A_BL T_TL, stored
  //    transposed (Xs[j][i]), then of T_BL = -T_BR X into AT's upper part. Zero blocks of the
  //    triangular factors are skipped (T_TL: k-blocks below the column block; T_BR: above the row block).
  if (warp < 8) {   // (a block of more than eight warps leaves the rest idle here)
    const int g = lane >> 2, t = lane & 3, m = warp & 1, n = warp >> 1;
    float dh[4] = {0.f, 0.f, 0.f, 0.f}, dc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (kk < n) continue;
      const float* ar = AT + (32 + 16 * m + g) * 68 + 8 * kk + t;   // A_BL(i, k) = A(32 + i, k)
      const float* br = AT + (8 * n + g) * 68 + 8 * kk + t;          // T_TL(k, j) = AT[j][k]
      const float a4[4] = {ar[0], ar[8 * 68], ar[4], ar[8 * 68 + 4]};
      const float b2[2] = {br[0], br[4]};
      mma_3xtf32(dh, dc, a4, b2);
    }
    const int i0 = 16 * m + g, j0 = 8 * n + 2 * t;
    Xs[j0 * 36 + i0] = dh[0] + dc[0];
    Xs[(j0 + 1) * 36 + i0] = dh[1] + dc[1];
    Xs[j0 * 36 + i0 + 8] = dh[2] + dc[2];
    Xs[(j0 + 1) * 36 + i0 + 8] = dh[3] + dc[3];
  }
  __syncthreads();
  if (warp < 8) {
    const int g = lane >> 2, t = lane & 3, m = warp & 1, n = warp >> 1;
    float dh[4] = {0.f, 0.f, 0.f, 0.f}, dc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (kk > 2 * m + 1) continue;
      const float* ar = Tm + (32 + 16 * m + g) * 68 + 32 + 8 * kk + t;   // T_BR(i, k), row-major
      const float* br = Xs + (8 * n + g) * 36 + 8 * kk + t;              // X(k, j) = Xs[j][k]
      const float a4[4] = {ar[0], ar[8 * 68], ar[4], ar[8 * 68 + 4]};
      const float b2[2] = {br[0], br[4]};
      mma_3xtf32(dh, dc, a4, b2);
    }
    const int i0 = 16 * m + g, j0 = 8 * n + 2 * t;   // T(32 + i, j) = AT[j][32 + i]
    AT[j0 * 68 + 32 + i0] = -(dh[0] + dc[0]);
    AT[(j0 + 1) * 68 + 32 + i0] = -(dh[1] + dc[1]);
    AT[j0 * 68 + 32 + i0 + 8] = -(dh[2] + dc[2]);
    AT[(j0 + 1) * 68 + 32 + i0 + 8] = -(dh[3] + dc[3]);
  }
  __syncthreads();
}

}  // namespace
}  // namespace gdr

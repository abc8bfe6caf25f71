// Chunked backward of the gated delta rule, bf16 rows: the chunk-local gradients and the key-head
// reduction. The sequential passes (the forward's chunk factors, the chunk-entry states S_c, Nb =
// Q'^T dO and the adjoint chain) run in gdr_chunk.cu (launch_chunk_bwd_chain); what is left is
// local to each (row, value head, chunk) unit once S_c and the adjoint dS' of the chunk's exiting
// state are known.
//
// The pages train through the recurrence but print no backward. With the chunk algebra of the
// forward (per 64-token chunk, entering state S: A_ij = beta_i (k^_i . k^_j) E_ij for j < i with
// E_ij = e^{gamma_i - gamma_j}, T = (I + A)^-1, W = T diag(beta Gamma) K^, U = T diag(beta) V,
// Delta = U - W S, P_ij = (q~_i . k^_j) E_ij for j <= i, O = diag(Gamma) Q~ S + P Delta,
// S' = Gamma_C S + K^T diag(e) Delta with e_i = e^{gamma_C - gamma_i}), the reverse given dO and
// dS' is, per chunk:
//   dDelta = P^T dO + diag(e) K^ dS',  dW = -dDelta S^T,  dP = dO Delta^T (j <= i)
//   dQ~ = diag(Gamma) dO S^T + (dP o E) K^
//   dK^ = (dP o E)^T Q~ + diag(e) Delta dS'^T + diag(beta Gamma) T^T dW + (dA~ + dA~^T) K^
//   dT = dDelta (diag(beta) V)^T + dW (diag(beta Gamma) K^)^T,  dA = -T^T dT T^T (j < i),
//   dA~ = dA o beta_i E,  dV = diag(beta) T^T dDelta
//   dbeta_i = V_i . (T^T dDelta)_i + Gamma_i K^_i . (T^T dW)_i + sum_j dA_ij (k^_i . k^_j) E_ij
//   dgamma_i = Gamma_i q~_i . (dO S^T)_i + rows - columns of (dP o P) and (dA o A)
//              + beta_i Gamma_i K^_i . (T^T dW)_i - e_i k^_i . (dS' Delta_i)
//              (+ Gamma_C <S, dS'> + sum_j e_j k^_j . (dS' Delta_j) at the chunk's last position)
//   dg_j = sum_{i >= j} dgamma_i within the chunk
// then the normalisations' backward and the sum over the value heads of a key head.
//
// Products run on warp-level tensor-core instructions (mma.sync m16n8k16, fp32 accumulation):
// they are 64-row products of K = 64 or 128, a dozen per unit, each feeding an elementwise
// epilogue, with both operands already in shared memory. The raw bf16 q, k enter the Gram
// products exactly (bf16 operands); every other operand is fp16, divided by the power of two of its
// tile's largest magnitude where that magnitude is not bounded (v, dO, S, dS', Delta and the
// gradients), the scales applied back in fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gdr_backward.h"
#include "gdr_internal.h"
#include "gdr_inverse.cuh"
#include "ptx.cuh"

namespace gdr {
namespace {
using namespace ptx;

constexpr int kLT = 512;                         // threads of the chunk-local kernel (16 warps)
constexpr int kLd = 136;                         // row stride (halves) of 128-column fp16 tiles
constexpr int kLs = 72;                          // row stride (halves) of 64-column fp16 tiles
constexpr int kLf = 68;                          // row stride (floats) of the fp32 64 x 64 tile
constexpr float kQs = 0.08838834764831845f;      // 128^-0.5
constexpr float kL2e = 1.4426950408889634f;
constexpr int kStateSlices = 4;                  // 32-column slices of a saved state, one scale each

constexpr uint32_t kT128 = 64 * kLd * 2;         // a 64 x 128 fp16 tile
constexpr uint32_t kT128x = 128 * kLd * 2;       // a 128 x 128 fp16 tile
constexpr uint32_t kT64 = 64 * kLs * 2;          // a 64 x 64 fp16 tile
constexpr uint32_t kOQ = 0;                      // q (bf16, then the fp16 unit rows q^)
constexpr uint32_t kOK = kOQ + kT128;            // k (bf16, then k^)
constexpr uint32_t kOV = kOK + kT128;            // v / 2^eV
constexpr uint32_t kOO = kOV + kT128;            // dO / 2^eO
constexpr uint32_t kOS = kOO + kT128;            // S / 2^eS [key][value]; later dPE, dT, Z
constexpr uint32_t kODS = kOS + kT128x;          // dS' / 2^eD; later dW, dA~
constexpr uint32_t kOX1 = kODS + kT128x;         // beta Gamma K^, beta V, then Delta
constexpr uint32_t kOX2 = kOX1 + kT128;          // W, then dDelta
constexpr uint32_t kOTf = kOX2 + kT128;          // fp32 A (strictly lower)
constexpr uint32_t kOT16 = kOTf + 64 * kLf * 4;  // T (fp16)
constexpr uint32_t kOP16 = kOT16 + kT64;         // P (fp16)
constexpr uint32_t kOVec = kOP16 + kT64;         // per-position vectors and reduction scratch
constexpr int kNVec = 26;
constexpr uint32_t kLocalSmem = kOVec + kNVec * 64 * 4;
// vectors (64 floats each)
enum : int { vG2 = 0, vGam, vE, vBet, vSq, vSk, vRowG0, vRowB0 = vRowG0 + 4, vRowD0 = vRowB0 + 4,
             vColG0 = vRowD0 + 4, vMax = vColG0 + 4, vDot, vScan };

__device__ __forceinline__ void pow2_up_dn(float m, float& up, float& dn) {
  // up = 2^e with m / up in [0.5, 1) (1 for m = 0), dn = 1 / up, e clamped to keep both normal
  const int eb = (int)((__float_as_uint(m) >> 23) & 0xFFu);
  int e = eb == 0 ? 0 : eb - 126;
  e = e < -125 ? -125 : (e > 125 ? 125 : e);
  up = __uint_as_float((uint32_t)(127 + e) << 23);
  dn = __uint_as_float((uint32_t)(127 - e) << 23);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
template <bool kBf>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if (kBf)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc (16 rows from m0, 8 NT columns from n0) += A B over K. A: 64 x K, stored [row][K] (AT false)
// or [K][row] (AT true: the product uses the transpose of the stored tile). B: K x N, stored
// [K][N] (BT false) or [N][K] (BT true). Strides in 16-bit elements. The fragment this thread
// holds: rows m0 + g and m0 + g + 8, columns n0 + 8 nt + 2 t and + 1 (g = lane / 4, t = lane % 4).
template <int NT, bool AT, bool BT, bool kBf = false>
__device__ __forceinline__ void tile_mma(float (&acc)[NT][4], const uint8_t* A, int lda, int m0, const uint8_t* B,
                                         int ldb, int n0, int K, int lane) {
  const uint16_t* a16 = reinterpret_cast<const uint16_t*>(A);
  const uint16_t* b16 = reinterpret_cast<const uint16_t*>(B);
#pragma unroll 2   // (K is a multiple of 32: two steps' fragment loads overlap, and fewer registers spill)
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t af[4];
    if (!AT)
      ldsm_x4(af, a16 + (m0 + (lane & 15)) * lda + k0 + 8 * (lane >> 4));
    else
      ldsm_x4_t(af, a16 + (k0 + (lane & 7) + 8 * (lane >> 4)) * lda + m0 + 8 * ((lane >> 3) & 1));
#pragma unroll
    for (int nt = 0; nt < NT; nt += 2) {
      uint32_t bf[4];
      if (!BT)
        ldsm_x4_t(bf, b16 + (k0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * ldb + n0 + 8 * nt + 8 * (lane >> 4));
      else
        ldsm_x4(bf, b16 + (n0 + 8 * nt + (lane & 7) + 8 * (lane >> 4)) * ldb + k0 + 8 * ((lane >> 3) & 1));
      mma16816<kBf>(acc[nt], af, bf[0], bf[1]);
      mma16816<kBf>(acc[nt + 1], af, bf[2], bf[3]);
    }
  }
}

template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
}
template <int NT>
__device__ __forceinline__ float absmax(const float (&acc)[NT][4]) {
  float m = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(acc[nt][e]));
  return m;
}
__device__ __forceinline__ float h2f(const uint8_t* tile, int ld, int r, int c) {
  return __half2float(reinterpret_cast<const __half*>(tile)[r * ld + c]);
}
// fragment element (row, column) of acc[nt][e]
__device__ __forceinline__ int frow(int m0, int lane, int e) { return m0 + (lane >> 2) + 8 * (e >> 1); }
__device__ __forceinline__ int fcol(int n0, int lane, int nt, int e) { return n0 + 8 * nt + 2 * (lane & 3) + (e & 1); }

// store a fragment as fp16 (times s) into a tile with stride ld
template <int NT>
__device__ __forceinline__ void store_h(uint8_t* tile, int ld, int m0, int n0, const float (&acc)[NT][4], float s,
                                        int lane) {
  __half* t = reinterpret_cast<__half*>(tile);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = frow(m0, lane, 2 * hh), c = fcol(n0, lane, nt, 0);
      *reinterpret_cast<__half2*>(t + r * ld + c) = __floats2half2_rn(acc[nt][2 * hh] * s, acc[nt][2 * hh + 1] * s);
    }
}

// CTA-wide max of a per-thread value (every thread gets it), with one block barrier (which also
// orders everything before the call against everything after it). The per-warp maxima alternate
// between vec[vMax][0..15] and [32..47] from one call to the next (par, the same in every thread):
// a buffer is rewritten two calls later, after the intervening call's barrier has passed every
// reader of it.
__device__ __forceinline__ float cta_max(float m, float* vmax, int warp, int lane, int& par) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float* buf = vmax + 32 * par;
  par ^= 1;
  if (lane == 0) buf[warp] = m;
  __syncthreads();
  float r = buf[0];
#pragma unroll
  for (int w = 1; w < kLT / 32; ++w) r = fmaxf(r, buf[w]);
  return r;
}

struct LocalArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  const __nv_bfloat16* dO;
  const __half* S_save;   // per unit four 32-column slice images (fp16, each over its S_scale [B, Hv, NC, 4])
  const float* S_scale;
  const __half* dS_save;  // likewise for the adjoints
  const float* dS_scale;
  const float* unit_scale;   // [B, Hv, NC, 8]: the powers of two of dO's four slices, then of v
  float* dq;              // [B, L, Hk, D]
  float* dk;
  float* dv;
  float* dg;
  float* dbeta;
  int B, L, Hk, Hv, NC;
};

// One CTA per (row, value head, chunk) unit. Warp w owns rows 16 (w % 4) .. + 15 of every 64-row
// product and the column quarter w / 4 (32 columns of a 128-column product, 16 of a 64-column one).
__device__ __forceinline__ void local_unit(const LocalArgs& a, uint8_t* sm, const int u) {
  float* vec = reinterpret_cast<float*>(sm + kOVec);
  auto V = [&](int i) { return vec + i * 64; };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = u % a.NC, hk = (u / a.NC) % a.Hk, b = u / (a.NC * a.Hk);
  const int r = a.Hv / a.Hk;
  const int m0 = 16 * (warp & 3), quarter = warp >> 2;
  const int n128 = 32 * quarter, n64 = 16 * quarter;
  const int p0 = c * kChunk;   // first position of the chunk
  int mpar = 0;                // cta_max's buffer parity
  uint8_t* tQ = sm + kOQ;
  uint8_t* tK = sm + kOK;
  uint8_t* tV = sm + kOV;
  uint8_t* tO = sm + kOO;
  uint8_t* tS = sm + kOS;
  uint8_t* tD = sm + kODS;
  uint8_t* tX1 = sm + kOX1;
  uint8_t* tX2 = sm + kOX2;
  float* Af = reinterpret_cast<float*>(sm + kOTf);
  uint8_t* tT = sm + kOT16;
  uint8_t* tP = sm + kOP16;

  // a value head's v and dO rows (zero past L) and its S and dS' (four 32-column slice images of 128
  // key rows x 64 bytes, 64-byte swizzle, each) into their tiles, as one group of asynchronous copies
  auto issue_head = [&](int h) {
#pragma unroll
    for (int it = 0; it < 2 * 1024 / kLT; ++it) {
      const int idx = tid + kLT * it;
      const int which = idx >> 10, row = (idx >> 4) & 63, ch = idx & 15;
      const int pos = p0 + row;
      const size_t ro = pos < a.L ? (((size_t)b * a.L + pos) * a.Hv + h) * kD : 0;
      cp_async16_zfill((which ? tO : tV) + row * kLd * 2 + ch * 16,
                       reinterpret_cast<const uint4*>((which ? a.dO : a.v) + ro) + ch, pos < a.L ? 16 : 0);
    }
    const size_t unit = ((size_t)b * a.Hv + h) * a.NC + c;
#pragma unroll
    for (int it = 0; it < 2 * 2048 / kLT; ++it) {
      const int idx = tid + kLT * it;
      const int which = idx >> 11, row = (idx >> 4) & 127, ch = idx & 15;
      const uint8_t* src = reinterpret_cast<const uint8_t*>(which ? a.dS_save : a.S_save) + unit * (kD * kD * 2) +
                           (ch >> 2) * 8192 + swz64(row * 64 + (ch & 3) * 16);
      cp_async16_zfill((which ? tD : tS) + row * kLd * 2 + ch * 16, src, 16);
    }
    cp_async_commit();
  };
  // the same inputs of a later value head into L2 only (the tiles are still in use)
  auto prefetch_head = [&](int h) {
    if (tid < 128) {
      const int pos = p0 + (tid & 63);
      if (pos < a.L)
        bulk_prefetch_l2(((tid < 64 ? a.v : a.dO) + (((size_t)b * a.L + pos) * a.Hv + h) * kD), kD * 2);
    } else if (tid < 136) {
      const size_t unit = ((size_t)b * a.Hv + h) * a.NC + c;
      const int piece = tid - 128;   // 8 KB pieces: S's four slices, then dS''s
      bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(piece < 4 ? a.S_save : a.dS_save) + unit * (kD * kD * 2) +
                       (piece & 3) * 8192, 8192);
    }
  };

  // ---- prologue (once per key head): raw q, k rows, their inverse norms, the Gram products
  //      K K^T and Q K^T from the raw bf16 rows (kept in registers: every value head's A and P are
  //      elementwise in them), then q^ = q / |q|, k^ = k / |k| as fp16 (q~ = q^ 128^-0.5) ----
#pragma unroll
  for (int it = 0; it < 2 * 1024 / kLT; ++it) {
    const int idx = tid + kLT * it;
    const int which = idx >> 10, row = (idx >> 4) & 63, ch = idx & 15;
    const int pos = p0 + row;
    const size_t ro = pos < a.L ? (((size_t)b * a.L + pos) * a.Hk + hk) * kD : 0;
    cp_async16_zfill((which ? tK : tQ) + row * kLd * 2 + ch * 16,
                     reinterpret_cast<const uint4*>((which ? a.k : a.q) + ro) + ch, pos < a.L ? 16 : 0);
  }
  cp_async_commit();
  issue_head(hk * r);   // the first value head's inputs load while q and k are prepared
  cp_async_wait<1>();   // q and k have landed
  __syncthreads();
  if (tid < 128) {
    // inverse norms of the raw q, k rows (threads 0-63: q, 64-127: k)
    const int row = tid & 63;
    const uint8_t* src = (tid < 64 ? tQ : tK) + row * kLd * 2;
    float s0 = 0.f;
#pragma unroll
    for (int ch = 0; ch < 16; ++ch) {
      const uint4 w = *reinterpret_cast<const uint4*>(src + ch * 16);
      const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xFFFF0000u);
        s0 = fmaf(lo, lo, fmaf(hi, hi, s0));
      }
    }
    V(tid < 64 ? vSq : vSk)[row] = rsqrtf(s0 + 1e-6f);
  }
  float G[2][4], Gq[2][4];
  zero(G);
  zero(Gq);
  tile_mma<2, false, true, true>(G, tK, kLd, m0, tK, kLd, n64, 128, lane);
  tile_mma<2, false, true, true>(Gq, tQ, kLd, m0, tK, kLd, n64, 128, lane);
  __syncthreads();   // the norms are in; the raw rows are read
  const float* sq = V(vSq);
  const float* sk = V(vSk);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = frow(m0, lane, e), j = fcol(n64, lane, nt, e);
      G[nt][e] *= sk[i] * sk[j];                 // k^_i . k^_j
      Gq[nt][e] *= kQs * sq[i] * sk[j];          // q~_i . k^_j
    }
  for (int idx = tid; idx < 2 * 1024; idx += kLT) {
    const int which = idx >> 10, row = (idx >> 4) & 63, ch = idx & 15;
    uint4* p = reinterpret_cast<uint4*>((which ? tK : tQ) + row * kLd * 2 + ch * 16);
    const float sc = V(which ? vSk : vSq)[row];
    const uint4 w = *p;
    *p = make_uint4(bf16x2_to_f16x2_scaled(w.x, sc), bf16x2_to_f16x2_scaled(w.y, sc),
                    bf16x2_to_f16x2_scaled(w.z, sc), bf16x2_to_f16x2_scaled(w.w, sc));
  }
  float dK[4][4], dQ[4][4];   // summed over the key head's value heads
  zero(dK);
  zero(dQ);

  for (int jh = 0; jh < r; ++jh) {
  const int h = hk * r + jh;
  __syncthreads();   // the previous value head's tiles are spent (and q^, k^ are in)
  if (jh + 1 < r) prefetch_head(h + 1);

  // ---- 0. the value head's inputs: gates, v and dO rows (zero past L), S and dS' (fp16) ----
  if (tid < 64) {
    const int pos = p0 + tid;
    const size_t gi = ((size_t)b * a.L + pos) * a.Hv + h;
    const float gg = pos < a.L ? a.g[gi] : 0.f;
    V(vBet)[tid] = pos < a.L ? a.beta[gi] : 0.f;
    float x = gg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    V(vScan)[tid] = x;
  }
  if (jh > 0) issue_head(h);   // (the first value head's inputs were issued with q and k)
  cp_async_wait<0>();
  __syncthreads();
  if (tid < 64) {
    const float gam = V(vScan)[tid] + (tid >= 32 ? V(vScan)[31] : 0.f);
    V(vG2)[tid] = gam * kL2e;
  }
  __syncthreads();
  if (tid < 64) {
    V(vGam)[tid] = exp2f(V(vG2)[tid]);
    V(vE)[tid] = exp2f(V(vG2)[63] - V(vG2)[tid]);
  }
  __syncthreads();   // the decays are in

  // per-thread partial sums: rows (this warp's column quarter, unshuffled) and columns of the 64 x 64
  // products (this thread's two rows)
  float rg[2] = {0.f, 0.f}, rb[2] = {0.f, 0.f}, rd[2] = {0.f, 0.f}, cg[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) cg[i] = 0.f;
  const float* gam2 = V(vG2);
  const float* Gam = V(vGam);
  const float* ev = V(vE);
  const float* bet = V(vBet);
  auto Eij = [&](int i, int j) { return exp2f(gam2[i] - gam2[j]); };   // j <= i only

  // ---- 1. A (fp32, 1 on the diagonal) and P (fp16) from the Gram products ----
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = frow(m0, lane, e), j = fcol(n64, lane, nt, e);
      const float E = j <= i ? Eij(i, j) : 0.f;
      Af[i * kLf + j] = j < i ? bet[i] * G[nt][e] * E : (j == i ? 1.f : 0.f);
      reinterpret_cast<__half*>(tP)[i * kLs + j] = __float2half_rn(Gq[nt][e] * E);
    }
  // v's and dO's powers of two (taken by the prep and adjoint-chain kernels over the same tiles: dO's
  // is the largest of its four slices'); S and dS' to one power of two per tile (their slices'
  // largest), <S, dS'>
  float dot = 0.f;
  float upV, dnV, upO, dnO;
  {
    const float* us = a.unit_scale + (((size_t)b * a.Hv + h) * a.NC + c) * 8;
    upV = us[4];
    upO = fmaxf(fmaxf(us[0], us[1]), fmaxf(us[2], us[3]));
    dnV = __uint_as_float((254u << 23) - __float_as_uint(upV));   // 1 / 2^e, exact
    dnO = __uint_as_float((254u << 23) - __float_as_uint(upO));
  }
  const size_t unit = ((size_t)b * a.Hv + h) * a.NC + c;
  const float4 scS = *reinterpret_cast<const float4*>(a.S_scale + unit * 4);
  const float4 scD = *reinterpret_cast<const float4*>(a.dS_scale + unit * 4);
  const float upS = fmaxf(fmaxf(scS.x, scS.y), fmaxf(scS.z, scS.w));
  const float upD = fmaxf(fmaxf(scD.x, scD.y), fmaxf(scD.z, scD.w));
  for (int idx = tid; idx < 2048; idx += kLT) {
    const int row = idx >> 4, ch = idx & 15, j = ch >> 2;   // slice j: columns 32 j .. + 31
    const float sj = j == 0 ? scS.x : j == 1 ? scS.y : j == 2 ? scS.z : scS.w;
    const float dj = j == 0 ? scD.x : j == 1 ? scD.y : j == 2 ? scD.z : scD.w;
    __half2* ps = reinterpret_cast<__half2*>(tS + row * kLd * 2 + ch * 16);
    __half2* pd = reinterpret_cast<__half2*>(tD + row * kLd * 2 + ch * 16);
    const float fs = sj / upS, fd = dj / upD;   // powers of two <= 1
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __half22float2(ps[e]), y = __half22float2(pd[e]);
      part = fmaf(x.x, y.x, fmaf(x.y, y.y, part));
      if (fs != 1.f) ps[e] = __floats2half2_rn(x.x * fs, x.y * fs);
      if (fd != 1.f) pd[e] = __floats2half2_rn(y.x * fd, y.y * fd);
    }
    dot = fmaf(part, sj * dj, dot);
  }
  {
    // <S, dS'> over the whole 128 x 128 state (fixed order: warp sums, then warps in order)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) V(vDot)[warp] = dot;
  }
  // v, dO -> fp16 scaled, in place; S, dS' -> fp16 scaled tiles [key][value]
  for (int idx = tid; idx < 1024; idx += kLT) {
    const int row = idx >> 4, ch = idx & 15;
    uint4* pv = reinterpret_cast<uint4*>(tV + row * kLd * 2 + ch * 16);
    uint4* po = reinterpret_cast<uint4*>(tO + row * kLd * 2 + ch * 16);
    const uint4 wv = *pv, wo = *po;
    *pv = make_uint4(bf16x2_to_f16x2_scaled(wv.x, dnV), bf16x2_to_f16x2_scaled(wv.y, dnV),
                     bf16x2_to_f16x2_scaled(wv.z, dnV), bf16x2_to_f16x2_scaled(wv.w, dnV));
    *po = make_uint4(bf16x2_to_f16x2_scaled(wo.x, dnO), bf16x2_to_f16x2_scaled(wo.y, dnO),
                     bf16x2_to_f16x2_scaled(wo.z, dnO), bf16x2_to_f16x2_scaled(wo.w, dnO));
  }
  __syncthreads();

  // ---- 2. T = (I + A)^-1 by recursive doubling (the forward's inverse: fp32-accurate merges), T
  //         row-major in fp32 over X2 with its scratch over T's fp16 tile; meanwhile the operand
  //         diag(beta Gamma) K^ into X1 ----
  {
    float* Tm = reinterpret_cast<float*>(tX2);
    for (int e = tid; e < 64 * 17; e += kLT) {   // Tm starts as the identity
      const int rr = e / 17, c4 = e - rr * 17;
      const int d = ((rr >> 2) == c4) ? (rr & 3) : -1;
      reinterpret_cast<float4*>(Tm + rr * kLf)[c4] =
          make_float4(d == 0 ? 1.f : 0.f, d == 1 ? 1.f : 0.f, d == 2 ? 1.f : 0.f, d == 3 ? 1.f : 0.f);
    }
    __syncthreads();
    invert_unit_lower(Af, Tm, reinterpret_cast<float*>(tT), tid, [&](int t) {
      for (int idx = t - 64; idx < 64 * 64; idx += kLT - 64) {
        const int row = idx >> 6, c2 = idx & 63;
        const float sc = bet[row] * Gam[row];
        const float2 f = __half22float2(reinterpret_cast<const __half2*>(tK + row * kLd * 2)[c2]);
        reinterpret_cast<__half2*>(tX1 + row * kLd * 2)[c2] = __floats2half2_rn(f.x * sc, f.y * sc);
      }
    });
    // T as fp16, row-major (over the inverse's scratch), from its transposed copy in A's upper part:
    // T(i, j) = Af[j][i] below the diagonal, 1 on it
    for (int e = tid; e < 64 * 64; e += kLT) {
      const int i = e >> 6, j = e & 63;
      reinterpret_cast<__half*>(tT)[i * kLs + j] = __float2half_rn(i > j ? Af[j * kLf + i] : (i == j ? 1.f : 0.f));
    }
  }
  __syncthreads();

  // ---- 3. W = T diag(beta Gamma) K^, U = T diag(beta) V, Delta = U - W S ----
  float acc[4][4], acc2[4][4];
  zero(acc);
  tile_mma<4, false, false>(acc, tT, kLs, m0, tX1, kLd, n128, 64, lane);   // W
  store_h(tX2, kLd, m0, n128, acc, 1.f, lane);
  __syncthreads();
  for (int idx = tid; idx < 64 * 64; idx += kLT) {
    const int row = idx >> 6, c2 = idx & 63;
    const float2 f = __half22float2(reinterpret_cast<const __half2*>(tV + row * kLd * 2)[c2]);
    reinterpret_cast<__half2*>(tX1 + row * kLd * 2)[c2] = __floats2half2_rn(f.x * bet[row], f.y * bet[row]);
  }
  __syncthreads();
  zero(acc);
  tile_mma<4, false, false>(acc, tT, kLs, m0, tX1, kLd, n128, 64, lane);    // U / 2^eV
  zero(acc2);
  tile_mma<4, false, false>(acc2, tX2, kLd, m0, tS, kLd, n128, 128, lane);  // W S / 2^eS
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = upV * acc[nt][e] - upS * acc2[nt][e];   // Delta
  float upDl, dnDl;
  pow2_up_dn(cta_max(absmax(acc), V(vMax), warp, lane, mpar), upDl, dnDl);   // (its barriers: X1 is free)
  store_h(tX1, kLd, m0, n128, acc, dnDl, lane);                         // Delta / 2^eDl
  __syncthreads();

  // ---- 4. dDelta = P^T dO + diag(e) K^ dS'; the rows e_i k^_i . (dS' Delta_i) ----
  zero(acc);
  tile_mma<4, true, false>(acc, tP, kLs, m0, tO, kLd, n128, 64, lane);     // P^T dO / 2^eO
  zero(acc2);
  tile_mma<4, false, false>(acc2, tK, kLd, m0, tD, kLd, n128, 128, lane);  // K^ dS' / 2^eD
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = frow(m0, lane, e), col = fcol(n128, lane, nt, e);
      const float kd = upD * acc2[nt][e];
      rd[e >> 1] += ev[i] * kd * (upDl * h2f(tX1, kLd, i, col));
      acc[nt][e] = upO * acc[nt][e] + ev[i] * kd;
    }
  float updD, dndD;
  pow2_up_dn(cta_max(absmax(acc), V(vMax), warp, lane, mpar), updD, dndD);
  store_h(tX2, kLd, m0, n128, acc, dndD, lane);                          // dDelta / 2^edD (W is spent)

  // ---- 5. dK^ += diag(e) Delta dS'^T ----
  zero(acc2);
  tile_mma<4, false, true>(acc2, tX1, kLd, m0, tD, kLd, n128, 128, lane);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) dK[nt][e] += acc2[nt][e] * ev[frow(m0, lane, e)] * upDl * upD;
  __syncthreads();   // dDelta is stored; dS' is read by every warp (its tile is reused below)

  // ---- 6. dW = -dDelta S^T; dQ~ += diag(Gamma) dO S^T; the rows Gamma_i q~_i . (dO S^T)_i ----
  zero(acc);
  tile_mma<4, false, true>(acc, tX2, kLd, m0, tS, kLd, n128, 128, lane);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] *= -updD * upS;
  float updW, dndW;
  pow2_up_dn(cta_max(absmax(acc), V(vMax), warp, lane, mpar), updW, dndW);
  uint8_t* tdW = tD;   // dS' is spent
  store_h(tdW, kLd, m0, n128, acc, dndW, lane);
  zero(acc2);
  tile_mma<4, false, true>(acc2, tO, kLd, m0, tS, kLd, n128, 128, lane);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = frow(m0, lane, e), col = fcol(n128, lane, nt, e);
      const float x = upO * upS * acc2[nt][e];
      rg[e >> 1] += Gam[i] * kQs * h2f(tQ, kLd, i, col) * x;
      dQ[nt][e] += Gam[i] * x;
    }
  __syncthreads();   // S is spent (its tile holds dPE, dT and Z below)

  // ---- 7. dP = dO Delta^T (j <= i); dQ~ += (dP o E) K^, dK^ += (dP o E)^T q~ ----
  uint8_t* tPE = tS;
  uint8_t* tdT = tS + kT64;
  uint8_t* tZ = tS + 2 * kT64;
  uint8_t* tdA = tD + kT128;
  {
    float dp[2][4];
    zero(dp);
    tile_mma<2, false, true>(dp, tO, kLd, m0, tX1, kLd, n64, 128, lane);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = frow(m0, lane, e), j = fcol(n64, lane, nt, e);
        const float d = j <= i ? upO * upDl * dp[nt][e] : 0.f;
        const float pp = d * h2f(tP, kLs, i, j);
        rg[e >> 1] += pp;
        cg[2 * nt + (e & 1)] -= pp;
        dp[nt][e] = j <= i ? d * Eij(i, j) : 0.f;
      }
    float up, dn;
    pow2_up_dn(cta_max(absmax(dp), V(vMax), warp, lane, mpar), up, dn);
    store_h(tPE, kLs, m0, n64, dp, dn, lane);
    __syncthreads();
    float t2[4][4];
    zero(t2);
    tile_mma<4, false, false>(t2, tPE, kLs, m0, tK, kLd, n128, 64, lane);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) dQ[nt][e] += up * t2[nt][e];
    zero(t2);
    tile_mma<4, true, false>(t2, tPE, kLs, m0, tQ, kLd, n128, 64, lane);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) dK[nt][e] += up * kQs * t2[nt][e];
  }

  // ---- 8. T^T dDelta -> dV, dbeta; T^T dW -> dK^, dbeta, dgamma ----
  zero(acc);
  tile_mma<4, true, false>(acc, tT, kLs, m0, tX2, kLd, n128, 64, lane);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int i = frow(m0, lane, 2 * hh), col = fcol(n128, lane, nt, 0);
      const float x0 = updD * acc[nt][2 * hh], x1 = updD * acc[nt][2 * hh + 1];
      rb[hh] += upV * (x0 * h2f(tV, kLd, i, col) + x1 * h2f(tV, kLd, i, col + 1));
      if (p0 + i < a.L)
        *reinterpret_cast<float2*>(a.dv + (((size_t)b * a.L + p0 + i) * a.Hv + h) * kD + col) =
            make_float2(bet[i] * x0, bet[i] * x1);
    }
  zero(acc);
  tile_mma<4, true, false>(acc, tT, kLs, m0, tdW, kLd, n128, 64, lane);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = frow(m0, lane, e), col = fcol(n128, lane, nt, e);
      const float x = updW * acc[nt][e];
      const float r = x * h2f(tK, kLd, i, col);
      rb[e >> 1] += Gam[i] * r;
      rg[e >> 1] += bet[i] * Gam[i] * r;
      dK[nt][e] += bet[i] * Gam[i] * x;
    }

  // ---- 9. dT = dDelta (beta V)^T + dW (beta Gamma K^)^T; dA = -T^T dT T^T (j < i) ----
  {
    float t1[2][4], t2[2][4];
    zero(t1);
    tile_mma<2, false, true>(t1, tX2, kLd, m0, tV, kLd, n64, 128, lane);
    zero(t2);
    tile_mma<2, false, true>(t2, tdW, kLd, m0, tK, kLd, n64, 128, lane);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = fcol(n64, lane, nt, e);
        t1[nt][e] = bet[j] * (updD * upV * t1[nt][e] + Gam[j] * updW * t2[nt][e]);
      }
    float upT, dnT;
    pow2_up_dn(cta_max(absmax(t1), V(vMax), warp, lane, mpar), upT, dnT);
    store_h(tdT, kLs, m0, n64, t1, dnT, lane);
    __syncthreads();
    zero(t2);
    tile_mma<2, false, true>(t2, tdT, kLs, m0, tT, kLs, n64, 64, lane);   // dT T^T
    float upZ, dnZ;
    pow2_up_dn(cta_max(absmax(t2), V(vMax), warp, lane, mpar), upZ, dnZ);
    store_h(tZ, kLs, m0, n64, t2, dnZ, lane);
    __syncthreads();
    zero(t1);
    tile_mma<2, true, false>(t1, tT, kLs, m0, tZ, kLs, n64, 64, lane);    // T^T (dT T^T)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = frow(m0, lane, e), j = fcol(n64, lane, nt, e);
        float dAt = 0.f;   // dA~ = dA beta_i E_ij
        if (j < i) {
          const float dA = -upT * upZ * t1[nt][e];
          const float E = Eij(i, j), gk = G[nt][e];   // k^_i . k^_j (the Gram fragment has this tiling)
          rb[e >> 1] += dA * gk * E;
          const float aa = dA * bet[i] * gk * E;                  // dA o A
          rg[e >> 1] += aa;
          cg[2 * nt + (e & 1)] -= aa;
          dAt = dA * bet[i] * E;
        }
        t1[nt][e] = dAt;
      }
    float upA, dnA;
    pow2_up_dn(cta_max(absmax(t1), V(vMax), warp, lane, mpar), upA, dnA);
    store_h(tdA, kLs, m0, n64, t1, dnA, lane);
    __syncthreads();
    float t3[4][4];
    zero(t3);
    tile_mma<4, false, false>(t3, tdA, kLs, m0, tK, kLd, n128, 64, lane);
    tile_mma<4, true, false>(t3, tdA, kLs, m0, tK, kLd, n128, 64, lane);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) dK[nt][e] += upA * t3[nt][e];
  }

  // ---- 10. reductions: dgamma -> dg, dbeta; outputs ----
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      rg[hh] += __shfl_xor_sync(0xffffffffu, rg[hh], o);
      rb[hh] += __shfl_xor_sync(0xffffffffu, rb[hh], o);
      rd[hh] += __shfl_xor_sync(0xffffffffu, rd[hh], o);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) cg[i] += __shfl_xor_sync(0xffffffffu, cg[i], o);
  if ((lane & 3) == 0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int i = m0 + (lane >> 2) + 8 * hh;
      V(vRowG0 + quarter)[i] = rg[hh];
      V(vRowB0 + quarter)[i] = rb[hh];
      V(vRowD0 + quarter)[i] = rd[hh];
    }
  }
  if (lane < 4) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int x = 0; x < 2; ++x) V(vColG0 + (warp & 3))[n64 + 8 * nt + 2 * lane + x] = cg[2 * nt + x];
  }
  __syncthreads();
  auto sum4 = [&](int v0, int r) { return (V(v0)[r] + V(v0 + 1)[r]) + (V(v0 + 2)[r] + V(v0 + 3)[r]); };
  if (warp < 2) {
    // sum_j e_j k^_j . (dS' Delta_j) over the chunk (two warp sums)
    float t = sum4(vRowD0, tid);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) V(vMax)[warp] = t;
  }
  __syncthreads();
  if (warp == 0 || warp == 1) {
    // dgamma_i, then dg_j = sum_{i >= j} dgamma_i (a reversed inclusive scan over two warps)
    const int i = 63 - tid;   // warp 0: positions 63..32, warp 1: 31..0
    const float de = sum4(vRowD0, i);
    float dga = sum4(vRowG0, i) + sum4(vColG0, i) - de;
    if (i == 63) {
      const float tot_de = V(vMax)[0] + V(vMax)[1];
      float dotS = 0.f;
      for (int w = 0; w < kLT / 32; ++w) dotS += V(vDot)[w];
      dga += Gam[63] * dotS + tot_de;
    }
    float x = dga;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    V(vScan)[tid] = x;
  }
  __syncthreads();
  if (tid < 64) {
    const int i = 63 - tid;
    const float dgi = V(vScan)[tid] + (tid >= 32 ? V(vScan)[31] : 0.f);
    if (p0 + i < a.L) {
      const size_t gi = ((size_t)b * a.L + p0 + i) * a.Hv + h;
      a.dg[gi] = dgi;
      a.dbeta[gi] = (V(vRowB0)[i] + V(vRowB0 + 1)[i]) + (V(vRowB0 + 2)[i] + V(vRowB0 + 3)[i]);
    }
  }
  }   // value heads

  // ---- the normalisations' backward: q~ = q s_q 128^-0.5, k^ = k s_k, from the raw bf16 rows:
  //      dq = 128^-0.5 (s_q dq~ - s_q^3 (q . dq~) q), dk = s_k dk^ - s_k^3 (k . dk^) k ----
  {
    float xq[4][4], xk[4][4];
    float rq[2] = {0.f, 0.f}, rk[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = frow(m0, lane, 2 * hh), col = fcol(n128, lane, nt, 0);
        float2 qv = make_float2(0.f, 0.f), kv = qv;
        if (p0 + i < a.L) {
          const size_t o = (((size_t)b * a.L + p0 + i) * a.Hk + hk) * kD + col;
          qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a.q + o));
          kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a.k + o));
        }
        xq[nt][2 * hh] = qv.x;
        xq[nt][2 * hh + 1] = qv.y;
        xk[nt][2 * hh] = kv.x;
        xk[nt][2 * hh + 1] = kv.y;
        rq[hh] += qv.x * dQ[nt][2 * hh] + qv.y * dQ[nt][2 * hh + 1];
        rk[hh] += kv.x * dK[nt][2 * hh] + kv.y * dK[nt][2 * hh + 1];
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        rq[hh] += __shfl_xor_sync(0xffffffffu, rq[hh], o);
        rk[hh] += __shfl_xor_sync(0xffffffffu, rk[hh], o);
      }
    __syncthreads();   // the last value head's reads of the vectors are done
    if ((lane & 3) == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = m0 + (lane >> 2) + 8 * hh;
        V(vRowG0 + quarter)[i] = rq[hh];
        V(vRowB0 + quarter)[i] = rk[hh];
      }
    }
    __syncthreads();
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = frow(m0, lane, 2 * hh), col = fcol(n128, lane, nt, 0);
        if (p0 + i >= a.L) continue;
        const float tq = (V(vRowG0)[i] + V(vRowG0 + 1)[i]) + (V(vRowG0 + 2)[i] + V(vRowG0 + 3)[i]);
        const float tk = (V(vRowB0)[i] + V(vRowB0 + 1)[i]) + (V(vRowB0 + 2)[i] + V(vRowB0 + 3)[i]);
        const float s_q = sq[i], s_k = sk[i];
        const size_t o = (((size_t)b * a.L + p0 + i) * a.Hk + hk) * kD + col;
        *reinterpret_cast<float2*>(a.dq + o) =
            make_float2(kQs * (s_q * dQ[nt][2 * hh] - s_q * s_q * s_q * tq * xq[nt][2 * hh]),
                        kQs * (s_q * dQ[nt][2 * hh + 1] - s_q * s_q * s_q * tq * xq[nt][2 * hh + 1]));
        *reinterpret_cast<float2*>(a.dk + o) =
            make_float2(s_k * dK[nt][2 * hh] - s_k * s_k * s_k * tk * xk[nt][2 * hh],
                        s_k * dK[nt][2 * hh + 1] - s_k * s_k * s_k * tk * xk[nt][2 * hh + 1]);
      }
  }
}

// One CTA per (row, key head, chunk) (its tiles take most of an SM's shared memory).
__global__ void __launch_bounds__(kLT, 1) chunk_bwd_local_kernel(const LocalArgs a) {
  static_assert(kLT == 512, "the warp tiling assumes 16 warps");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  local_unit(a, sm, blockIdx.x);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t chunk_bwd_workspace_bytes(int B, int L, int Hk, int Hv) {
  (void)Hk;
  const size_t NC = ((size_t)L + kChunk - 1) / kChunk;
  const size_t states = (size_t)B * Hv * NC * kD * kD * sizeof(__half);
  const size_t scales = (size_t)B * Hv * NC * kStateSlices * sizeof(float);
  const size_t uscales = (size_t)B * Hv * NC * 8 * sizeof(float);
  return align256(chunk_bwd_units_bytes(B, L, Hv)) + 2 * align256(states) + 2 * align256(scales) + align256(uscales);
}

// the chunked backward's workspace: the chunk factors, then S_save, dS_save, S_scale, dS_scale and
// the per-unit scales
struct BwdWorkspace {
  uint8_t* units;
  __half* S_save;
  __half* dS_save;
  float* S_scale;
  float* dS_scale;
  float* unit_scale;
};
static BwdWorkspace split_workspace(void* ws, int B, int L, int Hv) {
  const size_t NC = ((size_t)L + kChunk - 1) / kChunk;
  const size_t states = (size_t)B * Hv * NC * kD * kD * sizeof(__half);
  const size_t scales = (size_t)B * Hv * NC * kStateSlices * sizeof(float);
  BwdWorkspace r;
  uint8_t* w = static_cast<uint8_t*>(ws);
  r.units = w;
  w += align256(chunk_bwd_units_bytes(B, L, Hv));
  r.S_save = reinterpret_cast<__half*>(w);
  w += align256(states);
  r.dS_save = reinterpret_cast<__half*>(w);
  w += align256(states);
  r.S_scale = reinterpret_cast<float*>(w);
  w += align256(scales);
  r.dS_scale = reinterpret_cast<float*>(w);
  w += align256(scales);
  r.unit_scale = reinterpret_cast<float*>(w);
  return r;
}

cudaError_t launch_chunk_forward_saving(const void* q, const void* k, const void* v, const float* g,
                                        const float* beta, const float* S0, void* o, float* S_T, void* ws,
                                        int B, int L, int Hk, int Hv, int* err, cudaStream_t s) {
  const BwdWorkspace w = split_workspace(ws, B, L, Hv);
  ChunkFwdSaveLaunch fl{q, k, v, g, beta, S0, o, S_T, w.S_save, w.S_scale, w.unit_scale, w.units, B, L, Hk, Hv, err};
  return launch_chunk_fwd_save(fl, s);
}

cudaError_t launch_chunk_backward(const ChunkBackwardArgs& p, cudaStream_t s) {
  const size_t NC = ((size_t)p.L + kChunk - 1) / kChunk;
  const BwdWorkspace w = split_workspace(p.ws, p.B, p.L, p.Hv);
  __half* S_save = w.S_save;
  __half* dS_save = w.dS_save;
  float* S_scale = w.S_scale;
  float* dS_scale = w.dS_scale;
  float* unit_scale = w.unit_scale;
  ChunkBwdChainLaunch cl{p.q, p.k, p.v, p.g, p.beta, p.S0, p.dO, p.dS_T, p.dS0, S_save, S_scale, dS_save, dS_scale,
                         unit_scale, w.units, p.B, p.L, p.Hk, p.Hv, p.err};
  cl.saved = p.saved;
  cudaError_t e = launch_chunk_bwd_chain(cl, s);
  if (e != cudaSuccess) return e;
  LocalArgs la{static_cast<const __nv_bfloat16*>(p.q), static_cast<const __nv_bfloat16*>(p.k),
               static_cast<const __nv_bfloat16*>(p.v), p.g, p.beta, static_cast<const __nv_bfloat16*>(p.dO),
               S_save, S_scale, dS_save, dS_scale, unit_scale, p.dq, p.dk, p.dv, p.dg, p.dbeta, p.B, p.L, p.Hk, p.Hv, (int)NC};
  e = cudaFuncSetAttribute(chunk_bwd_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kLocalSmem + 128);
  if (e != cudaSuccess) return e;
  // one CTA per (row, key head, chunk): the key head's value heads one after the other
  int slot = stage_timer_begin(s, kKernChunkBwdLocal);
  chunk_bwd_local_kernel<<<(unsigned)((size_t)p.B * p.Hk * NC), kLT, kLocalSmem + 128, s>>>(la);
  stage_timer_end(slot, s);
  return cudaGetLastError();
}

}  // namespace gdr

// Chunked gated delta rule on tcgen05 tensor cores (fp16 / bf16 operands, float32 accumulation).
//
// Chunk algebra (64-token chunks; the "R64" form named in Kev-4B-LiteRT "r15_kernel_test.py",
// with the pair decay computed directly, never as a ratio of cumulative decays). For a chunk with
// entering state S, gamma_i = sum_{j<=i} g_j, Gamma_i = exp(gamma_i), raw q/k rows and their
// inverse norms qi_i = (|q_i|^2 + 1e-6)^-1/2, ki_i likewise, sq_i = Gamma_i qi_i D^-1/2 and
// sk_i = exp(gamma_C - gamma_i) ki_i:
//
//   A_ij  = beta_i ki_i ki_j (k_i . k_j) exp(gamma_i - gamma_j),  j < i         (strictly lower)
//   T     = (I + A)^-1                                                          (unit lower)
//   W     = T diag(beta Gamma ki) K,     U = T diag(beta) V                     (WY factors)
//   P_ij  = qi_i ki_j D^-1/2 (q_i . k_j) exp(gamma_i - gamma_j),  j <= i
//   Vnew  = U - W S
//   O     = diag(sq) Q S + P Vnew  =  Q' S + P U,      Q' = diag(sq) Q - P W
//   S'    = Gamma_C S + K^T diag(sk) Vnew  =  Gamma_C S + M' S + N,
//           M' = -K^T diag(sk) W,   N = K^T diag(sk) U
//
// Everything but S is chunk-local, so the sequential part of the recurrence is one product M' S
// per chunk (plus Q' S for the output, which nothing later depends on).
//
// Every product whose operands are computed values runs on fp16 operands: one fp16 rounding
// (11-bit significand) costs about an eighth of a bf16 one, and an emulation of every rounding
// point against the float64 oracle puts the outputs at the floor set by rounding o to bf16 (the
// M' form's final states come out slightly closer to the oracle than the two-product form's).
// Operands are assumed inside fp16's range (|x| < 65504), which holds for l2-normalised keys.
//
// Kernel 1 (gdr_chunk_prep, persistent, two CTAs per SM, each working through (row, value head,
//   chunk) units; every unit is independent): TMA loads raw q, k, v; a bf16 MMA gives [Q; K] K^T
//   (both Gram matrices, exact products); CUDA cores build A and P; a recursive-doubling fp32
//   inverse gives T; T's scaled columns form the operand [A1; A2]; MMAs give W = A1 K and U = A2 V,
//   then P [W | U], then K^T [diag(sk) W | diag(sk) U] = [-M' | N]. Per unit it writes, with bulk
//   copies from shared memory, M' and Q' as the 128B-swizzled images kernel 2 uses as MMA
//   operands, N and P U as four 32-column slices, and Gamma_C.
// Kernel 2 (gdr_chunk_state, four independent CTAs per (row, value head), CTA s owning value
//   columns [32 s, 32 s + 32), sequential over chunks): the float32 state slice stays in registers.
//   Per chunk one thread issues D = M' S (fp16 copy of S as the B operand); the state warps form
//   S = Gamma_C S + D + N and the next fp16 copy; a second thread issues O' = Q' S and two output
//   warps form o = O' + P U, off the critical path. Two producer warps keep a ring of chain tiles
//   (M', N, Gamma_C) and a ring of output tiles (Q', P U) filled ahead of the chain.
#include <algorithm>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "gdr_epilogue.h"
#include "gdr_backward.h"
#include "gdr_inverse.cuh"
#include "gdr_internal.h"
#include "ptx.cuh"

namespace gdr {

using namespace ptx;

namespace {

constexpr float kScale = 0.08838834764831845f;   // 128^-0.5
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kDrainBudget = 2000000000ll;  // cycles (~1 s) an aborting CTA waits for its own copies
constexpr int kSlices = 4;                        // value-column slices (state CTAs) per value head
constexpr int kN = kD / kSlices;                  // 32 value columns per state CTA

// Workspace. Per (row, value head, chunk) unit:
constexpr uint32_t kMBytes = 32768;     // M': 128 x 128 fp16, two 64-column 128B-swizzled K-atoms
constexpr uint32_t kQBytes = 16384;     // Q': 64 x 128 fp16, same layout
constexpr uint32_t kNBytes = 32768;     // N: four 128 x 32 fp16 slices, rows of 64 B, 64B-swizzled
constexpr uint32_t kPUBytes = 16384;    // P U: four 64 x 32 fp16 slices, same row layout
constexpr uint32_t kSBytes = 512;       // Gamma_C (16 bytes used)
constexpr uint32_t kSCopy = 16;         // bytes of the scale block kernel 2 copies
constexpr uint32_t kUnitQ = kMBytes, kUnitN = kUnitQ + kQBytes, kUnitPU = kUnitN + kNBytes;
constexpr uint32_t kUnitS = kUnitPU + kPUBytes;
constexpr uint32_t kUnitBytes = kUnitS + kSBytes;

struct ChunkArgs {
  const float* g;
  const float* beta;
  const float* S0;
  const int64_t* S0_idx;   // row b starts from S0[S0_idx[b]] (forks); NULL = S0[b]
  int n_S0;                // states S0 holds when S0_idx is set
  int fused;               // single-chunk rows: kernel 1 applies the chunk to S0 itself
  long long wait_budget;   // cycles before a wait gives up (GDR_ERR_TIMEOUT)
  __nv_bfloat16* o;
  float* S_T;
  uint8_t* ws;       // 1024-aligned
  int B, L, Hk, Hv, NC;
  int* err;
  const int32_t* lengths;  // valid tokens per row (NULL = L); positions at or past it are pads
  // gated RMSNorm epilogue (state kernel, clusters of the four column CTAs of a head): o is replaced
  // by w * o / sqrt(mean(o^2) + eps) * silu(z) over the 128 values of each position and value head
  const __nv_bfloat16* z;
  const float* w;
  float eps;
  // state kernel modes 1 and 2 (the backward's passes): the state at the top of each chunk's step
  // (mode 1: the chunk's entering state; mode 2: the adjoint of its exiting state) as the fp16
  // operand the step's product reads: per (row, value head, chunk) four 8 KiB images, one per
  // 32-column slice (128 key rows of 64 bytes, 64-byte swizzle), each divided by its own power of
  // two, kept in st_scale [B, Hv, NC, 4]
  __half* st_save;
  float* st_scale;
  // per unit [B, Hv, NC, 8]: the powers of two of dO's four 32-column slices (kMode 2) and of v
  // (word 4, kMode 1), for the backward's chunk-local kernel
  float* unit_scale;
  // the GDN prologue fused into the prep kernel (kPro): the q|k|v projection [B, L, C] and its carry
  // [B, 3, C] (bf16), the depthwise conv weights [C, 4], the gate projections a, b [B, L, Hv] and
  // A_log, dt_bias [Hv]; q, k, v tiles and the gates are formed from them in place of the loads
  const __nv_bfloat16* mixed;
  const __nv_bfloat16* tail;
  const float* conv_w;
  const float* proj_a;
  const float* proj_b;
  const float* A_log;
  const float* dt_bias;
  int C;
};

__device__ __forceinline__ uint8_t* unit_base(const ChunkArgs& a, int b, int h, int c) {
  return a.ws + ((size_t)((size_t)b * a.Hv + h) * a.NC + c) * kUnitBytes;
}

__device__ __forceinline__ void set_error(int* err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}
__device__ __forceinline__ uint4 pack8_f16(const float* v) {
  return make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                    pack_f16x2(v[6], v[7]));
}
__device__ __forceinline__ void unpack8_f16(uint4 w, float* v) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[e]));
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

// Power-of-two scale of a tile whose largest magnitude is m (>= 0): up = 2^e with m / up in
// [0.5, 1) (up = 1 when m is zero or subnormal; e clamped to [-125, 125]), dn = 1 / up. Both are
// exact powers of two, so scaling by them is exact, and scaling the tile by 2^k shifts e by k.
__device__ __forceinline__ void pow2_scales(float m, float& up, float& dn) {
  const int eb = (int)((__float_as_uint(m) >> 23) & 0xFFu);
  int e = eb == 0 ? 0 : eb - 126;
  e = e < -125 ? -125 : (e > 125 ? 125 : e);
  up = __uint_as_float((uint32_t)(127 + e) << 23);
  dn = __uint_as_float((uint32_t)(127 - e) << 23);
}

// -------------------------------------------------------------------------------------------
// Kernel 1: per-chunk factors
// -------------------------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr uint32_t kVBar = 4;   // named barrier of warps 4-7 (v's scale)
constexpr uint32_t kPQ0 = 0, kPK0 = 8192, kPQ1 = 16384, kPK1 = 24576;   // [q|k] K-atoms (Gram operand)
constexpr uint32_t kPV = 32768;       // the v atoms' region; then the MN-major operand [W0 | W1 | U0 | U1];
                                      // then the staged Q' image and P U slices
constexpr uint32_t kPVt = 40960;      // v atoms at +0 and +16384: with the k atoms (8192, 24576) they make
                                      // [K | V] one MN-major operand of stride 16384
constexpr uint32_t kPXs = 49152;      // inverse scratch, between the v atoms (free until U is written there)
// P: K-major fp16 rows 0-63. The P [W | U] products have M = 128: P W reads operand rows from P on
// (P in rows 0-63, lanes 0-63) and P U from 8 KB before P (P in rows 64-127, lanes 64-127), so that
// the epilogue spreads over all eight warps; the other operand rows (the tail of the [W | U]
// operand, the start of AT) yield products in lanes that nobody reads.
constexpr uint32_t kPP = 65536;
constexpr uint32_t kPAT = kPP + 8192;           // fp32 [64][68]: A strictly lower, 1 on the diagonal, T^T strictly upper
constexpr uint32_t kPTm = kPAT + 64 * 68 * 4;   // fp32 [64][68]: T row-major (zero above the diagonal)
constexpr uint32_t kPAop = kPTm;                // after the inverse: MN-major operand [A1 | A2], fp16
constexpr uint32_t kPWS = kPAT;                 // after [A1 | A2] is consumed: MN-major operand
                                                // [sk W | sk U] (32 KB over AT and T); then the staged N
constexpr uint32_t kPM = 0;                     // after the last products: the staged M' image (over q, k)
constexpr uint32_t kPVec = kPTm + 64 * 68 * 4;  // gam2, Gam, bet, qinv, kinv, e1, sk: 7 x 64 floats
constexpr uint32_t kPE2 = kPVec + 7 * 64 * 4;   // E2[I][j] = ki_j exp(gamma_16I - gamma_j): [4][68] floats
constexpr uint32_t kPrepSmem = kPE2 + 4 * 68 * 4 + 1024;
static_assert(kPTm % 1024 == 0 && kPP % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(kPP + 16384 <= kPrepSmem - 1024 && kPAop + 16384 <= kPVec, "M = 128 operands stay inside the buffer");
static_assert(kPWS % 1024 == 0 && kPWS + 32768 <= kPVec, "the [sk W | sk U] operand fits over AT and T");
static_assert(kPVt == kPK1 + 16384 && kPXs + 36 * 32 * 4 <= kPVt + 16384 && kPVt + 16384 + 8192 <= kPP,
              "v atoms continue the k atoms' stride; the inverse scratch fits between them");
// The fused prologue's staging, free from the end of the previous unit until the tiles are formed:
// the raw projection rows p0 - 3 .. p0 + 63 of q, k and v (67 rows of 256 bytes each, unswizzled)
// and the unit's conv weights as float4s in [tensor][channel % 8][channel / 8] order (a quarter-warp
// reads 128 contiguous bytes). q's rows lie under the q and k tiles, v's under the first v atom,
// k's under the second v atom and P: each tile is written only once the rows beneath it are read.
constexpr uint32_t kRawRow = 256, kRawRows = 67;
constexpr uint32_t kRawQ = 0, kRawV = 32768, kRawK = kRawV + kRawRows * kRawRow, kRawW = kRawK + kRawRows * kRawRow;
static_assert(kRawQ + kRawRows * kRawRow <= kRawV && kRawV >= kPK1 + 8192 && kRawW % 16 == 0 &&
              kRawW + 3 * 128 * 16 <= kPAT,
              "v's and k's rows clear of the q and k tiles, everything clear of the draining N store");

// Persistent: CTA i takes units i, i + gridDim.x, ... in the order value head fastest, then chunks
// from the last to the first (so the units the state kernel reads first were written last and are
// the likeliest to still sit in L2), then rows. While one unit computes, the next unit's gates are
// loaded into registers and its tiles prefetched into L2. kFused (rows of one chunk, a.fused) is a
// template parameter, so that the multi-chunk kernel carries none of the in-place apply's code.
// kPro: the GDN prologue runs here (DEG "model.py", _linear_layer: _conv_silu over [carry, mixed],
// _dn_gates): each unit forms its q, k, v tiles as the causal depthwise conv (4 taps) + SiLU of the
// projection's rows, rounded to bf16, in the prologue kernel's order of operations (so the tiles
// equal the separate prologue's output bit for bit), and its gates from a, b.
template <bool kFused, bool kPro = false>
__global__ void __launch_bounds__(kPrepThreads, 2)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_ld, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ float gbuf[2][128];   // gates of the current and the next unit: g[64] | beta[64]
  __shared__ uint32_t tile_max[6];   // largest |k_row|^2 (warps 2, 3: float bits), |v| (warps 4-7: bf16 bits)
  __shared__ float unit_scl[4];      // upK, dnK, upV, dnV of the current unit
  __shared__ uint32_t s0max[kPrepThreads / 32];   // per-warp largest |S0| (float bits), fused apply

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = a.Hv / a.Hk;
  const int total = a.B * a.Hv * a.NC;
  float* AT = reinterpret_cast<float*>(sm + kPAT);
  float* Tm = reinterpret_cast<float*>(sm + kPTm);
  float* Xs = reinterpret_cast<float*>(sm + kPXs);
  float* gam2 = reinterpret_cast<float*>(sm + kPVec);     // cumulative log-decay times log2(e)
  float* Gam = gam2 + 64;
  float* bet = gam2 + 128;
  float* qinv = gam2 + 192;
  float* kinv = gam2 + 256;
  float* e1 = gam2 + 320;                                  // exp(gamma_i - gamma_16I); scan scratch first
  float* skv = gam2 + 384;                                 // sk_i = exp(gamma_C - gamma_i) ki_i
  float* E2 = reinterpret_cast<float*>(sm + kPE2);

  // unit u -> (chunk c, value head h, row b)
  auto unit_of = [&](int u, int& c, int& h, int& b) {
    h = u % a.Hv;
    const int rest = u / a.Hv;
    c = a.NC - 1 - rest % a.NC;
    b = rest / a.NC;
  };
  // valid tokens of row b (its length when lengths are given)
  auto row_len = [&](int b) -> int { return a.lengths ? a.lengths[b] : a.L; };
  // a unit is skipped when its row's length is invalid (outside [0, L]) or, for rows of several
  // chunks, when the unit lies wholly at or past the length (the state kernel stops there); a
  // single-chunk row's unit always runs, since it also writes the row's final state
  auto valid = [&](int u) -> bool {
    if (!a.lengths) return true;
    int c, h, b;
    unit_of(u, c, h, b);
    const int lb = a.lengths[b];
    if (lb < 0 || lb > a.L) {
      if (tid == 0) set_error(a.err, kErrDeviceIndex);
      return false;
    }
    return kFused || c * 64 < lb;
  };
  auto next_valid = [&](int u) -> int {
    while (u < total && !valid(u)) u += (int)gridDim.x;
    return u;
  };
  // gates of a unit into gbuf[buf] (threads 0-63, one position each, asynchronous copies);
  // positions past L or past the row's length read as beta = g = 0 (pads). Every thread commits one
  // group per call.
  auto copy_gates = [&](int u, int buf) {
    if (tid < 64) {
      int c, h, b;
      unit_of(u, c, h, b);
      const int p = c * 64 + tid;
      if (p < a.L && p < row_len(b)) {
        cp_async4(&gbuf[buf][tid], (kPro ? a.proj_a : a.g) + ((size_t)b * a.L + p) * a.Hv + h);
        cp_async4(&gbuf[buf][64 + tid], (kPro ? a.proj_b : a.beta) + ((size_t)b * a.L + p) * a.Hv + h);
      } else {
        gbuf[buf][tid] = 0.f;
        gbuf[buf][64 + tid] = 0.f;
      }
    }
    cp_async_commit();
  };
  // raw q, k, v tiles of a unit (six 64 x 64 boxes) into shared memory, or only into L2; called
  // by every thread: lane 0 of warp t < 6 issues box t, so the six issues proceed in parallel
  // (warp 0 also posts the byte count; the order of count and bytes does not matter)
  // kPro: the unit's q, k, v tiles as conv + SiLU of the projection, stored like the TMA boxes (rows
  // past L zero). The raw rows (the carry for positions before 0, zeros past L) and the weights are
  // copied into shared memory at the top of the unit (pro_issue) and land during the gate scan.
  // Thread = (8-channel group cg, 4-row group rg) per tile, window ext rows p - 3 .. p + 3;
  // s = sum_j w_j x_{t-3+j} in tap order, then s / (1 + e^-s), one rounding to bf16.
  auto pro_chan = [&](int tsr, int h) {
    const int HkD = a.Hk * kD;
    return tsr == 0 ? (h / r) * kD : tsr == 1 ? HkD + (h / r) * kD : 2 * HkD + h * kD;
  };
  auto pro_issue = [&](int c, int h, int b) {
    const int p0 = c * 64 - 3;
#pragma unroll 1
    for (int i = tid; i < 3 * (int)kRawRows * 16; i += kPrepThreads) {
      const int tsr = i / ((int)kRawRows * 16), rem = i - tsr * (int)kRawRows * 16, row = rem >> 4, ch = rem & 15;
      const int pos = p0 + row, chan = pro_chan(tsr, h) + ch * 8;
      const __nv_bfloat16* src = a.mixed;   // (a valid address; nothing is read when n = 0)
      uint32_t n = 0;
      if (pos < 0) {
        if (a.tail) {
          src = a.tail + ((size_t)b * 3 + pos + 3) * a.C + chan;
          n = 16;
        }
      } else if (pos < a.L) {
        src = a.mixed + ((size_t)b * a.L + pos) * a.C + chan;
        n = 16;
      }
      const uint32_t base = tsr == 0 ? kRawQ : tsr == 1 ? kRawK : kRawV;
      cp_async16_zfill(sm + base + row * kRawRow + ch * 16, src, n);
    }
    for (int i = tid; i < 3 * 128; i += kPrepThreads) {
      const int tsr = i >> 7, cc = i & 127;
      cp_async16_zfill(sm + kRawW + ((tsr * 8 + (cc & 7)) * 16 + (cc >> 3)) * 16,
                       a.conv_w + (size_t)(pro_chan(tsr, h) + cc) * 4, 16);
    }
  };
  auto pro_window = [&](int tsr, uint4 (&raw)[7]) {
    const uint8_t* src = sm + (tsr == 0 ? kRawQ : tsr == 1 ? kRawK : kRawV) + 4 * (tid >> 4) * kRawRow + (tid & 15) * 16;
#pragma unroll
    for (int j = 0; j < 7; ++j) raw[j] = *reinterpret_cast<const uint4*>(src + j * kRawRow);
  };
  auto pro_conv = [&](int tsr, int c, const uint4 (&raw)[7]) {
    const int cg = tid & 15, rg = tid >> 4, col = cg * 8;
    const float4* wsm = reinterpret_cast<const float4*>(sm + kRawW) + tsr * 128 + cg;
    uint32_t out[4][4];   // [row][channel pair], bf16x2
#pragma unroll
    for (int ep = 0; ep < 4; ++ep) {
      // channels 2 ep (the low half of each raw word ep) and 2 ep + 1 (the high half)
      const float4 wa = wsm[(2 * ep) * 16], wb = wsm[(2 * ep + 1) * 16];
      float xa[7], xb[7];
#pragma unroll
      for (int j = 0; j < 7; ++j) {
        const uint32_t wv = ep == 0 ? raw[j].x : ep == 1 ? raw[j].y : ep == 2 ? raw[j].z : raw[j].w;
        xa[j] = __uint_as_float(wv << 16);
        xb[j] = __uint_as_float(wv & 0xFFFF0000u);
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        float sa = 0.f, sb = 0.f;
        sa = fmaf(wa.x, xa[rr], sa);
        sb = fmaf(wb.x, xb[rr], sb);
        sa = fmaf(wa.y, xa[rr + 1], sa);
        sb = fmaf(wb.y, xb[rr + 1], sb);
        sa = fmaf(wa.z, xa[rr + 2], sa);
        sb = fmaf(wb.z, xb[rr + 2], sb);
        sa = fmaf(wa.w, xa[rr + 3], sa);
        sb = fmaf(wb.w, xb[rr + 3], sb);
        out[rr][ep] = pack_bf16x2(__fdividef(sa, 1.f + __expf(-sa)), __fdividef(sb, 1.f + __expf(-sb)));
      }
    }
    uint8_t* base = sm + (tsr == 0 ? kPQ0 : tsr == 1 ? kPK0 : kPVt) + (col >> 6) * 16384;   // atoms 16 KB apart
    const int ch = (col & 63) >> 3;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int row = 4 * rg + rr;
      const uint4 v = c * 64 + row < a.L ? make_uint4(out[rr][0], out[rr][1], out[rr][2], out[rr][3])
                                         : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(base + row * 128 + ((ch ^ (row & 7)) << 4)) = v;
    }
  };
  // kPro: the next unit's projection rows into L2 (67 positions x 256 bytes for each of q, k, v)
  auto pro_prefetch = [&](int u) {
    if (tid >= 3 * 67) return;
    int c, h, b;
    unit_of(u, c, h, b);
    const int tsr = tid / 67, pos = c * 64 - 3 + tid % 67;
    if (pos < 0 || pos >= a.L) return;
    const int HkD = a.Hk * kD, hk = h / r;
    const int chan = tsr == 0 ? hk * kD : tsr == 1 ? HkD + hk * kD : 2 * HkD + h * kD;
    bulk_prefetch_l2(a.mixed + ((size_t)b * a.L + pos) * a.C + chan, kD * 2);
  };
  auto tiles = [&](int u, bool to_smem) {
    if (kPro) {
      if (!to_smem) pro_prefetch(u);
      return;
    }
    if (warp >= 6 || lane != 0) return;
    const int t = warp;
    int c, h, b;
    unit_of(u, c, h, b);
    const int hk = h / r;
    const CUtensorMap* map = t < 2 ? &tm_q : (t < 4 ? &tm_k : &tm_v);
    const int c0 = (t & 1) * 64, c1 = t < 4 ? hk : h;
    // shared-memory order: q0 k0 q1 k1 (the Gram operand), then v0 v1
    const uint32_t dst = t < 4 ? (uint32_t)((t & 1) * 16384 + (t >> 1) * 8192) : kPVt + (uint32_t)(t - 4) * 16384;
    if (to_smem) {
      if (t == 0) mbar_arrive_expect_tx(&bar_ld, 49152);
      tma_load_4d(sm + dst, map, &bar_ld, c0, c1, c * 64, b);
    } else {
      tma_prefetch_4d(map, c0, c1, c * 64, b);
    }
  };

  int u = next_valid(blockIdx.x);
  if (u < total) copy_gates(u, 0);
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (u < total) tiles(u, true);
  if (warp == 1) tmem_alloc(&tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  bool ok = true;
  uint32_t mma_phase = 0;   // completions of bar_mma so far (4 per unit, 5 with the fused apply)
  // a wait that gives up leaves its copy or product in flight: the parity it waited for is kept so
  // that the CTA can drain it before exiting
  int ld_fail = -1, mma_fail = -1;
  auto wait_mma = [&]() -> bool {
    const uint32_t par = mma_phase++ & 1;
    const bool r = mbar_wait(&bar_mma, par, a.wait_budget);
    if (!r) mma_fail = (int)par;
    return r;
  };

  for (int it = 0; u < total; ++it) {
  int c, h, b;
  unit_of(u, c, h, b);
  uint8_t* ub = unit_base(a, b, h, c);
  float pro_dtb = 0.f, pro_alog = 0.f;
  if (kPro) {
    // the previous unit's stores staged over this region have been read (the end of its loop)
    pro_issue(c, h, b);   // its own group, between this unit's gates and the next unit's
    cp_async_commit();
    if (tid < 64) {
      pro_dtb = __ldg(a.dt_bias + h);
      pro_alog = __ldg(a.A_log + h);
    }
  }
  const int un = next_valid(u + (int)gridDim.x);
  if (un < total) {
    copy_gates(un, (it + 1) & 1);
  } else {
    cp_async_commit();
  }
  // this unit's gates have landed (the next unit's, and with kPro the staged rows, may still be in flight)
  if (kPro)
    cp_async_wait<2>();
  else
    cp_async_wait<1>();
  // inclusive scan of g over the chunk (warps 0 and 1, then warp 1 adds warp 0's total)
  if (tid < 64) {
    float gg = gbuf[it & 1][tid], bb = gbuf[it & 1][64 + tid];
    if (kPro) {
      // the prologue's gates from the projections: beta = sigmoid(b), g = -exp(A_log) softplus(a +
      // dt_bias) at valid positions, 0 at pads (as the prologue kernel computes them)
      float beta = 0.f, g = 0.f;
      if (c * 64 + tid < a.L) {
        beta = 1.f / (1.f + expf(-bb));
        const float xa = gg + pro_dtb;
        const float sp = xa > 20.f ? xa : log1pf(expf(xa));
        g = -expf(pro_alog) * sp;
      }
      gg = g;
      bb = beta;
    }
    float x = gg;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    e1[tid] = x;
    bet[tid] = bb;
  }
  __syncthreads();
  if (tid < 64) {
    const float gam = e1[tid] + (tid >= 32 ? e1[31] : 0.f);
    gam2[tid] = gam * kLog2e;
    Gam[tid] = exp2f(gam * kLog2e);
  }

  if (kPro) {
    cp_async_wait<1>();   // the staged rows and weights (the next unit's gates may still be in flight)
    __syncthreads();
    uint4 raw[7];
    pro_window(0, raw);
    __syncthreads();   // q's rows are read before the q tiles overwrite them
    pro_conv(0, c, raw);
    pro_window(1, raw);
    pro_conv(1, c, raw);
    pro_window(2, raw);
    __syncthreads();   // k's and v's rows are read before the v tiles overwrite them
    pro_conv(2, c, raw);
    fence_async_smem();   // generic writes, then the Gram product reads them
    ok = true;
  } else {
    ok = mbar_wait(&bar_ld, it & 1, a.wait_budget);
  }
  if (!ok) ld_fail = it & 1;
  if (!__syncthreads_and(ok)) break;

  // Gram MMA (bf16, exact products): D[0:128, 0:64] = [Q; K] K^T, issued by warp 7 while warps
  // 0-3 form the inverse norms and warps 4-6 the decay factors
  if (warp == 7) {
    if (lane == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t atom = smem_u32(sm) + (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tb, smem_desc(atom, 16, 1024), smem_desc(atom + 8192, 16, 1024), idesc, kk > 0);
      }
      mma_commit(&bar_mma);
    }
  } else if (warp < 4) {
    // inverse norms, one thread per row (rows 0-63 q, 64-127 k), both 64-column atoms. The sum
    // does not care about the order of the 16-byte chunks, so each row starts at a different one
    // and the eight lanes of a quarter-warp hit eight different banks.
    const int rr = tid & 63;
    const uint8_t* base = sm + (tid < 64 ? kPQ0 : kPK0) + rr * 128;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + half * 16384 + (((ch + rr) & 7) << 4));
        const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xFFFF0000u);
          s0 = fmaf(lo, lo, s0);
          s1 = fmaf(hi, hi, s1);
        }
      }
    }
    (tid < 64 ? qinv : kinv)[rr] = rsqrtf(s0 + s1 + 1e-6f);
    // the largest squared row norm of k (for k's scale, which only guards fp16's range)
    const uint32_t kn = __reduce_max_sync(0xffffffffu, __float_as_uint(s0 + s1));
    if (warp >= 2 && lane == 0) tile_max[warp - 2] = kn;
  } else {
    // decay factors through the 16-block anchors: for j < 16 I <= i,
    // exp(gamma_i - gamma_j) = exp(gamma_i - gamma_16I) * exp(gamma_16I - gamma_j), both factors
    // <= 1; the k scales ki_j of E2 and ki_i of sk are applied once the norms are known
    for (int e = tid - 128; e < 320; e += 96) {
      if (e < 64) {
        e1[e] = ex2_approx(gam2[e] - gam2[e & ~15]);
      } else if (e < 128) {
        skv[e - 64] = exp2f(gam2[63] - gam2[e - 64]);
      } else {
        const int I = 1 + ((e - 128) >> 6), j = e & 63;
        E2[I * 68 + j] = (j < 16 * I) ? ex2_approx(gam2[16 * I] - gam2[j]) : 0.f;
      }
    }
  }
  __syncthreads();
  // The unit's power-of-two scales: k and v enter the fp16 products as k dnK and v dnV; upK = 1 / dnK
  // is folded into the scalings that multiply K (A1 and sk), so W, M' and the rest come out as before,
  // while U, N and P U are formed in v's scale (upV goes to the state kernel with Gamma_C). v is
  // always scaled (exactness under power-of-two scaling of v); k only when its largest row norm is
  // outside [2^-6, 2^6), where k or the inverse norms folded into A1 and sk would leave fp16's
  // normal range. They are published in unit_scl for the uses after the next barrier: k's by thread 0
  // now, v's by warps 4-7, which take v's maximum and convert v while the Gram product completes.
  auto k_scales = [&](float& upK, float& dnK) {
    const float kn = sqrtf(__uint_as_float(max(tile_max[0], tile_max[1])));
    upK = dnK = 1.f;
    if (kn >= 64.f || (kn > 0.f && kn < 0.015625f)) pow2_scales(kn, upK, dnK);
  };
  if (tid < 64) {
    float upK, dnK;
    k_scales(upK, dnK);
    skv[tid] *= kinv[tid] * upK;
    if (tid == 0) {
      unit_scl[0] = upK;
      unit_scl[1] = dnK;
    }
  } else {
    const int I = 1 + ((tid - 64) >> 6), j = tid & 63;
    E2[I * 68 + j] *= kinv[j];
  }
  if (tid >= 128) {
    // while the Gram product completes: the largest |v| of the tile (two 8 KB atoms), for its
    // power-of-two scale; warp 4 + t takes 16-byte chunks t, t + 4, ... of the 1024, as per-halfword
    // maxima of the bf16 magnitude bits (|x| orders like its bits with the sign cleared)
    uint32_t mv2 = 0;
#pragma unroll 4
    for (int c16 = tid - 128; c16 < 1024; c16 += 128) {
      const uint4 w = *reinterpret_cast<const uint4*>(sm + kPVt + (c16 >> 9) * 16384 + (c16 & 511) * 16);
      mv2 = __vmaxu2(mv2, __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu), __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu)));
    }
    const uint32_t mv = __reduce_max_sync(0xffffffffu, max(mv2 & 0xFFFFu, mv2 >> 16));
    if (lane == 0) tile_max[warp - 2] = mv;
    named_bar_and(kVBar, 128, true);
    // v's power of two, and v to fp16 in place times dnV (the Gram product does not read v)
    float upV, dnV;
    pow2_scales(__uint_as_float(max(max(tile_max[2], tile_max[3]), max(tile_max[4], tile_max[5])) << 16), upV, dnV);
    if (tid == 128) {
      unit_scl[2] = upV;
      unit_scl[3] = dnV;
    }
#pragma unroll 4
    for (int c16 = tid - 128; c16 < 1024; c16 += 128) {
      uint4* p = reinterpret_cast<uint4*>(sm + kPVt + (c16 >> 9) * 16384 + (c16 & 511) * 16);
      const uint4 w = *p;
      *p = make_uint4(bf16x2_to_f16x2_scaled(w.x, dnV), bf16x2_to_f16x2_scaled(w.y, dnV),
                      bf16x2_to_f16x2_scaled(w.z, dnV), bf16x2_to_f16x2_scaled(w.w, dnV));
    }
  }
  if (tid == 0) bulk_wait_read();   // the previous unit's N store has read the AT / Tm region
  ok = wait_mma();
  if (!__syncthreads_and(ok)) break;
  tc_fence_after();

  // T's row-major copy starts as the identity (its upper part stays zero)
  for (int e = tid; e < 64 * 17; e += kPrepThreads) {
    const int rr = e / 17, c4 = e - rr * 17;
    const int d = ((rr >> 2) == c4) ? (rr & 3) : -1;
    reinterpret_cast<float4*>(Tm + rr * 68)[c4] =
        make_float4(d == 0 ? 1.f : 0.f, d == 1 ? 1.f : 0.f, d == 2 ? 1.f : 0.f, d == 3 ? 1.f : 0.f);
  }
  {
    // this thread's half Gram row: TMEM lane 32 (warp % 4) + lane, columns jb .. jb + 31
    // (rows 0-63: (Q K^T)_i,:, rows 64-127: (K K^T)_i,:), as two 16-column blocks J
    const int row = 32 * (warp & 3) + lane, i = row & 63, jb = (warp >> 2) * 32, I = i >> 4;
    const bool isK = row >= 64;
    float G[32];
    tmem_ld32(tb + lane_base + jb, G);
    tc_fence_before();
    const float rowf = isK ? bet[i] * kinv[i] : qinv[i] * kScale;
    const float rowe = rowf * e1[i];
    const float gi = gam2[i];
    const int jlim = isK ? i : i + 1;     // A keeps j < i, P keeps j <= i
    float v[32];
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int J = (jb >> 4) + hb;
      float* vv = v + 16 * hb;
      const float* Gv = G + 16 * hb;
      if (J < I) {
        const float4* e4 = reinterpret_cast<const float4*>(E2 + I * 68 + 16 * J);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 t = e4[q];
          vv[4 * q] = rowe * t.x * Gv[4 * q];
          vv[4 * q + 1] = rowe * t.y * Gv[4 * q + 1];
          vv[4 * q + 2] = rowe * t.z * Gv[4 * q + 2];
          vv[4 * q + 3] = rowe * t.w * Gv[4 * q + 3];
        }
      } else if (J == I) {
        const float4* k4 = reinterpret_cast<const float4*>(kinv + 16 * J);
        const float4* g4 = reinterpret_cast<const float4*>(gam2 + 16 * J);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 kq = k4[q], gq = g4[q];
          const float kk[4] = {kq.x, kq.y, kq.z, kq.w}, gm[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 16 * J + 4 * q + u;
            const float d = rowf * kk[u] * ex2_approx(gi - gm[u]);
            vv[4 * q + u] = (j < jlim) ? d * Gv[4 * q + u] : 0.f;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) vv[e] = 0.f;
      }
    }
    if (isK) {
      // row i of A into AT (1 on the diagonal; the upper part is overwritten by the inverse)
      float4* arow = reinterpret_cast<float4*>(AT + i * 68 + jb);
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        float t[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) t[e] = (jb + 4 * j4 + e == i) ? 1.f : v[4 * j4 + e];
        arow[j4] = make_float4(t[0], t[1], t[2], t[3]);
      }
    } else {
      // row i of P (lower, diagonal included) as fp16 K-major operand row
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ch = (jb >> 3) + q;
        *reinterpret_cast<uint4*>(sm + kPP + i * 128 + ((ch ^ (i & 7)) << 4)) = pack8_f16(v + 8 * q);
      }
    }
  }
  __syncthreads();

  invert_unit_lower(AT, Tm, Xs, tid, [&](int t) {
    // the k tile to fp16 in place, for the fp16 products (the Gram MMA that read k as bf16 has
    // completed); 1024 chunks of 16 B, times k's scale (1 unless k needs scaling). (v was converted,
    // times its own power of two, while the Gram product ran.)
    const float sc = unit_scl[1];
    for (int chunk16 = t - 64; chunk16 < 1024; chunk16 += kPrepThreads - 64) {
      const int which = chunk16 >> 9, off = (chunk16 & 511) * 16;
      uint4* p = reinterpret_cast<uint4*>(sm + (which == 0 ? kPK0 : kPK1) + off);
      uint4 w = *p;
      if (sc == 1.f)
        w = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
      else
        w = make_uint4(bf16x2_to_f16x2_scaled(w.x, sc), bf16x2_to_f16x2_scaled(w.y, sc),
                       bf16x2_to_f16x2_scaled(w.z, sc), bf16x2_to_f16x2_scaled(w.w, sc));
      *p = w;
    }
  });

  // operand [A1; A2] = [T diag(beta Gamma ki); T diag(beta)], MN-major: K-row j holds column j of T
  {
    const int j = tid & 63, blk = (tid >> 6) & 1, hf = tid >> 7;
    const float s = blk ? bet[j] : bet[j] * Gam[j] * kinv[j] * unit_scl[0];
    const float4* trow = reinterpret_cast<const float4*>(AT + j * 68);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int ch = 4 * hf + q;
      const float4 t0 = trow[2 * ch], t1 = trow[2 * ch + 1];
      const float tt[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = (8 * ch + e >= j) ? tt[e] * s : 0.f;
      *reinterpret_cast<uint4*>(sm + kPAop + blk * 8192 + j * 128 + ((ch ^ (j & 7)) << 4)) = pack8_f16(v);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // [A1; A2] [K | V]: W = A1 K in rows 0-63 of columns 0-127, U = A2 V in rows 64-127 of columns
  // 128-255 (the other two blocks are not read)
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = idesc_f16(128, 256, true, true);
    const uint32_t aop = smem_u32(sm + kPAop);
    const uint32_t kv = smem_u32(sm + kPK0);   // k atoms at +8192, +24576, v atoms at +40960, +57344
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(tb, smem_desc(aop + kk * 2048, 8192, 1024), smem_desc(kv + kk * 2048, 16384, 1024), idesc, kk > 0);
    mma_commit(&bar_mma);
  }
  if (un < total) tiles(un, false);   // the next unit's tiles into L2, while W and U are formed
  ok = wait_mma();
  if (!__syncthreads_and(ok)) break;
  tc_fence_after();

  {
    // W rows (TMEM lanes 0-63, warps 0, 1, 4, 5) and U rows (lanes 64-127, warps 2, 3, 6, 7);
    // warps 0-3 take columns 0-63, warps 4-7 columns 64-127. Each goes to its fp16 operand block
    // over v (consumed) for P [W | U], and scaled by sk_i to the operand [sk W | sk U] for K^T.
    const int row = 32 * (warp & 3) + lane, i = row & 63, cb = (warp >> 2) * 64;
    const bool isU = row >= 64;
    const float sk = skv[i];
    float w[64];
    tmem_ld64(tb + lane_base + (isU ? 128 : 0) + cb, w);
#pragma unroll
    for (int q8 = 0; q8 < 8; ++q8) {
      const int col = cb + q8 * 8;
      const int atom = col >> 6, ch = (col & 63) >> 3;
      const uint32_t off = (isU ? 16384 : 0) + atom * 8192 + i * 128 + ((ch ^ (i & 7)) << 4);
      float ws[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ws[e] = sk * w[q8 * 8 + e];
      *reinterpret_cast<uint4*>(sm + kPV + off) = pack8_f16(w + q8 * 8);
      *reinterpret_cast<uint4*>(sm + kPWS + off) = pack8_f16(ws);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // P W into columns 0-127 of TMEM lanes 0-63 and P U into columns 128-255 of lanes 64-127
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = idesc_f16(128, 128, false, true);
    const uint32_t pa = smem_u32(sm + kPP), wu = smem_u32(sm + kPV);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(tb, smem_desc(pa + kk * 32, 16, 1024), smem_desc(wu + kk * 2048, 8192, 1024), idesc, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(tb + 128, smem_desc(pa - 8192 + kk * 32, 16, 1024), smem_desc(wu + 16384 + kk * 2048, 8192, 1024),
               idesc, kk > 0);
    mma_commit(&bar_mma);
  }
  ok = wait_mma();
  if (!__syncthreads_and(ok)) break;
  tc_fence_after();

  {
    // warps 0, 1, 4, 5 (lanes 0-63): Q'_i = sq_i q_i - (P W)_i, the fp16 image, on columns cb .. cb + 63;
    // warps 2, 3, 6, 7 (lanes 64-127): (P U)_i, the fp16 slices, on columns cb .. cb + 63. Both are
    // staged over the consumed [W | U] operand, Gamma_C over P.
    const int row = 32 * (warp & 3) + lane, i = row & 63, cb = (warp >> 2) * 64;
    float w[64];
    if (row < 64) {
      const float sq = Gam[i] * qinv[i] * kScale;
      tmem_ld64(tb + lane_base + cb, w);
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const int col = cb + q8 * 8;
        const int atom = col >> 6, ch = (col & 63) >> 3;
        const uint32_t off = atom * 8192 + i * 128 + ((ch ^ (i & 7)) << 4);
        const uint4 qr = *reinterpret_cast<const uint4*>(sm + (atom ? kPQ1 : kPQ0) + i * 128 + ((ch ^ (i & 7)) << 4));
        const uint32_t q4w[4] = {qr.x, qr.y, qr.z, qr.w};
        float v[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = sq * __uint_as_float(q4w[e] << 16) - w[q8 * 8 + 2 * e];
          v[2 * e + 1] = sq * __uint_as_float(q4w[e] & 0xFFFF0000u) - w[q8 * 8 + 2 * e + 1];
        }
        *reinterpret_cast<uint4*>(sm + kPV + off) = pack8_f16(v);
      }
    } else {
      tmem_ld64(tb + lane_base + 128 + cb, w);
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const int col = cb + q8 * 8;
        *reinterpret_cast<uint4*>(sm + kPV + 16384 + (col >> 5) * 4096 + swz64(i * 64 + (q8 & 3) * 16)) =
            pack8_f16(w + q8 * 8);
      }
    }
    if (tid == 0) *reinterpret_cast<float4*>(sm + kPP) = make_float4(Gam[63], unit_scl[2], 0.f, 0.f);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // K^T [sk W | sk U] = [-M' | N] into columns 0-255 (the P [W | U] results have been read); Q',
  // P U and Gamma_C leave for the workspace meanwhile
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = idesc_f16(128, 256, true, true);
    const uint32_t kt = smem_u32(sm + kPK0);    // k atoms (M blocks) at +8192 and +24576: stride 16384
    const uint32_t wsu = smem_u32(sm + kPWS);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(tb, smem_desc(kt + kk * 2048, 16384, 1024), smem_desc(wsu + kk * 2048, 8192, 1024), idesc, kk > 0);
    mma_commit(&bar_mma);
    if (!kFused) {
      bulk_store(ub + kUnitQ, sm + kPV, kQBytes);
      bulk_store(ub + kUnitPU, sm + kPV + 16384, kPUBytes);
      bulk_store(ub + kUnitS, sm + kPP, kSCopy);
      bulk_commit();
    }
  }
  ok = wait_mma();
  if (!__syncthreads_and(ok)) break;
  tc_fence_after();

  {
    // every warp: key row i = TMEM lane, columns cb .. cb + 63 of M' = -D[:, 0:128] (fp16 K-major
    // image over q and k, consumed) and of N = D[:, 128:256] (fp16 slices over [sk W | sk U]),
    // staged for bulk stores (per-thread 16-byte global stores of these row layouts are far slower)
    const int i = 32 * (warp & 3) + lane, cb = (warp >> 2) * 64;
    {
      float w[64];
      tmem_ld64(tb + lane_base + cb, w);
#pragma unroll
      for (int e = 0; e < 64; ++e) w[e] = -w[e];
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const int col = cb + q8 * 8;
        const int atom = col >> 6, ch = (col & 63) >> 3;
        *reinterpret_cast<uint4*>(sm + kPM + atom * 16384 + i * 128 + ((ch ^ (i & 7)) << 4)) = pack8_f16(w + q8 * 8);
      }
    }
    {
      float n[64];
      tmem_ld64(tb + lane_base + 128 + cb, n);
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const int col = cb + q8 * 8;
        *reinterpret_cast<uint4*>(sm + kPWS + (col >> 5) * 8192 + swz64(i * 64 + (q8 & 3) * 16)) =
            pack8_f16(n + q8 * 8);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  if constexpr (kFused) {
    // Single-chunk row: apply the chunk to the initial state here (no workspace, no kernel 2).
    //   S_T = Gamma_C S0 + M' S0 + N,   o = Q' S0 + P U
    // computed transposed, with S0^T (fp16) as the A operand in TMEM: D^T = S0^T M'^T (values x
    // keys, columns 64-191), O^T = S0^T Q'^T (values x positions, columns 192-255). Thread
    // (warp w, lane l) owns value v = 32 (w % 4) + l and keys / positions of half w / 4.
    tc_fence_after();
    const int v = 32 * (warp & 3) + lane, hb = warp >> 2;
    const float upV = unit_scl[2];
    const float* s0 = nullptr;
    bool write = true;
    if (a.S0) {
      size_t row = b;
      if (a.S0_idx) {
        const long long ix = a.S0_idx[b];
        write = ix >= 0 && ix < a.n_S0;
        row = write ? (size_t)ix : 0;
        if (!write && tid == 0) set_error(a.err, kErrDeviceIndex);
      }
      s0 = a.S0 + (row * a.Hv + h) * kD * kD;
    } else if (a.S0_idx) {
      const long long ix = a.S0_idx[b];
      write = ix >= 0 && ix < a.n_S0;
      if (!write && tid == 0) set_error(a.err, kErrDeviceIndex);
    }
    // this thread's 64 S0 entries (keys 64 hb .., value v), kept in registers for the Gamma_C S0
    // term of S_T (S_T may alias S0: each entry is read here, before any store, by the one thread
    // that later writes it)
    float x0[64];
#pragma unroll
    for (int e = 0; e < 64; ++e) x0[e] = s0 ? __ldg(s0 + (size_t)(64 * hb + e) * kD + v) : 0.f;
    // S0 enters the fp16 operand scaled by its power of two (dnS: the head's largest |S0| lands in
    // [0.5, 1)); the products are scaled back by upS
    float upS, dnS;
    {
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 64; ++e) m = fmaxf(m, fabsf(x0[e]));
      const uint32_t mw = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
      if (lane == 0) s0max[warp] = mw;
      __syncthreads();
      uint32_t mall = 0;
#pragma unroll
      for (int w8 = 0; w8 < kPrepThreads / 32; ++w8) mall = max(mall, s0max[w8]);
      pow2_scales(__uint_as_float(mall), upS, dnS);
    }
    {
      uint32_t r32[32];
#pragma unroll
      for (int c2 = 0; c2 < 32; ++c2) r32[c2] = pack_f16x2(x0[2 * c2] * dnS, x0[2 * c2 + 1] * dnS);
      tmem_st32(tb + lane_base + 32 * hb, r32);
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_d = idesc_f16(128, 128, false, false), id_o = idesc_f16(128, 64, false, false);
      const uint32_t mp = smem_u32(sm + kPM), qp = smem_u32(sm + kPV);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_f16_tmem_a(tb + 64, tb + kk * 8, smem_desc(mp + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), id_d,
                       kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_f16_tmem_a(tb + 192, tb + kk * 8, smem_desc(qp + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id_o,
                       kk > 0);
      mma_commit(&bar_mma);
    }
    ok = wait_mma();
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();
    if (write && a.S_T) {
      // S_T[i][v] for keys i = 64 hb .. + 63; N[i][v] from its staged fp16 slice
      float* so = a.S_T + (((size_t)b * a.Hv + h) * kD) * kD;
      const float gc = Gam[63];
      const uint8_t* nsl = sm + kPWS + (v >> 5) * 8192;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float d[32];
        tmem_ld32(tb + lane_base + 64 + 64 * hb + 32 * part, d);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int i = 64 * hb + 32 * part + e;
          const float n = __half2float(*reinterpret_cast<const __half*>(nsl + swz64(i * 64 + (v & 31) * 2)));
          so[(size_t)i * kD + v] = fmaf(gc, x0[32 * part + e], fmaf(upS, d[e], upV * n));
        }
      }
    }
    if (write) {
      // o at positions 32 hb .. + 31 of this chunk; (P U)[pos][v] from its staged fp16 slice. The
      // bf16 rows are staged over the consumed Q' image and leave by one bulk store per position.
      float ov[32];
      tmem_ld32(tb + lane_base + 192 + 32 * hb, ov);
      const uint8_t* psl = sm + kPV + 16384 + (v >> 5) * 4096;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int pos = 32 * hb + e;
        const float pu = __half2float(*reinterpret_cast<const __half*>(psl + swz64(pos * 64 + (v & 31) * 2)));
        *reinterpret_cast<__nv_bfloat16*>(sm + kPV + pos * 256 + v * 2) =
            __float2bfloat16_rn(fmaf(upS, ov[e], upV * pu));
      }
    }
    fence_async_smem();
    __syncthreads();
    if (write && tid < 64 && c * 64 + tid < a.L && c * 64 + tid < row_len(b)) {
      bulk_store(a.o + (((size_t)b * a.L + c * 64 + tid) * a.Hv + h) * kD, sm + kPV + tid * 256, 256);
      bulk_commit();
      bulk_wait_read();   // the next unit's tiles overwrite the staging
    }
  } else if (tid == 0) {
    bulk_store(ub, sm + kPM, kMBytes);
    bulk_commit();
    bulk_store(ub + kUnitN, sm + kPWS, kNBytes);   // its own group: it may drain into the next unit
    bulk_commit();
    // the next unit's tile loads overwrite q, k, v once the stores staged there have read them
    // (every group but the last, N, which is staged over AT and T)
    bulk_wait_read_but_last();
  }
  // the next unit's tile loads (async proxy) overwrite what this unit wrote to shared memory
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  u = un;
  if (u >= total) break;
  tiles(u, true);
  }   // units

  if (!ok && tid == 0) {
    set_error(a.err, kErrTimeout);
    // drain what this CTA still has in flight before its shared and tensor memory are released
    if (ld_fail >= 0) mbar_wait(&bar_ld, (uint32_t)ld_fail, kDrainBudget);
    if (mma_fail >= 0) mbar_wait(&bar_mma, (uint32_t)mma_fail, kDrainBudget);
  }
  cp_async_wait<0>();
  if (tid == 0) bulk_wait_read();
  tc_fence_before();
  __syncthreads();
  launch_dependents();   // the state kernel may start its set-up; it waits for this grid before reading
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 256);
  }
}

// -------------------------------------------------------------------------------------------
// Kernel 2: sequential state recurrence over chunks; four CTAs per (row, value head)
// -------------------------------------------------------------------------------------------
// CTA s (blockIdx.x) owns value columns [32 s, 32 s + 32) of one value head. The four CTAs of a
// head are independent: each reads the head's M' and Q' tiles itself (the other three read the
// same lines, so they come from L2) and its own slices of N and P U. No CTA waits on another.
// Warp roles (warp w reads TMEM lanes 32 (w % 4) .. + 31):
//   warps 0-3: own the state rows (key row = tid, 32 value columns, float32 registers), form
//              S = Gamma_C S + D + N and write its fp16 copy, the operand of the next products.
//   warps 4, 5 and 8, 9: output rows o = O' + P U for positions 0-63 (TMEM lanes 0-63), columns
//              0-15 (warps 4, 5) and 16-31 (warps 8, 9) of the slice; named barrier 2. Four
//              warps, so that the gated epilogue's per-position work is spread over two warps on
//              each of the two SMSPs that may read those TMEM lanes.
//   warp 6: loads the chain ring (M', this CTA's N slice, Gamma_C) up to CS chunks ahead, and
//           prefetches the chunk kPrefetchAhead beyond each load into L2.
//   warp 7: issues the output product O' = Q' S, so that its issue time stays off the chain.
//   warp 10: loads the output ring (Q', this CTA's P U slice) up to OS chunks ahead (with the
//           same L2 prefetch).
//   warp 11: issues the state product D = M' S (in a warp of its own, so that its issue is not
//           serialised with the state update of a diverged state warp).
// Per chunk c: chain stage c % CS (chFull / chFree: each state warp releases it after its
// update), output stage c % OS (outFull / outFree: released by the output warps), state operand
// q = c % kSb (opReady: the state warps have written S_c; sReady: the state product was issued, so
// the output product may read it too; sFree: the output product has read it), TMEM buffers
// p = c % 2 (D[p] with bar_d; O'[p] with bar_o: product done, oFree: the output warps have read
// it). Every barrier completes once per CS, OS, kSb, 2 chunks or per chunk, and none can run two
// phases ahead of its waiters.
constexpr int kStateThreads = 384;
constexpr uint32_t kOutBar = 2, kOutCount = 128;
constexpr int kOutCols = kN / 2;       // value columns per output warp
constexpr uint32_t kStateBar = 3;      // named barrier of the four state warps (the state scale)
constexpr uint32_t kCStage = 40960;    // M' (two 16 KB K-atoms), then this CTA's N slice (8 KB)
constexpr uint32_t kCN = 32768;
constexpr uint32_t kOStage = 20480;    // Q' (two 8 KB K-atoms), then this CTA's P U slice (4 KB)
constexpr uint32_t kOPU = 16384;
constexpr uint32_t kTmemState = 128;   // D[2] at 0, 32; O'[2] at 64, 96
// Rings: 3 chain and 3 output stages. After the rings: kSb fp16 state operands (MN-major, 128 rows
// of 64 B). The M = 128 output product reads 8 KB past each Q' tile
// (operand rows 64-127, whose products land in TMEM lanes nobody reads), which stays inside the
// buffer because the state operands follow the output ring.
constexpr int kPrefetchAhead = 3;      // ring loads also prefetch the chunk this far beyond them into L2
constexpr int kSb = 5;                 // fp16 state operands: the output path may trail the chain by 4 chunks
constexpr uint32_t state_smem(int cs, int os) { return cs * kCStage + os * kOStage + kSb * 8192 + 1024; }
static_assert(kCN == kMBytes && kOPU == kQBytes, "stage layout");

// kMode 0: the forward (o and S_T). kMode 1: the forward recomputed for the backward: no output
// side; the entering state of every chunk is saved (st_save, st_scale). kMode 2: the backward's adjoint
// chain dS <- Gamma_C dS + M'^T dS + Nb, chunks from the last to the first: the chain product reads
// the M' image transposed (an MN-major A operand); the output side forms Nb = Q'^T dO for the CTA's
// 32 columns a step or more ahead (the output ring brings Q' and a box of dO, tm_do; the output
// warps turn dO into fp16 divided by its power of two; warp 7 issues the product into the TMEM
// slots the forward's O' uses) and the state warps read it from TMEM; the initial state is dS_T
// (a.S0), the final one dS0 (a.S_T), and the adjoint entering each chunk's step (that of its
// exiting state) is saved likewise. kMode 3: the forward of kMode 0 that also saves what kMode 1
// saves (for a backward that then skips its forward passes); a state operand buffer is free once
// both the output product and its store have read it.
template <int CS, int OS, bool kGated, int kMode>
__global__ void __launch_bounds__(kStateThreads, 1)
chunk_state_kernel(const ChunkArgs a, const __grid_constant__ CUtensorMap tm_do) {
  constexpr bool kOut = kMode == 0 || kMode == 3;   // the output side forms o
  constexpr bool kNb = kMode == 2;    // the output side forms Nb = Q'^T dO
  constexpr uint32_t kOffO = CS * kCStage;
  constexpr uint32_t kOffSb = kOffO + OS * kOStage;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t chFull[CS], chFree[CS], outFull[OS], outFree[OS], bar_d, opReady, bar_o[2], oFree[2], sReady[kSb],
      sFree[kSb];
  __shared__ __align__(16) float4 gam_ring[CS];   // Gamma_C, upV of the chunk in each chain stage
  __shared__ __align__(16) float4 out_scl[OS];    // Gamma_C, upV of the chunk in each output stage
  __shared__ uint64_t scRdy[8];                    // the state scale of chunk c is in sc_ring[c % 8]
  __shared__ float sc_ring[8];
  __shared__ uint32_t smax[2][4];                  // per state warp: largest |S| of its rows of the slice
  // gated epilogue: red[p][2 r + hc][i] = the sum of o^2 over the 16 values of column half hc of
  // CTA r at position i of a chunk of parity p (written by CTA r into every CTA of the cluster as
  // asynchronous stores that complete transaction bytes on the receiver's fullR[p]); fullR[p]: all
  // 8 x 64 partials of the chunk are here (one local arrival posts the 2048 bytes); freeR[p]: every
  // CTA of the cluster has read its red[p], so it may be rewritten (one arrival per CTA)
  __shared__ float red[kGated ? 2 : 1][2 * kSlices][64];
  __shared__ uint64_t fullR[2], freeR[2];
  __shared__ __align__(16) float w_s[kN];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  // kMode 2: doRdy[s]: the dO box of output stage s is fp16 (for the product's issuer); nbRdy[c % 8]:
  // its scale is in nb_scl[c % 8] (for the state warps, which the output warps may lead by up to five
  // chunks: an eight-deep ring never runs two phases ahead of them, a three-deep one would)
  __shared__ uint64_t doRdy[OS], nbRdy[8];
  __shared__ float nb_scl[8];
  __shared__ uint32_t nbmax[4];

  const int sl = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // With row lengths (up to 64 rows), the grid's z index is a rank: z runs the row with the z-th
  // most chunks (ties by row index), so that CTAs, which launch in z order, start the longest chains
  // first and the shorter rows fill the SMs around them. Every warp ranks the rows itself (a lane per
  // row, a scan of the lengths); a length outside [0, L] counts as no chunks.
  int b = blockIdx.z;
  if (a.lengths && gridDim.z > 1 && gridDim.z <= 64) {
    const int nrows = (int)gridDim.z;
    auto nchunks = [&](int r) {
      const int l = a.lengths[r];
      return (l < 0 || l > a.L) ? 0 : (l + kChunk - 1) / kChunk;
    };
    int found = -1;
    for (int r = lane; r < nrows; r += 32) {
      const int nr = nchunks(r);
      int rank = 0;
      for (int q = 0; q < nrows; ++q) {
        const int nq = nchunks(q);
        rank += (nq > nr || (nq == nr && q < r)) ? 1 : 0;
      }
      if (rank == (int)blockIdx.z) found = r;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) found = max(found, __shfl_xor_sync(0xffffffffu, found, o));
    b = found;   // (the ranks are a permutation of 0 .. nrows - 1: exactly one row has this one)
  }
  // the row's valid tokens: chunks wholly past them are not run (the state there is final) and
  // output positions past them are not written; a length outside [0, L] skips the row
  const int len = a.lengths ? a.lengths[b] : a.L;
  const bool bad_len = len < 0 || len > a.L;
  const int NC = bad_len ? 0 : (len + kChunk - 1) / kChunk;

  if (tid == 0) {
    for (int s = 0; s < CS; ++s) {
      mbar_init(&chFull[s], 1);
      mbar_init(&chFree[s], 4);
    }
    for (int s = 0; s < OS; ++s) {
      mbar_init(&outFull[s], 1);
      mbar_init(&outFree[s], 1);
    }
    mbar_init(&bar_d, 1);
    mbar_init(&opReady, 4);
    for (int p = 0; p < 2; ++p) {
      mbar_init(&bar_o[p], 1);
      mbar_init(&oFree[p], 1);
    }
    for (int q = 0; q < kSb; ++q) {
      mbar_init(&sReady[q], 1);
      mbar_init(&sFree[q], kMode == 3 ? 2 : 1);
    }
    for (int r = 0; r < 8; ++r) mbar_init(&scRdy[r], 4);
    for (int s2 = 0; s2 < OS; ++s2) mbar_init(&doRdy[s2], 1);
    for (int r = 0; r < 8; ++r) mbar_init(&nbRdy[r], 1);
    if (kGated) {
      for (int q = 0; q < 2; ++q) {
        mbar_init(&fullR[q], 1);
        mbar_init(&freeR[q], kSlices);
      }
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (kGated && tid < kN) w_s[tid] = a.w[sl * kN + tid];
  if (warp == 0) tmem_alloc(&tmem_base, kTmemState);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (kGated) cluster_sync_all();   // every CTA's barriers are initialised before any remote arrive
  const uint32_t tb = tmem_base;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  bool ok = true;
  // the row's initial state: S0[b], or for forks the trunk state S0[S0_idx[b]]; an index out of
  // range skips the row entirely (nothing of it is written) and records the error
  size_t s0row = b;
  bool skip = bad_len;
  if (skip && tid == 0) set_error(a.err, kErrDeviceIndex);
  if (a.S0_idx) {
    const long long ix = a.S0_idx[b];
    skip = skip || ix < 0 || ix >= a.n_S0;
    s0row = (ix < 0 || ix >= a.n_S0) ? 0 : (size_t)ix;
    if ((ix < 0 || ix >= a.n_S0) && tid == 0) set_error(a.err, kErrDeviceIndex);
  }

  if (skip) {
    // every CTA of the row reads the same index and skips
  } else if (warp == 6 || warp == 10) {
    // ---------------- producers (lane 0): the chain ring (warp 6) and the output ring (warp 10) ---
    if (lane == 0 && (warp == 6 || kOut || kNb)) {
      wait_prerequisite();   // the workspace is complete once the prep kernel has finished
      const bool chain = warp == 6;
      const int S = chain ? CS : OS;
      int last = -1;   // last chunk whose tiles were issued
      for (int c = 0; c < NC; ++c) {
        const int s = c % S;
        if (c >= S) ok = mbar_wait(chain ? &chFree[s] : &outFree[s], ((c - S) / S) & 1, a.wait_budget);
        if (!ok || *(volatile int*)&abort_flag) break;
        const int cu = kMode == 2 ? NC - 1 - c : c;   // the chunk of step c
        const uint8_t* ub = unit_base(a, b, h, cu);
        if (chain) {
          uint8_t* st = sm + s * kCStage;
          mbar_arrive_expect_tx(&chFull[s], kMBytes + (kNb ? 0 : 8192) + kSCopy);
          bulk_load(st, ub, 16384, &chFull[s]);
          bulk_load(st + 16384, ub + 16384, 16384, &chFull[s]);
          if (!kNb) bulk_load(st + kCN, ub + kUnitN + sl * 8192, 8192, &chFull[s]);   // (Nb comes from TMEM)
          bulk_load(&gam_ring[s], ub + kUnitS, kSCopy, &chFull[s]);
          if (c + kPrefetchAhead < NC) {   // the chunk kPrefetchAhead steps further on into L2
            const uint8_t* uf = unit_base(a, b, h, kMode == 2 ? cu - kPrefetchAhead : cu + kPrefetchAhead);
            bulk_prefetch_l2(uf, kMBytes);
            if (!kNb) bulk_prefetch_l2(uf + kUnitN + sl * 8192, 8192);
          }
        } else if (kNb) {
          // Q' and this CTA's 32 columns of dO (a 64 x 32 box, 64-byte swizzle) over the P U slot
          uint8_t* st = sm + kOffO + s * kOStage;
          mbar_arrive_expect_tx(&outFull[s], kQBytes + 4096);
          bulk_load(st, ub + kUnitQ, kQBytes, &outFull[s]);
          tma_load_4d(st + kOPU, &tm_do, &outFull[s], sl * kN, h, cu * kChunk, b);
          if (c + kPrefetchAhead < NC) {
            bulk_prefetch_l2(unit_base(a, b, h, cu - kPrefetchAhead) + kUnitQ, kQBytes);
            tma_prefetch_4d(&tm_do, sl * kN, h, (cu - kPrefetchAhead) * kChunk, b);
          }
        } else {
          uint8_t* st = sm + kOffO + s * kOStage;
          mbar_arrive_expect_tx(&outFull[s], kQBytes + 4096 + kSCopy);
          bulk_load(st, ub + kUnitQ, kQBytes, &outFull[s]);
          bulk_load(st + kOPU, ub + kUnitPU + sl * 4096, 4096, &outFull[s]);
          bulk_load(&out_scl[s], ub + kUnitS, kSCopy, &outFull[s]);
          if (c + kPrefetchAhead < NC) {
            const uint8_t* uf = unit_base(a, b, h, c + kPrefetchAhead);
            bulk_prefetch_l2(uf + kUnitQ, kQBytes);
            bulk_prefetch_l2(uf + kUnitPU + sl * 4096, 4096);
          }
        }
        last = c;
      }
      if (!ok) {
        // drain: the tiles of the last S issued chunks land before the CTA's memory is released
        for (int c = (last - S + 1 > 0 ? last - S + 1 : 0); c <= last; ++c)
          mbar_wait(chain ? &chFull[c % S] : &outFull[c % S], (c / S) & 1, kDrainBudget);
      }
    }
  } else if (warp < 4) {
    // ---------------- state warps ----------------
    const int kr = tid;
    float Sm[kN];
#pragma unroll
    for (int n = 0; n < kN; ++n) Sm[n] = 0.f;
    if (a.S0) {
      const float* s0 = a.S0 + ((s0row * a.Hv + h) * kD + kr) * kD + sl * kN;
#pragma unroll
      for (int n = 0; n < kN; n += 4) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(s0 + n));
        Sm[n] = x.x; Sm[n + 1] = x.y; Sm[n + 2] = x.z; Sm[n + 3] = x.w;
      }
    }
    // The fp16 copy of S_c is S_c / sc_c with sc_c the power of two of max |S_c| over this CTA's
    // slice (a function of the state alone: results do not depend on where a sequence is split, and
    // scaling (v, S0) by 2^k scales every sc_c by 2^k). The four state warps take the maximum
    // together (one named barrier per chunk); sc_c goes to the output warps through sc_ring.
    int mpar = 0;   // which half of smax the next maximum uses (a warp may start the next chunk's
                    // maximum while another still reads this one)
    auto slice_scale = [&](bool ok_in, float& up, float& dn) -> bool {
      float m = 0.f;
#pragma unroll
      for (int n = 0; n < kN; ++n) m = fmaxf(m, fabsf(Sm[n]));
      const uint32_t mw = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
      if (lane == 0) smax[mpar][warp] = mw;
      const bool all = named_bar_and(kStateBar, 128, ok_in);
      const uint32_t mall = max(max(smax[mpar][0], smax[mpar][1]), max(smax[mpar][2], smax[mpar][3]));
      mpar ^= 1;
      pow2_scales(__uint_as_float(mall), up, dn);
      return all;
    };
    // fp16 state operand q: MN-major, row kr = 32 value columns (64 bytes), 64-byte swizzle. Modes 1
    // and 2 save its scale up as that of the state at the top of step `step` (if < NC); the operand
    // itself leaves by the state-product issuer's bulk store.
    auto write_state_operand = [&](int q, float dn, int step, float up) {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = Sm[8 * ch + e] * dn;
        *reinterpret_cast<uint4*>(sm + kOffSb + q * 8192 + swz64(kr * 64 + ch * 16)) = pack8_f16(t);
      }
      if (kMode != 0 && step < NC && kr == 0) {
        const int cu = kMode == 2 ? NC - 1 - step : step;
        a.st_scale[(((size_t)b * a.Hv + h) * NC + cu) * kSlices + sl] = up;
      }
    };
    float sc, dn;
    slice_scale(true, sc, dn);
    write_state_operand(0, dn, 0, sc);
    if (tid == 0) sc_ring[0] = sc;
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&opReady);     // S_0 is in Sb[0]
      mbar_arrive(&scRdy[0]);    // and its scale in sc_ring[0]
    }
    for (int c = 0; c < NC; ++c) {
      const int cs = c % CS, p = c & 1, qn = (c + 1) % kSb;
      const uint8_t* st = sm + cs * kCStage;
      ok = ok && mbar_wait(&chFull[cs], (c / CS) & 1, a.wait_budget) && !*(volatile int*)&abort_flag;
      if ((kMode == 1 || kMode == 3) && sl == 0 && tid == 0 && ok)
        a.unit_scale[(((size_t)b * a.Hv + h) * NC + c) * 8 + 4] = gam_ring[cs].y;   // v's power of two
      if (kNb) {
        // Nb_c = Q'_c^T dO_c in TMEM slot p (and its scale in nb_scl)
        ok = ok && mbar_wait(&nbRdy[c & 7], (c >> 3) & 1, a.wait_budget) &&
             mbar_wait(&bar_o[p], (c >> 1) & 1, a.wait_budget);
        ok = __all_sync(0xffffffffu, ok);   // the TMEM load below is warp-collective
      }
      if (ok) {
        // while the product D = M' S_c runs: S <- Gamma_C S + upV N (S_c is already in the fp16
        // operand; N is in its chunk's v scale upV), or S <- Gamma_C S + Nb in the adjoint chain
        const float gc = gam_ring[cs].x;
        if (kNb) {
          tc_fence_after();
          float nb[kN];
          tmem_ld32(tb + lane_base + 64 + 32 * p, nb);
          const float up = nb_scl[c & 7];
#pragma unroll
          for (int n = 0; n < kN; ++n) Sm[n] = fmaf(gc, Sm[n], up * nb[n]);
          tc_fence_before();
        } else {
          const float upV = gam_ring[cs].y;
          const uint8_t* nrow = st + kCN;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            float nv[8];
            unpack8_f16(*reinterpret_cast<const uint4*>(nrow + swz64(kr * 64 + ch * 16)), nv);
#pragma unroll
            for (int e = 0; e < 8; ++e) Sm[8 * ch + e] = fmaf(gc, Sm[8 * ch + e], upV * nv[e]);
          }
        }
        // Sb[qn] is rewritten below: the output product (modes 1, 2: the bulk store; mode 3: both)
        // of chunk c + 1 - kSb must have read it
        ok = mbar_wait(&bar_d, c & 1, a.wait_budget) &&
             (c + 1 < kSb || mbar_wait(&sFree[qn], ((c + 1 - kSb) / kSb) & 1, a.wait_budget));
      }
      ok = __all_sync(0xffffffffu, ok);   // the TMEM load below is warp-collective
      if (ok) {
        tc_fence_after();
        float d[kN];
        tmem_ld32(tb + lane_base + 32 * p, d);
#pragma unroll
        for (int n = 0; n < kN; ++n) Sm[n] = fmaf(sc, d[n], Sm[n]);   // D = M' (S_c / sc_c)
      }
      // every state warp reaches this barrier once per chunk, so a warp that gave up stops them all
      ok = slice_scale(ok, sc, dn);
      if (!ok) break;
      if (kNb && tid == 0) mbar_arrive(&oFree[p]);   // the four state warps have read Nb's slot
      write_state_operand(qn, dn, c + 1, sc);
      if (tid == 0) sc_ring[(c + 1) & 7] = sc;
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&opReady);                        // S_{c+1} is in Sb[qn]
        mbar_arrive(&scRdy[(c + 1) & 7]);             // and its scale in sc_ring
        if (c + CS < NC) mbar_arrive(&chFree[cs]);   // this warp is done with N and Gamma_C
      }
    }
    if (ok && a.S_T) {
      float* dst = a.S_T + (((size_t)b * a.Hv + h) * kD + kr) * kD + sl * kN;
#pragma unroll
      for (int n = 0; n < kN; n += 4)
        *reinterpret_cast<float4*>(dst + n) = make_float4(Sm[n], Sm[n + 1], Sm[n + 2], Sm[n + 3]);
    }
  } else if (warp == 11) {
    // ---------------- state-product issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, kN, kMode == 2, true);
      int last = -1;   // last chunk whose state product was issued
      for (int c = 0; c < NC; ++c) {
        const int cs = c % CS, p = c & 1, q = c % kSb;
        ok = mbar_wait(&chFull[cs], (c / CS) & 1, a.wait_budget) && mbar_wait(&opReady, c & 1, a.wait_budget);
        if (!ok || *(volatile int*)&abort_flag) break;
        tc_fence_after();
        const uint32_t sb = smem_u32(sm + kOffSb + q * 8192);
        const uint32_t sm_m = smem_u32(sm + cs * kCStage);
        // D[p] = M' S_c: the product on the chain (kMode 2: M'^T dS, the K-major M' image read as an
        // MN-major operand: K-row j is row j of M', the two 64-row M blocks its two column atoms)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t adesc = kMode == 2 ? smem_desc(sm_m + kk * 2048, 16384, 1024)
                                            : smem_desc(sm_m + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          mma_bf16(tb + 32 * p, adesc, smem_desc(sb + kk * 1024, 4096, 512, kSwizzle64B), idesc, kk > 0);
        }
        mma_commit(&bar_d);
        mbar_arrive(&sReady[q]);   // Sb[q] holds S_c: warp 7 may issue the output product
        if (kMode != 0) {
          // modes 1, 2, 3: the step's operand (the state at its top, over its slice's power of two)
          // to st_save; the previous step's buffer is free once its store has read it (mode 3:
          // and once the output product has read it, the barrier's other arrival)
          const int cu = kMode == 2 ? NC - 1 - c : c;
          bulk_store(a.st_save + (((size_t)b * a.Hv + h) * NC + cu) * kD * kD + sl * kD * kN, sm + kOffSb + q * 8192,
                     8192);
          bulk_commit();
          if (c > 0) {
            bulk_wait_read_but_last();
            mbar_arrive(&sFree[(c - 1) % kSb]);
          }
        }
        last = c;
      }
      if (!ok && last >= 0) mbar_wait(&bar_d, last & 1, kDrainBudget);   // drain
      if (kMode != 0) bulk_wait_all();   // the saved states are complete before the kernel ends
    }
  } else if (warp == 7) {
    // ---------------- output-product issuer ----------------
    if (lane == 0 && kNb) {
      // Nb[p] = Q'^T dO: A = the Q' image read as an MN-major operand (keys = M in its two 64-column
      // atoms 8 KB apart, positions = K in rows of 128 B), B = the fp16 dO box (positions = K in rows
      // of 64 B, 64-byte swizzle, N = 32)
      const uint32_t idesc = idesc_f16(128, kN, true, true);
      int last = -1;
      for (int c = 0; c < NC; ++c) {
        const int os = c % OS, p = c & 1;
        ok = mbar_wait(&doRdy[os], (c / OS) & 1, a.wait_budget) &&
             (c < 2 || mbar_wait(&oFree[p], ((c - 2) >> 1) & 1, a.wait_budget));
        if (!ok || *(volatile int*)&abort_flag) break;
        tc_fence_after();
        const uint32_t sq = smem_u32(sm + kOffO + os * kOStage), sd = sq + kOPU;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tb + 64 + 32 * p, smem_desc(sq + kk * 2048, 8192, 1024),
                   smem_desc(sd + kk * 1024, 4096, 512, kSwizzle64B), idesc, kk > 0);
        mma_commit(&bar_o[p]);
        mma_commit(&outFree[os]);   // the stage is read once the product completes
        last = c;
      }
      if (!ok && last >= 0) mbar_wait(&bar_o[last & 1], (last >> 1) & 1, kDrainBudget);   // drain
    } else if (lane == 0 && kOut) {
      const uint32_t idesc = idesc_f16(128, kN, false, true);
      int last = -1;   // last chunk whose output product was issued
      for (int c = 0; c < NC; ++c) {
        const int os = c % OS, p = c & 1, q = c % kSb;
        ok = mbar_wait(&outFull[os], (c / OS) & 1, a.wait_budget) &&
             mbar_wait(&sReady[q], (c / kSb) & 1, a.wait_budget) &&
             (c < 2 || mbar_wait(&oFree[p], ((c - 2) >> 1) & 1, a.wait_budget));
        if (!ok || *(volatile int*)&abort_flag) break;
        tc_fence_after();
        const uint32_t sb = smem_u32(sm + kOffSb + q * 8192);
        const uint32_t sm_q = smem_u32(sm + kOffO + os * kOStage);
        // O'[p] = Q' S  (M = 128; operand rows 64-127 run past the tile and are not read)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16(tb + 64 + 32 * p, smem_desc(sm_q + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                   smem_desc(sb + kk * 1024, 4096, 512, kSwizzle64B), idesc, kk > 0);
        mma_commit(&bar_o[p]);
        mma_commit(&sFree[q]);
        last = c;
      }
      if (!ok && last >= 0) mbar_wait(&bar_o[last & 1], (last >> 1) & 1, kDrainBudget);   // drain
    }
  } else if (kNb) {
    // ---------------- output warps 4, 5, 8, 9 (adjoint chain): the dO box to fp16 ----------------
    const int ot = (warp < 8 ? tid - 128 : tid - 192);   // 0 .. 127
    const int wi = ot >> 5;
    for (int c = 0; c < NC; ++c) {
      const int os = c % OS;
      ok = ok && mbar_wait(&outFull[os], (c / OS) & 1, a.wait_budget) && !*(volatile int*)&abort_flag;
      uint4* box = reinterpret_cast<uint4*>(sm + kOffO + os * kOStage + kOPU);   // 256 chunks of 16 B
      uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
      uint32_t m2 = 0;
      if (ok) {
        w0 = box[ot];
        w1 = box[ot + 128];
        m2 = __vmaxu2(__vmaxu2(__vmaxu2(w0.x & 0x7FFF7FFFu, w0.y & 0x7FFF7FFFu), __vmaxu2(w0.z & 0x7FFF7FFFu, w0.w & 0x7FFF7FFFu)),
                      __vmaxu2(__vmaxu2(w1.x & 0x7FFF7FFFu, w1.y & 0x7FFF7FFFu), __vmaxu2(w1.z & 0x7FFF7FFFu, w1.w & 0x7FFF7FFFu)));
      }
      const uint32_t mw = __reduce_max_sync(0xffffffffu, max(m2 & 0xFFFFu, m2 >> 16));
      if (lane == 0) nbmax[wi] = mw;
      if (!named_bar_and(kOutBar, kOutCount, ok)) break;
      float up, dn;
      pow2_scales(__uint_as_float(max(max(nbmax[0], nbmax[1]), max(nbmax[2], nbmax[3])) << 16), up, dn);
      box[ot] = make_uint4(bf16x2_to_f16x2_scaled(w0.x, dn), bf16x2_to_f16x2_scaled(w0.y, dn),
                           bf16x2_to_f16x2_scaled(w0.z, dn), bf16x2_to_f16x2_scaled(w0.w, dn));
      box[ot + 128] = make_uint4(bf16x2_to_f16x2_scaled(w1.x, dn), bf16x2_to_f16x2_scaled(w1.y, dn),
                                 bf16x2_to_f16x2_scaled(w1.z, dn), bf16x2_to_f16x2_scaled(w1.w, dn));
      fence_async_smem();   // generic writes, then the product (async proxy) reads them
      if (!named_bar_and(kOutBar, kOutCount, true)) break;
      if (ot == 0) {
        nb_scl[c & 7] = up;
        mbar_arrive(&nbRdy[c & 7]);
        mbar_arrive(&doRdy[os]);
        a.unit_scale[(((size_t)b * a.Hv + h) * NC + (NC - 1 - c)) * 8 + sl] = up;   // dO's power of two
      }
    }
  } else if (kOut) {
    // ---------------- output warps 4, 5, 8, 9 ----------------
    const int i = 32 * (warp & 1) + lane;   // position in the chunk = TMEM lane
    const int hc = warp >> 3;               // column half: slice columns 16 hc .. 16 hc + 15
    const int col0 = sl * kN + kOutCols * hc;
    // gated: this thread's 16 gate values z of the chunk, loaded one chunk ahead
    uint4 zc[2] = {};
    auto load_z = [&](int c) {
      const int pos = c * 64 + i;
      if (kGated && c < NC && pos < len) {
        const uint4* zrow = reinterpret_cast<const uint4*>(a.z + (((size_t)b * a.L + pos) * a.Hv + h) * kD + col0);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) zc[ch] = __ldg(zrow + ch);
      }
    };
    load_z(0);
    for (int c = 0; c < NC && ok; ++c) {
      const int os = c % OS, p = c & 1;
      const uint8_t* st = sm + kOffO + os * kOStage;
      ok = mbar_wait(&outFull[os], (c / OS) & 1, a.wait_budget) &&
           mbar_wait(&bar_o[p], (c >> 1) & 1, a.wait_budget) &&
           mbar_wait(&scRdy[c & 7], (c >> 3) & 1, a.wait_budget) && !*(volatile int*)&abort_flag;
      ok = __all_sync(0xffffffffu, ok);   // the TMEM load below is warp-collective
      if (ok) {
        tc_fence_after();
        float qs[kOutCols];
        tmem_ld16(tb + lane_base + 64 + 32 * p + kOutCols * hc, qs);
        const int pos = c * 64 + i;
        float pu[kOutCols];
        const uint8_t* purow = st + kOPU;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
          unpack8_f16(*reinterpret_cast<const uint4*>(purow + swz64(i * 64 + (2 * hc + ch) * 16)), pu + 8 * ch);
        const float upV = out_scl[os].y;   // P U is in its chunk's v scale
        const float sc = sc_ring[c & 7];     // O' = Q' (S_c / sc_c)
#pragma unroll
        for (int n = 0; n < kOutCols; ++n) qs[n] = fmaf(sc, qs[n], upV * pu[n]);
        if (kGated) {
          // o (float32) for these 16 values, its sum of squares to every CTA of the cluster, then
          // w * o / rms(o) * silu(z) once all eight partials of the position are in
          float ss = 0.f;
#pragma unroll
          for (int n = 0; n < kOutCols; ++n) ss = fmaf(qs[n], qs[n], ss);
          // red[p] of every CTA may be rewritten once every CTA has read it for chunk c - 2
          ok = c < 2 || mbar_wait(&freeR[p], ((c >> 1) - 1) & 1, a.wait_budget);
          if (ok) {
            if (tid == 128) mbar_arrive_expect_tx(&fullR[p], 2 * kSlices * 64 * 4);
#pragma unroll
            for (uint32_t r = 0; r < kSlices; ++r)
              st_async_f32(dsmem_addr(&red[p][2 * sl + hc][i], r), ss, dsmem_addr(&fullR[p], r));
            // while the partials travel: w silu(z), which does not depend on o
            float gz[kOutCols];
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
              const uint32_t zu[4] = {zc[ch].x, zc[ch].y, zc[ch].z, zc[ch].w};
              const float4 w0 = reinterpret_cast<const float4*>(w_s + kOutCols * hc)[2 * ch];
              const float4 w1 = reinterpret_cast<const float4*>(w_s + kOutCols * hc)[2 * ch + 1];
              const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float zz = __uint_as_float((e & 1) ? (zu[e >> 1] & 0xFFFF0000u) : (zu[e >> 1] << 16));
                gz[8 * ch + e] = wv[e] * __fdividef(zz, 1.f + __expf(-zz));
              }
            }
            ok = mbar_wait(&fullR[p], (c >> 1) & 1, a.wait_budget);
            if (ok) {
              float tot = 0.f;
#pragma unroll
              for (int r = 0; r < 2 * kSlices; ++r) tot += red[p][r][i];
              const float rs = rsqrtf(tot * (1.f / kD) + a.eps);
              if (pos < len) {
                __nv_bfloat16* orow_p = a.o + (((size_t)b * a.L + pos) * a.Hv + h) * kD + col0;
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                  float y[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) y[e] = (qs[8 * ch + e] * rs) * gz[8 * ch + e];
                  *reinterpret_cast<uint4*>(orow_p + 8 * ch) = pack8_bf16(y);
                }
              }
              load_z(c + 1);
            }
          }
        } else if (pos < len) {
          __nv_bfloat16* orow_p = a.o + (((size_t)b * a.L + pos) * a.Hv + h) * kD + col0;
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) *reinterpret_cast<uint4*>(orow_p + 8 * ch) = pack8_bf16(qs + 8 * ch);
        }
      }
      tc_fence_before();
      if (!named_bar_and(kOutBar, kOutCount, ok)) break;
      if (tid == 128) {
        mbar_arrive(&oFree[p]);
        if (c + OS < NC) mbar_arrive(&outFree[os]);   // the Q' product complete, P U read
        if (kGated) {
          // both output warps of each column half have read red[p]: every CTA may rewrite it
#pragma unroll
          for (uint32_t r = 0; r < kSlices; ++r) remote_arrive_relaxed(&freeR[p], r);
        }
      }
    }
  }
  if (!ok) {
    atomicExch(&abort_flag, 1);
    set_error(a.err, kErrTimeout);
  }
  __syncwarp();         // the producer and issuer warps' lanes reconverge before the block barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, kTmemState);
  }
  // no CTA of the cluster leaves while another may still write its shared memory (every thread of
  // every CTA reaches this point: all loops above are bounded)
  if (kGated) cluster_sync_all();
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

// [B, L, H, 128] bf16 tensor, box {width columns, 1 head, 64 positions, 1 row}: 64 columns with
// 128-byte swizzle (the prep kernel's tiles) or 32 with 64-byte swizzle (the adjoint chain's dO box).
bool make_map(CUtensorMap* m, const void* base, int B, int L, int H, int width = 64) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2, (cuuint64_t)L * H * kD * 2};
  cuuint32_t box[4] = {(cuuint32_t)width, 1, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, width == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// SMs of the current device (cached per device ordinal)
int num_sms() {
  static int cache[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

size_t units_bytes(int B, int L, int Hv) {
  return (size_t)B * Hv * ((L + kChunk - 1) / kChunk) * kUnitBytes;
}

}  // namespace

size_t chunk_workspace_bytes(int B, int Hk, int L, int Hv) {
  (void)Hk;
  if (L <= kChunk) return 0;   // single-chunk rows are finished by kernel 1 without a workspace
  return units_bytes(B, L, Hv) + 1024;
}

cudaError_t launch_chunk_bf16(const ChunkLaunch& p, cudaStream_t s) {
  CUtensorMap mq{}, mk{}, mv{};   // (the fused prologue forms its tiles without them)
  if (!p.mixed && (!make_map(&mq, p.q, p.B, p.L, p.Hk) || !make_map(&mk, p.k, p.B, p.L, p.Hk) ||
                   !make_map(&mv, p.v, p.B, p.L, p.Hv)))
    return cudaErrorInvalidValue;
  ChunkArgs a{};
  a.g = p.g;
  a.beta = p.beta;
  a.S0 = p.S0;
  a.S0_idx = p.S0_idx;
  a.n_S0 = p.n_S0;
  // (with the fused prologue, rows of one chunk also take the two-kernel path through the workspace)
  a.fused = (p.L <= kChunk && !p.mixed) ? 1 : 0;
  a.wait_budget = wait_budget_cycles();
  a.o = static_cast<__nv_bfloat16*>(p.o);
  a.S_T = p.S_T;
  a.ws = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p.ws) + 1023) & ~uintptr_t(1023));
  a.B = p.B;
  a.L = p.L;
  a.Hk = p.Hk;
  a.Hv = p.Hv;
  a.NC = (p.L + kChunk - 1) / kChunk;
  a.err = p.err;
  a.lengths = p.lengths;
  a.z = static_cast<const __nv_bfloat16*>(p.z);
  a.w = p.w;
  a.eps = p.eps;
  a.mixed = static_cast<const __nv_bfloat16*>(p.mixed);
  a.tail = static_cast<const __nv_bfloat16*>(p.tail);
  a.conv_w = p.conv_w;
  a.proj_a = p.proj_a;
  a.proj_b = p.proj_b;
  a.A_log = p.A_log;
  a.dt_bias = p.dt_bias;
  a.C = (2 * p.Hk + p.Hv) * kD;
  const bool pro = p.mixed != nullptr;   // the prologue fused into the prep kernel

  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
  if (e == cudaSuccess && pro)
    e = cudaFuncSetAttribute(chunk_prep_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(p.z ? chunk_state_kernel<3, 3, true, 0> : chunk_state_kernel<3, 3, false, 0>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem(3, 3));
  if (e != cudaSuccess) return e;
  int slot = stage_timer_begin(s, kKernChunkPrep);
  const long long units = (long long)a.B * a.Hv * a.NC;
  const int grid = (int)std::min<long long>(units, 2ll * num_sms());
  if (pro)
    chunk_prep_kernel<false, true><<<grid, kPrepThreads, kPrepSmem, s>>>(mq, mk, mv, a);
  else if (a.fused)
    chunk_prep_kernel<true><<<grid, kPrepThreads, kPrepSmem, s>>>(mq, mk, mv, a);
  else
    chunk_prep_kernel<false><<<grid, kPrepThreads, kPrepSmem, s>>>(mq, mk, mv, a);
  stage_timer_end(slot, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.fused) {
    // single-chunk rows are complete after kernel 1; the gated epilogue then runs over o in place
    if (!p.z) return cudaSuccess;
    EpilogueArgs ea{p.o, p.z, p.w, p.eps, p.o, (long long)p.B * p.L * p.Hv};
    return launch_gated_rmsnorm(ea, s);
  }
  slot = stage_timer_begin(s, kKernChunkState);
  // launched as a programmatic dependent of the prep kernel: its set-up (barriers, tensor memory,
  // the initial state) overlaps the prep kernel's tail; its loads of the workspace wait for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSlices, p.Hv, p.B);
  cfg.blockDim = dim3(kStateThreads, 1, 1);
  cfg.dynamicSmemBytes = state_smem(3, 3);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // the gated epilogue reduces over a head's 128 values: its four column CTAs form a cluster
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kSlices;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.z ? 2 : 1;
  const CUtensorMap no_map{};   // (the forward's state kernel reads no dO)
  e = p.z ? cudaLaunchKernelEx(&cfg, chunk_state_kernel<3, 3, true, 0>, a, no_map)
          : cudaLaunchKernelEx(&cfg, chunk_state_kernel<3, 3, false, 0>, a, no_map);
  stage_timer_end(slot, s);
  if (e != cudaSuccess) return e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (pro && p.new_tail) {
    // the carry for the next call: ext positions L .. L + 2 of every row, ext = [tail; mixed], i.e.
    // tail rows L .. 2 (zeros without a tail) when L < 3, then mixed rows max(L - 3, 0) .. L - 1
    const size_t row = (size_t)a.C * 2;
    const int nt = std::max(0, 3 - p.L), nm = 3 - nt;
    uint8_t* dst = static_cast<uint8_t*>(p.new_tail);
    if (nt > 0)
      e = p.tail ? cudaMemcpy2DAsync(dst, 3 * row, static_cast<const uint8_t*>(p.tail) + (size_t)p.L * row, 3 * row,
                                     nt * row, (size_t)p.B, cudaMemcpyDeviceToDevice, s)
                 : cudaMemset2DAsync(dst, 3 * row, 0, nt * row, (size_t)p.B, s);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(dst + nt * row, 3 * row,
                            static_cast<const uint8_t*>(p.mixed) + (size_t)(p.L - nm) * row, (size_t)p.L * row,
                            nm * row, (size_t)p.B, cudaMemcpyDeviceToDevice, s);
  }
  return e;
}

size_t chunk_prologue_workspace_bytes(int B, int L, int Hv) { return units_bytes(B, L, Hv) + 1024; }

size_t chunk_bwd_units_bytes(int B, int L, int Hv) { return units_bytes(B, L, Hv) + 1024; }

cudaError_t launch_chunk_bwd_chain(const ChunkBwdChainLaunch& p, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, p.q, p.B, p.L, p.Hk) || !make_map(&mk, p.k, p.B, p.L, p.Hk) ||
      !make_map(&mv, p.v, p.B, p.L, p.Hv) || !make_map(&mo, p.dO, p.B, p.L, p.Hv, kN))
    return cudaErrorInvalidValue;
  ChunkArgs a{};
  a.g = p.g;
  a.beta = p.beta;
  a.S0 = p.S0;
  a.fused = 0;   // rows of one chunk also go through the workspace: the backward needs their factors
  a.wait_budget = wait_budget_cycles();
  a.ws = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p.ws) + 1023) & ~uintptr_t(1023));
  a.B = p.B;
  a.L = p.L;
  a.Hk = p.Hk;
  a.Hv = p.Hv;
  a.NC = (p.L + kChunk - 1) / kChunk;
  a.err = p.err;
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_state_kernel<3, 3, false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             state_smem(3, 3));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_state_kernel<3, 3, false, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             state_smem(3, 3));
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.B * a.Hv * a.NC;
  int slot = -1;
  if (!p.saved) {
    // 1. the forward's chunk factors
    slot = stage_timer_begin(s, kKernChunkPrep);
    chunk_prep_kernel<false><<<(int)std::min<long long>(units, 2ll * num_sms()), kPrepThreads, kPrepSmem, s>>>(mq, mk, mv, a);
    stage_timer_end(slot, s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // 2. the chunk-entry states (a programmatic dependent of the prep kernel, as in the forward)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSlices, p.Hv, p.B);
  cfg.blockDim = dim3(kStateThreads, 1, 1);
  cfg.dynamicSmemBytes = state_smem(3, 3);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  a.st_save = p.S_save;
  a.st_scale = p.S_scale;
  a.unit_scale = p.unit_scale;
  a.S_T = nullptr;
  if (!p.saved) {
    const CUtensorMap no_map{};   // (the forward pass reads no dO)
    slot = stage_timer_begin(s, kKernChunkState);
    e = cudaLaunchKernelEx(&cfg, chunk_state_kernel<3, 3, false, 1>, a, no_map);
    stage_timer_end(slot, s);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // 3. the adjoint chain (Nb = Q'^T dO formed on its output side): dS_T in, dS0 out, the adjoint
  //    entering each chunk's step saved
  a.S0 = p.dS_T;
  a.S_T = p.dS0;
  a.st_save = p.dS_save;
  a.st_scale = p.dS_scale;
  slot = stage_timer_begin(s, kKernChunkAdjoint);
  e = cudaLaunchKernelEx(&cfg, chunk_state_kernel<3, 3, false, 2>, a, mo);
  stage_timer_end(slot, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_chunk_fwd_save(const ChunkFwdSaveLaunch& p, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.B, p.L, p.Hk) || !make_map(&mk, p.k, p.B, p.L, p.Hk) ||
      !make_map(&mv, p.v, p.B, p.L, p.Hv))
    return cudaErrorInvalidValue;
  ChunkArgs a{};
  a.g = p.g;
  a.beta = p.beta;
  a.S0 = p.S0;
  a.fused = 0;   // rows of one chunk also go through the workspace: the backward reads their factors
  a.wait_budget = wait_budget_cycles();
  a.o = static_cast<__nv_bfloat16*>(p.o);
  a.S_T = p.S_T;
  a.ws = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p.ws) + 1023) & ~uintptr_t(1023));
  a.B = p.B;
  a.L = p.L;
  a.Hk = p.Hk;
  a.Hv = p.Hv;
  a.NC = (p.L + kChunk - 1) / kChunk;
  a.err = p.err;
  a.st_save = p.S_save;
  a.st_scale = p.S_scale;
  a.unit_scale = p.unit_scale;
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(chunk_state_kernel<3, 3, false, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             state_smem(3, 3));
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.B * a.Hv * a.NC;
  int slot = stage_timer_begin(s, kKernChunkPrep);
  chunk_prep_kernel<false><<<(int)std::min<long long>(units, 2ll * num_sms()), kPrepThreads, kPrepSmem, s>>>(mq, mk, mv, a);
  stage_timer_end(slot, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSlices, p.Hv, p.B);
  cfg.blockDim = dim3(kStateThreads, 1, 1);
  cfg.dynamicSmemBytes = state_smem(3, 3);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const CUtensorMap no_map{};
  slot = stage_timer_begin(s, kKernChunkState);
  e = cudaLaunchKernelEx(&cfg, chunk_state_kernel<3, 3, false, 3>, a, no_map);
  stage_timer_end(slot, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gdr

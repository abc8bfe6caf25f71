// Backward of the gated delta rule, token by token on CUDA cores with a float32 state.
//
// Reverse mode through the recurrence of the forward (Kev-4B-LiteRT "r15_kernel_test.py",
// truth_f64; DEG "model.py", delta_rule_reference; the pages train through it but print no
// backward). Per (row, value head), with S_{t-1} the state before token t, e = exp(g_t),
// S_a = e S_{t-1}, kv = S_a^T k^, vm = v - kv, delta = beta vm, S_t = S_a + k^ delta^T and
// o_t = S_t^T q~, the adjoint dS of S_t runs from the last token to the first:
//   dq~ = S_t dO_t;     dS += q~ dO_t^T
//   dk^ = dS delta;     ddelta = dS^T k^;   dbeta = ddelta . vm;   dv = beta ddelta
//   dkv = -beta ddelta; dS_a = dS + k^ dkv^T;  dk^ += S_a dkv;  dg = <S_a, dS_a>
//   dS = e dS_a                                   (the adjoint of S_{t-1})
// and dS0 is the dS left after the first token.
//
// The states S_{t-1} are recomputed, not kept by the forward: a first pass stores the state at
// the start of every 32-token segment (a checkpoint); then each segment, last first, runs forward
// again from its checkpoint keeping its 32 states, and then in reverse. Both stores are private to
// the thread that reads them back, so they need no synchronisation.
//
// A CTA owns 16 value columns (one of 8 column blocks) of one (row, value head): thread t holds
// key rows (t/8) + 16m, m = 0..7, and columns 2(t%8), 2(t%8) + 1 of both S and dS. Eight chains
// per head (two CTAs on most SMs) hide more of each token's latency than four wider ones. The
// per-column results (dv, dS0) are the CTA's own. The per-key-row ones (dq~, dk^) and the sums
// over columns (dbeta, dg) are partial over the CTA's columns: they go to the workspace, and a
// second kernel sums them over the 8 column blocks and the value heads of each key head in a
// fixed order (the result does not depend on scheduling), then takes dq~ and dk^ back through the
// normalisations, dx = s dx^ - s^3 (x . dx^) x with s = (|x|^2 + 1e-6)^-1/2 (and D^-1/2 for q).
#include <cuda_bf16.h>

#include "gdr_backward.h"
#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kNcb = kBwdColBlocks;       // CTAs per (row, value head)
constexpr int kCols = kD / kNcb;          // value columns per CTA
constexpr int kCpt = kCols / 8;           // value columns per thread
constexpr int kThreads = 128;
constexpr int kSlice = kD * kCols;        // floats of one CTA's state slice
constexpr float kScale = 0.08838834764831845f;   // 128^-0.5
static_assert(kCpt == 2 || kCpt == 4, "a thread holds 2 or 4 adjacent value columns");

__device__ __forceinline__ float ld_in(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_in(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// kCpt adjacent floats as one vector access (p aligned to kCpt floats)
__device__ __forceinline__ void ld_vec(const float* p, float (&x)[kCpt]) {
  if constexpr (kCpt == 4) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
  } else {
    const float2 u = *reinterpret_cast<const float2*>(p);
    x[0] = u.x; x[1] = u.y;
  }
}
__device__ __forceinline__ void st_vec(float* p, const float (&x)[kCpt]) {
  if constexpr (kCpt == 4)
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
}

// Workspace carve-up (floats): checkpoints [cta][segment][slice], segment states
// [cta][kBwdSeg][slice], then the partials dq~, dk^ [B L Hv][kNcb][kD] and dg, dbeta
// [B L Hv][kNcb]. A slice is stored as [m][thread][kCpt], so thread t's m-th vector of slot s
// starts at float ((s * 8 + m) * kThreads + t) * kCpt.
struct Workspace {
  float* ckpt;
  float* tok;
  float* pq;
  float* pk;
  float* pg;
  float* pb;
};

Workspace carve(void* ws, int B, int L, int Hv) {
  const size_t nCta = (size_t)kNcb * B * Hv;
  const size_t nSeg = ((size_t)L + kBwdSeg - 1) / kBwdSeg;
  const size_t tokens = (size_t)B * L * Hv;
  float* p = static_cast<float*>(ws);
  Workspace w;
  w.ckpt = p; p += nCta * nSeg * kSlice;
  w.tok = p;  p += nCta * kBwdSeg * kSlice;
  w.pq = p;   p += tokens * kNcb * kD;
  w.pk = p;   p += tokens * kNcb * kD;
  w.pg = p;   p += tokens * kNcb;
  w.pb = p;
  return w;
}

// One segment's inputs are staged here by a cooperative load (one memory latency per segment
// instead of one per token), and normalised there once (a warp per token), so the token steps
// read q~, k^ and e ready-made.
struct BwdSmem {
  float qt[kBwdSeg][kD];        // raw q, then q~
  float kh[kBwdSeg][kD];        // raw k, then k^
  float vseg[kBwdSeg][kCols];   // v (this CTA's columns)
  float dOseg[kBwdSeg][kCols];  // dO (this CTA's columns)
  float vm[kBwdSeg][kCols];     // v - kv
  float gseg[kBwdSeg], bseg[kBwdSeg], es[kBwdSeg];
  float red[2][4][8][kCpt];     // per-warp column partials of S^T k^
  float cred[2][4][8][kCpt];    // per-warp column partials of dS^T k^
  float gred[2][4];             // per-warp partials of <S_{t-1}, dS_a>
};
static_assert(sizeof(BwdSmem) <= 48 * 1024, "static shared memory limit");


template <typename T>
__global__ void __launch_bounds__(kThreads) backward_kernel(BackwardArgs a, Workspace w) {
  __shared__ BwdSmem sm;
  const int cb = blockIdx.x % kNcb;
  const int b = blockIdx.x / kNcb;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int cg = tid & 7, rg = tid >> 3;
  const int warp = tid >> 5, lane = tid & 31;
  const int hk = h / (a.Hv / a.Hk);
  const int L = a.L;
  const int nSeg = (L + kBwdSeg - 1) / kBwdSeg;
  const size_t cta = ((size_t)b * a.Hv + h) * kNcb + cb;
  float* ck = w.ckpt + cta * nSeg * kSlice;
  float* tk = w.tok + cta * kBwdSeg * kSlice;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* dO = static_cast<const T*>(a.dO);
  const size_t row_tok = (size_t)b * L;
  const int col0 = cb * kCols + kCpt * cg;
  const size_t state_off = ((size_t)b * a.Hv + h) * kD * kD;
  // thread-private vector m of slot s in a checkpoint or segment-state array
  auto slot = [&](float* base, int s, int m) { return base + ((size_t)(s * 8 + m) * kThreads + tid) * kCpt; };

  float S[8][kCpt];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    if (a.S0) {
      ld_vec(a.S0 + state_off + (size_t)(rg + 16 * m) * kD + col0, S[m]);
    } else {
#pragma unroll
      for (int c = 0; c < kCpt; ++c) S[m][c] = 0.f;
    }
  }

  // Stages tokens [t0, t0 + n) of this CTA's inputs (dO too with with_dO) in shared memory.
  auto load_segment = [&](int t0, int n, bool with_dO) {
#pragma unroll 8
    for (int i = 0; i < n; ++i) {
      const size_t qk_off = ((row_tok + t0 + i) * a.Hk + hk) * kD + tid;
      sm.qt[i][tid] = ld_in(q + qk_off);
      sm.kh[i][tid] = ld_in(k + qk_off);
    }
    for (int j = tid; j < n * kCols; j += kThreads) {
      const int i = j / kCols, c = j % kCols;
      const size_t off = ((row_tok + t0 + i) * a.Hv + h) * kD + cb * kCols + c;
      sm.vseg[i][c] = ld_in(v + off);
      if (with_dO) sm.dOseg[i][c] = ld_in(dO + off);
    }
    if (tid < n) {
      sm.gseg[tid] = __ldg(a.g + (row_tok + t0 + tid) * a.Hv + h);
      sm.bseg[tid] = __ldg(a.beta + (row_tok + t0 + tid) * a.Hv + h);
    }
    __syncthreads();
    // q~ = q (|q|^2 + 1e-6)^-1/2 D^-1/2, k^ = k (|k|^2 + 1e-6)^-1/2, e = exp(g): warp w takes
    // tokens w, w + 4, ..., each lane four elements
    for (int i = warp; i < n; i += 4) {
      float x[4], y[4], sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[j] = sm.qt[i][lane + 32 * j];
        y[j] = sm.kh[i][lane + 32 * j];
        sq = fmaf(x[j], x[j], sq);
        sk = fmaf(y[j], y[j], sk);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
      }
      const float qs = rsqrtf(sq + 1e-6f) * kScale, kinv = rsqrtf(sk + 1e-6f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sm.qt[i][lane + 32 * j] = x[j] * qs;
        sm.kh[i][lane + 32 * j] = y[j] * kinv;
      }
      if (lane == 0) sm.es[i] = expf(sm.gseg[i]);
    }
    __syncthreads();
  };

  // One forward token of the staged segment, S_{t-1} -> S_t (one barrier). With rec, keeps
  // S_{t-1} (thread-private, workspace) and v - kv (shared memory) for the reverse in slot i.
  auto forward_token = [&](int i, int buf, bool rec) {
    float pk[kCpt];
#pragma unroll
    for (int c = 0; c < kCpt; ++c) pk[c] = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float kk = sm.kh[i][rg + 16 * m];
#pragma unroll
      for (int c = 0; c < kCpt; ++c) pk[c] = fmaf(S[m][c], kk, pk[c]);
    }
#pragma unroll
    for (int c = 0; c < kCpt; ++c) {
      pk[c] += __shfl_xor_sync(0xffffffffu, pk[c], 8);
      pk[c] += __shfl_xor_sync(0xffffffffu, pk[c], 16);
    }
    if (lane < 8) {
#pragma unroll
      for (int c = 0; c < kCpt; ++c) sm.red[buf][warp][lane][c] = pk[c];
    }
    __syncthreads();

    const float e = sm.es[i], bt = sm.bseg[i];
    float delta[kCpt];
#pragma unroll
    for (int c = 0; c < kCpt; ++c) {
      const float fk = sm.red[buf][0][cg][c] + sm.red[buf][1][cg][c] + sm.red[buf][2][cg][c] + sm.red[buf][3][cg][c];
      const float vmc = sm.vseg[i][kCpt * cg + c] - e * fk;
      delta[c] = bt * vmc;
      if (rec && rg == 0) sm.vm[i][kCpt * cg + c] = vmc;
    }
    if (rec) {
#pragma unroll
      for (int m = 0; m < 8; ++m) st_vec(slot(tk, i, m), S[m]);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float kk = sm.kh[i][rg + 16 * m];
#pragma unroll
      for (int c = 0; c < kCpt; ++c) S[m][c] = fmaf(e, S[m][c], kk * delta[c]);
    }
  };

  // Pass 1: checkpoints at every segment start (the last segment's tokens are not needed).
  for (int seg = 0; seg < nSeg; ++seg) {
#pragma unroll
    for (int m = 0; m < 8; ++m) st_vec(slot(ck, seg, m), S[m]);
    if (seg == nSeg - 1) break;
    __syncthreads();    // the previous segment is done with the staged inputs
    load_segment(seg * kBwdSeg, kBwdSeg, false);
    for (int i = 0; i < kBwdSeg; ++i) forward_token(i, i & 1, false);
  }

  float dS[8][kCpt];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    if (a.dS_T) {
      ld_vec(a.dS_T + state_off + (size_t)(rg + 16 * m) * kD + col0, dS[m]);
    } else {
#pragma unroll
      for (int c = 0; c < kCpt; ++c) dS[m][c] = 0.f;
    }
  }

  // dg of a token is written by thread 0 once the next barrier has passed (pending until then).
  bool pend = false;
  size_t pend_tv = 0;
  int pend_buf = 0;
  float pend_e = 0.f;
  auto flush_dg = [&]() {
    if (pend && tid == 0)
      w.pg[pend_tv * kNcb + cb] = pend_e * (sm.gred[pend_buf][0] + sm.gred[pend_buf][1] + sm.gred[pend_buf][2] + sm.gred[pend_buf][3]);
    pend = false;
  };

  // One reverse token: dS (adjoint of S_t) -> adjoint of S_{t-1}, from slot i.
  // Sp holds S_{t-1} of the token being reversed; the next one's is fetched while it runs.
  float Sp[8][kCpt];
  auto backward_token = [&](int t, int buf, int i) {
    const size_t tv = (row_tok + t) * a.Hv + h;
    float nxt[8][kCpt];
    if (i > 0) {
#pragma unroll
      for (int m = 0; m < 8; ++m) ld_vec(slot(tk, i - 1, m), nxt[m]);
    }
    const float e = sm.es[i], bt = sm.bseg[i];
    float dOc[kCpt], vmc[kCpt], dl[kCpt], dcol[kCpt];
#pragma unroll
    for (int c = 0; c < kCpt; ++c) {
      dOc[c] = sm.dOseg[i][kCpt * cg + c];
      vmc[c] = sm.vm[i][kCpt * cg + c];
      dl[c] = bt * vmc[c];
      dcol[c] = 0.f;
    }
    float dqr[8], dkr[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float qr = sm.qt[i][rg + 16 * m], kr = sm.kh[i][rg + 16 * m];
      float aq = 0.f, ak = 0.f;
#pragma unroll
      for (int c = 0; c < kCpt; ++c) {
        const float st = fmaf(e, Sp[m][c], kr * dl[c]);     // S_t, as the forward formed it
        aq = fmaf(st, dOc[c], aq);
        dS[m][c] = fmaf(qr, dOc[c], dS[m][c]);
        ak = fmaf(dS[m][c], dl[c], ak);
        dcol[c] = fmaf(dS[m][c], kr, dcol[c]);
      }
      dqr[m] = aq;
      dkr[m] = ak;
    }
#pragma unroll
    for (int c = 0; c < kCpt; ++c) {
      dcol[c] += __shfl_xor_sync(0xffffffffu, dcol[c], 8);
      dcol[c] += __shfl_xor_sync(0xffffffffu, dcol[c], 16);
    }
    if (lane < 8) {
#pragma unroll
      for (int c = 0; c < kCpt; ++c) sm.cred[buf][warp][lane][c] = dcol[c];
    }
    __syncthreads();
    flush_dg();

    float ddl[kCpt], dkv[kCpt], dvv[kCpt];
    float xb = 0.f;
#pragma unroll
    for (int c = 0; c < kCpt; ++c) {
      ddl[c] = sm.cred[buf][0][cg][c] + sm.cred[buf][1][cg][c] + sm.cred[buf][2][cg][c] + sm.cred[buf][3][cg][c];
      dkv[c] = -bt * ddl[c];
      dvv[c] = bt * ddl[c];
      xb = fmaf(ddl[c], vmc[c], xb);
    }
    // dbeta: lanes 0..7 of warp 0 hold the 8 column groups
    xb += __shfl_xor_sync(0xffffffffu, xb, 1);
    xb += __shfl_xor_sync(0xffffffffu, xb, 2);
    xb += __shfl_xor_sync(0xffffffffu, xb, 4);
    if (tid == 0) w.pb[tv * kNcb + cb] = xb;
    if (rg == 0) st_vec(a.dv + tv * kD + col0, dvv);

    float gp[2] = {0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float kr = sm.kh[i][rg + 16 * m];
      float a2 = 0.f;
#pragma unroll
      for (int c = 0; c < kCpt; ++c) {
        a2 = fmaf(Sp[m][c], dkv[c], a2);
        dS[m][c] = fmaf(kr, dkv[c], dS[m][c]);               // dS_a
        gp[m & 1] = fmaf(Sp[m][c], dS[m][c], gp[m & 1]);
        dS[m][c] *= e;
      }
      dkr[m] = fmaf(e, a2, dkr[m]);
    }
    // Row sums over the 8 lanes of a column group by recursive halving (xor 4, 2, 1; 14 shuffles
    // instead of 48): values 0..7 are the dq~ rows rg + 16m, 8..15 the dk^ rows, and lane cg ends
    // with the sums of values b and b + 1, b = 8 (cg >> 2 & 1) + 4 (cg >> 1 & 1) + 2 (cg & 1).
    float r16[16];
#pragma unroll
    for (int m = 0; m < 8; ++m) { r16[m] = dqr[m]; r16[8 + m] = dkr[m]; }
#pragma unroll
    for (int half = 8, bit = 4; half >= 2; half >>= 1, bit >>= 1) {
      const bool up = (cg & bit) != 0;
#pragma unroll
      for (int j = 0; j < half; ++j) {
        const float send = up ? r16[j] : r16[j + half];
        const float keep = up ? r16[j + half] : r16[j];
        r16[j] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
      }
    }
    {
      const int b0 = 8 * ((cg >> 2) & 1) + 4 * ((cg >> 1) & 1) + 2 * (cg & 1);
      float* dst = (b0 < 8 ? w.pq : w.pk) + (tv * kNcb + cb) * kD;
      const int m0 = b0 & 7;
      dst[rg + 16 * m0] = r16[0];
      dst[rg + 16 * (m0 + 1)] = r16[1];
    }
    float g2 = gp[0] + gp[1];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) g2 += __shfl_xor_sync(0xffffffffu, g2, off);
    if (lane == 0) sm.gred[buf][warp] = g2;
    pend = true;
    pend_tv = tv;
    pend_buf = buf;
    pend_e = e;
    if (i > 0) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
#pragma unroll
        for (int c = 0; c < kCpt; ++c) Sp[m][c] = nxt[m][c];
      }
    }
  };

  // Pass 2: segments last to first, each recomputed forward, then reversed.
  for (int seg = nSeg - 1; seg >= 0; --seg) {
    const int t0 = seg * kBwdSeg;
    const int n = min(kBwdSeg, L - t0);
#pragma unroll
    for (int m = 0; m < 8; ++m) ld_vec(slot(ck, seg, m), S[m]);
    __syncthreads();    // the previous segment's reverse is done with the shared arrays
    load_segment(t0, n, true);
    for (int i = 0; i < n; ++i) forward_token(i, i & 1, true);
    __syncthreads();    // the segment's records are complete
#pragma unroll
    for (int m = 0; m < 8; ++m) ld_vec(slot(tk, n - 1, m), Sp[m]);
    for (int i = n - 1; i >= 0; --i) backward_token(t0 + i, i & 1, i);
    __syncthreads();
    flush_dg();
  }

  if (a.dS0) {
#pragma unroll
    for (int m = 0; m < 8; ++m) st_vec(a.dS0 + state_off + (size_t)(rg + 16 * m) * kD + col0, dS[m]);
  }
}

// One (row, token, key head) per CTA, one key row per thread: sums the partials over the value
// heads of the key head and the column blocks, then applies the normalisations' backward.
template <typename T>
__global__ void __launch_bounds__(kD) backward_reduce_kernel(BackwardArgs a, Workspace w) {
  __shared__ float red[4][4];
  const size_t bt = blockIdx.x;          // b L + t
  const int hk = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = a.Hv / a.Hk;
  float dqt = 0.f, dkh = 0.f;
  for (int j = 0; j < r; ++j) {
    const size_t base = (bt * a.Hv + (size_t)hk * r + j) * kNcb * kD + tid;
#pragma unroll
    for (int c = 0; c < kNcb; ++c) { dqt += w.pq[base + c * kD]; dkh += w.pk[base + c * kD]; }
  }
  const size_t off = (bt * a.Hk + hk) * kD + tid;
  const float qv = ld_in(static_cast<const T*>(a.q) + off), kv = ld_in(static_cast<const T*>(a.k) + off);
  float s[4] = {qv * qv, qv * dqt, kv * kv, kv * dkh};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s[j] += __shfl_xor_sync(0xffffffffu, s[j], o);
    if (lane == 0) red[warp][j] = s[j];
  }
  __syncthreads();
  float tot[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) tot[j] = red[0][j] + red[1][j] + red[2][j] + red[3][j];
  const float sq = rsqrtf(tot[0] + 1e-6f), sk = rsqrtf(tot[2] + 1e-6f);
  a.dq[off] = kScale * (sq * dqt - sq * sq * sq * tot[1] * qv);
  a.dk[off] = sk * dkh - sk * sk * sk * tot[3] * kv;
  for (int j = tid; j < r; j += kD) {
    const size_t tv = bt * a.Hv + (size_t)hk * r + j;
    float sg = 0.f, sb = 0.f;
#pragma unroll
    for (int c = 0; c < kNcb; ++c) { sg += w.pg[tv * kNcb + c]; sb += w.pb[tv * kNcb + c]; }
    a.dg[tv] = sg;
    a.dbeta[tv] = sb;
  }
}

}  // namespace

size_t backward_workspace_bytes(int B, int L, int Hk, int Hv) {
  (void)Hk;
  const size_t nCta = (size_t)kNcb * B * Hv;
  const size_t nSeg = ((size_t)L + kBwdSeg - 1) / kBwdSeg;
  const size_t tokens = (size_t)B * L * Hv;
  return sizeof(float) * (nCta * (nSeg + kBwdSeg) * kSlice + tokens * kNcb * (2 * kD + 2));
}

cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s) {
  const Workspace w = carve(a.ws, a.B, a.L, a.Hv);
  const dim3 grid((unsigned)(kNcb * a.B), (unsigned)a.Hv);
  int slot = stage_timer_begin(s, kKernBackward);
  if (a.bf16)
    backward_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a, w);
  else
    backward_kernel<float><<<grid, kThreads, 0, s>>>(a, w);
  stage_timer_end(slot, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid2((unsigned)((size_t)a.B * a.L), (unsigned)a.Hk);
  slot = stage_timer_begin(s, kKernBackwardReduce);
  if (a.bf16)
    backward_reduce_kernel<__nv_bfloat16><<<grid2, kD, 0, s>>>(a, w);
  else
    backward_reduce_kernel<float><<<grid2, kD, 0, s>>>(a, w);
  stage_timer_end(slot, s);
  return cudaGetLastError();
}

}  // namespace gdr

// C ABI of libgdr: host-side argument checks, dispatch to the kernels, the sticky device error
// word, and the stage timer. Every check runs before any CUDA call, so a rejected call never
// touches the GPU.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "gdr.h"
#include "gdr_internal.h"
#include "gdr_backward.h"
#include "gdr_epilogue.h"

namespace gdr {

__device__ int g_error_word;   // first device-side error wins (atomicCAS from 0)

namespace {

thread_local std::string t_msg;

gdr_status fail(gdr_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_msg = buf;
  return st;
}

gdr_status ok() {
  t_msg.clear();
  return GDR_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::mutex g_err_mu;
// device address of g_error_word per device ordinal, with the context it was looked up in: a
// symbol's address belongs to the context that loaded the module, so a new context (after
// cudaDeviceReset, say) needs a new lookup
struct SymbolCache {
  void* ctx = nullptr;
  int* ptr = nullptr;
};
SymbolCache g_err_cache[128];

constexpr long long kDefaultWaitBudget = 2000000000ll;   // cycles, about 1 s
std::atomic<long long> g_wait_budget{kDefaultWaitBudget};

// Stage timer: one (start, end) event pair per recorded launch.
struct StageTimer {
  std::mutex mu;
  bool on = false;
  int cap = 0;
  int used = 0;
  std::vector<cudaEvent_t> ev;
  std::vector<int> id;
} g_timer;

}  // namespace

int stage_timer_begin(cudaStream_t s, int kid) {
  std::lock_guard<std::mutex> lk(g_timer.mu);
  if (!g_timer.on || g_timer.used >= g_timer.cap) return -1;
  const int slot = g_timer.used++;
  g_timer.id[slot] = kid;
  cudaEventRecord(g_timer.ev[2 * slot], s);
  return slot;
}

void stage_timer_end(int slot, cudaStream_t s) {
  if (slot < 0) return;
  cudaEventRecord(g_timer.ev[2 * slot + 1], s);
}

namespace {

// Checks shared by every entry point.
gdr_status check_common(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const void* o, int B, int L, int Hk, int Hv, int D,
                        gdr_dtype dt, const char* who) {
  if (!q || !k || !v || !g || !beta || !o)
    return fail(GDR_ERR_INVALID_ARG, "%s: q, k, v, g, beta and o must be non-NULL", who);
  if (B < 1 || L < 1 || Hk < 1 || Hv < 1)
    return fail(GDR_ERR_INVALID_ARG, "%s: sizes must be >= 1 (B=%d L=%d Hk=%d Hv=%d)", who, B, L, Hk, Hv);
  if (Hv % Hk != 0)
    return fail(GDR_ERR_INVALID_ARG, "%s: Hv=%d is not a multiple of Hk=%d", who, Hv, Hk);
  if (dt != GDR_F32 && dt != GDR_BF16)
    return fail(GDR_ERR_INVALID_ARG, "%s: unknown dtype %d", who, (int)dt);
  if (D != kD)
    return fail(GDR_ERR_UNSUPPORTED, "%s: head dimension D=%d is not implemented (only 128)", who, D);
  if ((long long)Hv > 65535)
    return fail(GDR_ERR_UNSUPPORTED, "%s: Hv=%d exceeds 65535", who, Hv);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(g) || !aligned16(beta))
    return fail(GDR_ERR_INVALID_ARG, "%s: q, k, v, o, g and beta must be 16-byte aligned", who);
  return GDR_OK;
}

gdr_status launch_status(cudaError_t e, const char* who) {
  if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
  return ok();
}

}  // namespace

long long wait_budget_cycles() { return g_wait_budget.load(); }

int record_error(int status, const char* message) {
  t_msg = message;
  return status;
}

void* current_context() {
  using CtxGetCurrent = int (*)(void**);   // CUresult cuCtxGetCurrent(CUcontext*)
  static CtxGetCurrent fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuCtxGetCurrent", &p, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetCurrent>(p);
  }();
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  void* ctx = current_context();   // NULL before the runtime has made a context current
  std::lock_guard<std::mutex> lk(g_err_mu);
  SymbolCache& c = g_err_cache[dev];
  if (!c.ptr || !ctx || c.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    c.ptr = static_cast<int*>(p);
    c.ctx = current_context();     // the lookup has made the device's primary context current
  }
  return c.ptr;
}

}  // namespace gdr

using namespace gdr;

extern "C" {

size_t gdr_chunk_workspace_bytes(int B, int L, int Hk, int Hv, int D, gdr_dtype dt) {
  if (B < 1 || L < 1 || Hk < 1 || Hv < 1 || D != kD || Hv % Hk != 0) return 0;
  if (dt != GDR_BF16) return 0;   // the float32 path keeps everything in registers
  return chunk_workspace_bytes(B, Hk, L, Hv);
}

}  // extern "C"

namespace {

// gdr_chunk_fwd and gdr_chunk_fwd_varlen (lengths NULL = every row has L tokens)
gdr_status chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                     const float* S0, const int32_t* lengths, void* o, float* S_T, int B, int L, int Hk, int Hv,
                     int D, gdr_dtype dt, void* ws, size_t ws_bytes, gdr_stream_t stream, const char* who,
                     const void* z = nullptr, const float* w = nullptr, float eps = 0.f) {
  gdr_status st = check_common(q, k, v, g, beta, o, B, L, Hk, Hv, D, dt, who);
  if (st != GDR_OK) return st;
  if ((S0 && !aligned16(S0)) || (S_T && !aligned16(S_T)))
    return fail(GDR_ERR_INVALID_ARG, "%s: S0 and S_T must be 16-byte aligned", who);
  if (lengths && (reinterpret_cast<uintptr_t>(lengths) & 3u))
    return fail(GDR_ERR_INVALID_ARG, "%s: lengths must be 4-byte aligned", who);
  const size_t need = gdr_chunk_workspace_bytes(B, L, Hk, Hv, D, dt);
  if (need > 0 && (ws == nullptr || ws_bytes < need))
    return fail(GDR_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", who, need,
                ws == nullptr ? (size_t)0 : ws_bytes);
  int* err = device_error_word();
  if (!err) return fail(GDR_ERR_CUDA, "%s: no CUDA device available", who);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (dt == GDR_BF16) {
    if (B > 65535 || Hk > 65535)
      return fail(GDR_ERR_UNSUPPORTED, "%s: B=%d or Hk=%d exceeds 65535", who, B, Hk);
    ChunkLaunch c{q, k, v, g, beta, S0, o, S_T, ws, B, L, Hk, Hv, err};
    c.lengths = lengths;
    c.z = z;
    c.w = w;
    c.eps = eps;
    return launch_status(launch_chunk_bf16(c, s), who);
  }
  RecurrentArgs a{q, k, v, g, beta, S0, nullptr, B, o, S_T, B, L, Hk, Hv, false, err};
  a.lengths = lengths;
  const int slot = stage_timer_begin(s, kKernRecurrent);
  cudaError_t e = launch_recurrent(a, s);
  stage_timer_end(slot, s);
  return launch_status(e, who);
}

}  // namespace

extern "C" {

gdr_status gdr_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* S0, void* o, float* S_T, int B, int L,
                         int Hk, int Hv, int D, gdr_dtype dt, void* ws, size_t ws_bytes,
                         gdr_stream_t stream) {
  return chunk_fwd(q, k, v, g, beta, S0, nullptr, o, S_T, B, L, Hk, Hv, D, dt, ws, ws_bytes, stream,
                   "gdr_chunk_fwd");
}

gdr_status gdr_chunk_fwd_gated(const void* q, const void* k, const void* v, const float* g,
                               const float* beta, const float* S0, const void* z, const float* w, float eps,
                               void* out, float* S_T, int B, int L, int Hk, int Hv, int D, gdr_dtype dt, void* ws,
                               size_t ws_bytes, gdr_stream_t stream) {
  const char* who = "gdr_chunk_fwd_gated";
  if (!z || !w) return fail(GDR_ERR_INVALID_ARG, "%s: z and w must be non-NULL", who);
  if (dt != GDR_BF16) return fail(GDR_ERR_UNSUPPORTED, "%s: the gated epilogue takes bfloat16 q, k, v, z (dt=%d)", who, (int)dt);
  if (!(eps >= 0.f)) return fail(GDR_ERR_INVALID_ARG, "%s: eps must be >= 0", who);
  if (!aligned16(z) || !aligned16(w)) return fail(GDR_ERR_INVALID_ARG, "%s: z and w must be 16-byte aligned", who);
  if (out) {
    // out is written while z is read: they must not overlap
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), z0 = reinterpret_cast<uintptr_t>(z);
    const uintptr_t n = (uintptr_t)B * L * Hv * kD * 2;
    if (o0 < z0 + n && z0 < o0 + n) return fail(GDR_ERR_INVALID_ARG, "%s: out overlaps z", who);
  }
  return chunk_fwd(q, k, v, g, beta, S0, nullptr, out, S_T, B, L, Hk, Hv, D, dt, ws, ws_bytes, stream, who, z, w, eps);
}

gdr_status gdr_chunk_fwd_varlen(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* S0, const int32_t* lengths, void* o,
                                float* S_T, int B, int L, int Hk, int Hv, int D, gdr_dtype dt, void* ws,
                                size_t ws_bytes, gdr_stream_t stream) {
  if (!lengths) return fail(GDR_ERR_INVALID_ARG, "gdr_chunk_fwd_varlen: lengths must be non-NULL");
  return chunk_fwd(q, k, v, g, beta, S0, lengths, o, S_T, B, L, Hk, Hv, D, dt, ws, ws_bytes, stream,
                   "gdr_chunk_fwd_varlen");
}

size_t gdr_chunk_fwd_prologue_workspace_bytes(int B, int L, int Hk, int Hv, int D, int K) {
  if (B < 1 || L < 1 || Hk < 1 || Hv < 1 || D != kD || Hv % Hk != 0 || K != 4) return 0;
  return chunk_prologue_workspace_bytes(B, L, Hv);
}

gdr_status gdr_chunk_fwd_prologue(const void* mixed, const void* tail, const float* conv_w, const float* a,
                                  const float* b, const float* A_log, const float* dt_bias, const float* S0,
                                  void* o, float* S_T, void* new_tail, int B, int L, int Hk, int Hv, int D,
                                  int K, void* ws, size_t ws_bytes, gdr_stream_t stream) {
  const char* who = "gdr_chunk_fwd_prologue";
  if (!mixed || !conv_w || !a || !b || !A_log || !dt_bias || !o)
    return fail(GDR_ERR_INVALID_ARG, "%s: mixed, conv_w, a, b, A_log, dt_bias and o must be non-NULL", who);
  if (B < 1 || L < 1 || Hk < 1 || Hv < 1)
    return fail(GDR_ERR_INVALID_ARG, "%s: sizes must be >= 1 (B=%d L=%d Hk=%d Hv=%d)", who, B, L, Hk, Hv);
  if (Hv % Hk != 0) return fail(GDR_ERR_INVALID_ARG, "%s: Hv=%d is not a multiple of Hk=%d", who, Hv, Hk);
  if (K < 1 || K > 8) return fail(GDR_ERR_INVALID_ARG, "%s: conv width K=%d is outside [1, 8]", who, K);
  if (K != 4) return fail(GDR_ERR_UNSUPPORTED, "%s: the fused prologue takes a 4-tap conv (K=%d)", who, K);
  if (D != kD) return fail(GDR_ERR_UNSUPPORTED, "%s: head dimension D=%d is not implemented (only 128)", who, D);
  if (B > 65535 || Hv > 65535)
    return fail(GDR_ERR_UNSUPPORTED, "%s: B=%d or Hv=%d exceeds 65535", who, B, Hv);
  const void* ptrs16[] = {mixed, tail, conv_w, S0, o, S_T, new_tail};
  for (const void* p : ptrs16)
    if (p && !aligned16(p))
      return fail(GDR_ERR_INVALID_ARG, "%s: mixed, tail, conv_w, S0, o, S_T and new_tail must be 16-byte aligned", who);
  const void* ptrs4[] = {a, b, A_log, dt_bias};
  for (const void* p : ptrs4)
    if (reinterpret_cast<uintptr_t>(p) & 3u)
      return fail(GDR_ERR_INVALID_ARG, "%s: a, b, A_log and dt_bias must be 4-byte aligned", who);
  // o is written while mixed and tail may still be read (the carry is gathered after the path), and
  // new_tail is gathered from both: half-open byte ranges, checked pairwise
  const uintptr_t C = (uintptr_t)(2 * Hk + Hv) * kD;
  struct Range { const void* p; uintptr_t n; };
  const Range in_mixed{mixed, (uintptr_t)B * L * C * 2}, in_tail{tail, (uintptr_t)B * 3 * C * 2};
  const Range out_o{o, (uintptr_t)B * L * Hv * kD * 2}, out_tail{new_tail, (uintptr_t)B * 3 * C * 2};
  auto overlap = [](const Range& x, const Range& y) {
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(x.p), y0 = reinterpret_cast<uintptr_t>(y.p);
    return x.p && y.p && x0 < y0 + y.n && y0 < x0 + x.n;
  };
  if (overlap(out_o, in_mixed) || overlap(out_o, in_tail) || overlap(out_tail, in_mixed) ||
      overlap(out_tail, in_tail) || overlap(out_tail, out_o))
    return fail(GDR_ERR_INVALID_ARG, "%s: o and new_tail must overlap neither mixed, tail nor each other", who);
  const size_t need = gdr_chunk_fwd_prologue_workspace_bytes(B, L, Hk, Hv, D, K);
  if (ws == nullptr || ws_bytes < need)
    return fail(GDR_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", who, need,
                ws == nullptr ? (size_t)0 : ws_bytes);
  int* err = device_error_word();
  if (!err) return fail(GDR_ERR_CUDA, "%s: no CUDA device available", who);
  ChunkLaunch c{nullptr, nullptr, nullptr, nullptr, nullptr, S0, o, S_T, ws, B, L, Hk, Hv, err};
  c.mixed = mixed;
  c.tail = tail;
  c.conv_w = conv_w;
  c.proj_a = a;
  c.proj_b = b;
  c.A_log = A_log;
  c.dt_bias = dt_bias;
  c.new_tail = new_tail;
  return launch_status(launch_chunk_bf16(c, reinterpret_cast<cudaStream_t>(stream)), who);
}

size_t gdr_fork_workspace_bytes(int F, int L_pad, int Hk, int Hv, int D, gdr_dtype dt) {
  return gdr_chunk_workspace_bytes(F, L_pad, Hk, Hv, D, dt);
}

gdr_status gdr_fork_fwd(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const float* trunk, const int64_t* trunk_idx, int N,
                        void* o, float* states_out, int F, int L_pad, int Hk, int Hv, int D,
                        gdr_dtype dt, void* ws, size_t ws_bytes, gdr_stream_t stream) {
  const char* who = "gdr_fork_fwd";
  gdr_status st = check_common(q, k, v, g, beta, o, F, L_pad, Hk, Hv, D, dt, who);
  if (st != GDR_OK) return st;
  if (!trunk || !trunk_idx || N < 1)
    return fail(GDR_ERR_INVALID_ARG, "%s: trunk and trunk_idx must be non-NULL and N >= 1", who);
  if (!aligned16(trunk) || (states_out && !aligned16(states_out)) || (reinterpret_cast<uintptr_t>(trunk_idx) & 7u))
    return fail(GDR_ERR_INVALID_ARG, "%s: trunk/states_out must be 16-byte and trunk_idx 8-byte aligned", who);
  if (states_out) {
    const size_t per = (size_t)Hv * kD * kD * sizeof(float);
    const char* t0 = reinterpret_cast<const char*>(trunk);
    const char* t1 = t0 + (size_t)N * per;
    const char* s0 = reinterpret_cast<const char*>(states_out);
    const char* s1 = s0 + (size_t)F * per;
    if (s0 < t1 && t0 < s1)
      return fail(GDR_ERR_INVALID_ARG, "%s: states_out overlaps trunk", who);
  }
  const size_t need = gdr_fork_workspace_bytes(F, L_pad, Hk, Hv, D, dt);
  if (need > 0 && (ws == nullptr || ws_bytes < need))
    return fail(GDR_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", who, need,
                ws == nullptr ? (size_t)0 : ws_bytes);
  int* err = device_error_word();
  if (!err) return fail(GDR_ERR_CUDA, "%s: no CUDA device available", who);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == GDR_BF16) {
    if (F > 65535 || Hk > 65535)
      return fail(GDR_ERR_UNSUPPORTED, "%s: F=%d or Hk=%d exceeds 65535", who, F, Hk);
    ChunkLaunch c{q, k, v, g, beta, trunk, o, states_out, ws, F, L_pad, Hk, Hv, err, trunk_idx, N};
    return launch_status(launch_chunk_bf16(c, s), who);
  }
  RecurrentArgs a{q, k, v, g, beta, trunk, trunk_idx, N, o, states_out, F, L_pad, Hk, Hv, false, err};
  const int slot = stage_timer_begin(s, kKernRecurrent);
  cudaError_t e = launch_recurrent(a, s);
  stage_timer_end(slot, s);
  return launch_status(e, who);
}

gdr_status gdr_decode_step(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float* states, void* o, int F, int Hk, int Hv,
                           int D, gdr_dtype dt, gdr_stream_t stream) {
  const char* who = "gdr_decode_step";
  gdr_status st = check_common(q, k, v, g, beta, o, F, 1, Hk, Hv, D, dt, who);
  if (st != GDR_OK) return st;
  if (!states || !aligned16(states))
    return fail(GDR_ERR_INVALID_ARG, "%s: states must be non-NULL and 16-byte aligned", who);
  int* err = device_error_word();
  if (!err) return fail(GDR_ERR_CUDA, "%s: no CUDA device available", who);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  RecurrentArgs a{q, k, v, g, beta, states, nullptr, F, o, states, F, 1, Hk, Hv, dt == GDR_BF16, err};
  const int slot = stage_timer_begin(s, kKernRecurrent);
  cudaError_t e = launch_recurrent(a, s);
  stage_timer_end(slot, s);
  return launch_status(e, who);
}

gdr_status gdr_prologue(const void* mixed, const void* tail, const float* conv_w, const float* a,
                        const float* b, const float* A_log, const float* dt_bias, const int32_t* lengths,
                        void* q, void* k, void* v, float* g, float* beta, void* new_tail, int B, int L,
                        int Hk, int Hv, int D, int K, gdr_stream_t stream) {
  const char* who = "gdr_prologue";
  if (!mixed || !conv_w || !a || !b || !A_log || !dt_bias || !q || !k || !v || !g || !beta)
    return fail(GDR_ERR_INVALID_ARG, "%s: mixed, conv_w, a, b, A_log, dt_bias, q, k, v, g and beta must be non-NULL", who);
  if (B < 1 || L < 1 || Hk < 1 || Hv < 1)
    return fail(GDR_ERR_INVALID_ARG, "%s: sizes must be >= 1 (B=%d L=%d Hk=%d Hv=%d)", who, B, L, Hk, Hv);
  if (Hv % Hk != 0) return fail(GDR_ERR_INVALID_ARG, "%s: Hv=%d is not a multiple of Hk=%d", who, Hv, Hk);
  if (K < 1 || K > 8) return fail(GDR_ERR_INVALID_ARG, "%s: conv width K=%d is outside [1, 8]", who, K);
  if (D != kD) return fail(GDR_ERR_UNSUPPORTED, "%s: head dimension D=%d is not implemented (only 128)", who, D);
  // launch limits: rows are the grid's z dimension, tiles of 16 positions its y dimension
  if ((long long)B > 65535 || (long long)L > 16LL * 65535)
    return fail(GDR_ERR_UNSUPPORTED, "%s: B=%d or L=%d too large (B <= 65535, L <= 1048560)", who, B, L);
  const void* ptrs16[] = {mixed, q, k, v, tail, new_tail};
  for (const void* p : ptrs16)
    if (p && !aligned16(p)) return fail(GDR_ERR_INVALID_ARG, "%s: mixed, tail, q, k, v and new_tail must be 16-byte aligned", who);
  if (!aligned16(conv_w)) return fail(GDR_ERR_INVALID_ARG, "%s: conv_w must be 16-byte aligned", who);
  const void* ptrs4[] = {a, b, A_log, dt_bias, g, beta, lengths};
  for (const void* p : ptrs4)
    if (p && (reinterpret_cast<uintptr_t>(p) & 3u))
      return fail(GDR_ERR_INVALID_ARG, "%s: a, b, A_log, dt_bias, g, beta and lengths must be 4-byte aligned", who);
  const long long C = (2LL * Hk + Hv) * kD;
  if (new_tail && K > 1) {
    // the carry is gathered from tail and mixed: it must not overlap either
    const uintptr_t nt0 = reinterpret_cast<uintptr_t>(new_tail), nt1 = nt0 + (uintptr_t)B * (K - 1) * C * 2;
    auto overlaps = [&](const void* p, uintptr_t bytes) {
      const uintptr_t p0 = reinterpret_cast<uintptr_t>(p);
      return p && p0 < nt1 && nt0 < p0 + bytes;
    };
    if (overlaps(tail, (uintptr_t)B * (K - 1) * C * 2) || overlaps(mixed, (uintptr_t)B * L * C * 2))
      return fail(GDR_ERR_INVALID_ARG, "%s: new_tail must not overlap tail or mixed", who);
  }
  int* err = device_error_word();
  if (!err) return fail(GDR_ERR_CUDA, "%s: no CUDA device available", who);
  PrologueArgs pa{mixed, tail, conv_w, a, b, A_log, dt_bias, lengths, q, k, v, g, beta, new_tail,
                  B, L, Hk, Hv, (int)C, K, err};
  pa.wait_budget = wait_budget_cycles();
  return launch_status(launch_prologue(pa, reinterpret_cast<cudaStream_t>(stream)), who);
}

gdr_status gdr_gated_rmsnorm(const void* x, const void* z, const float* w, float eps, void* out,
                             long long rows, int D, gdr_stream_t stream) {
  const char* who = "gdr_gated_rmsnorm";
  if (!x || !z || !w || !out) return fail(GDR_ERR_INVALID_ARG, "%s: x, z, w and out must be non-NULL", who);
  if (rows < 1) return fail(GDR_ERR_INVALID_ARG, "%s: rows=%lld must be >= 1", who, rows);
  if (D != kD) return fail(GDR_ERR_UNSUPPORTED, "%s: row length D=%d is not implemented (only 128)", who, D);
  if (!(eps >= 0.f)) return fail(GDR_ERR_INVALID_ARG, "%s: eps must be >= 0", who);
  if (rows > ((long long)1 << 34)) return fail(GDR_ERR_UNSUPPORTED, "%s: rows=%lld too large (<= 2^34)", who, rows);
  if (!aligned16(x) || !aligned16(z) || !aligned16(w) || !aligned16(out))
    return fail(GDR_ERR_INVALID_ARG, "%s: x, z, w and out must be 16-byte aligned", who);
  if (out != x && out != z) {
    // out may be x or z exactly (each row is read before it is written) but must not partly overlap
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + (uintptr_t)rows * kD * 2;
    for (const void* p : {x, z}) {
      const uintptr_t p0 = reinterpret_cast<uintptr_t>(p);
      if (p0 < o1 && o0 < p0 + (uintptr_t)rows * kD * 2)
        return fail(GDR_ERR_INVALID_ARG, "%s: out overlaps x or z without being one of them", who);
    }
  }
  EpilogueArgs ea{x, z, w, eps, out, rows};
  return launch_status(launch_gated_rmsnorm(ea, reinterpret_cast<cudaStream_t>(stream)), who);
}

// The backward's outputs (and the workspace) must not overlap one another or any input: half-open
// byte ranges, checked pairwise.
static gdr_status check_backward_buffers(const void* q, const void* k, const void* v, const float* g,
                                         const float* beta, const float* S0, const void* dO, const float* dS_T,
                                         const float* dq, const float* dk, const float* dv, const float* dg,
                                         const float* dbeta, const float* dS0, const void* ws, size_t need, int B,
                                         int L, int Hk, int Hv, size_t es, const char* who) {
  const size_t nq = (size_t)B * L * Hk * kD, nv = (size_t)B * L * Hv * kD, ng = (size_t)B * L * Hv;
  const size_t ns = (size_t)B * Hv * kD * kD;
  struct Range {
    const void* p;
    size_t bytes;
    const char* name;
  };
  const Range outs[] = {{dq, nq * 4, "dq"},       {dk, nq * 4, "dk"},     {dv, nv * 4, "dv"},
                        {dg, ng * 4, "dg"},       {dbeta, ng * 4, "dbeta"}, {dS0, ns * 4, "dS0"},
                        {ws, need, "ws"}};
  const Range ins[] = {{q, nq * es, "q"}, {k, nq * es, "k"},     {v, nv * es, "v"},   {g, ng * 4, "g"},
                       {beta, ng * 4, "beta"}, {S0, ns * 4, "S0"}, {dO, nv * es, "dO"}, {dS_T, ns * 4, "dS_T"}};
  auto overlap = [](const Range& a, const Range& b) {
    if (!a.p || !b.p) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
  };
  const int n_out = sizeof(outs) / sizeof(outs[0]);
  for (int i = 0; i < n_out; ++i) {
    for (int j = i + 1; j < n_out; ++j)
      if (overlap(outs[i], outs[j]))
        return fail(GDR_ERR_INVALID_ARG, "%s: %s overlaps %s", who, outs[i].name, outs[j].name);
    for (const Range& in : ins)
      if (overlap(outs[i], in))
        return fail(GDR_ERR_INVALID_ARG, "%s: %s overlaps the input %s", who, outs[i].name, in.name);
  }
  return GDR_OK;
}

size_t gdr_backward_workspace_bytes(int B, int L, int Hk, int Hv, int D) {
  if (B < 1 || L < 1 || Hk < 1 || Hv < 1 || D != kD || Hv % Hk != 0) return 0;
  return backward_workspace_bytes(B, L, Hk, Hv);
}

gdr_status gdr_backward(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        const float* S0, const void* dO, const float* dS_T, float* dq, float* dk,
                        float* dv, float* dg, float* dbeta, float* dS0, int B, int L, int Hk, int Hv,
                        int D, gdr_dtype dt, void* ws, size_t ws_bytes, gdr_stream_t stream) {
  const char* who = "gdr_backward";
  if (!dO) return fail(GDR_ERR_INVALID_ARG, "%s: dO must be non-NULL", who);
  gdr_status st = check_common(q, k, v, g, beta, dO, B, L, Hk, Hv, D, dt, who);
  if (st != GDR_OK) return st;
  if (!dq || !dk || !dv || !dg || !dbeta)
    return fail(GDR_ERR_INVALID_ARG, "%s: dq, dk, dv, dg and dbeta must be non-NULL", who);
  const void* ptrs16[] = {dq, dk, dv, dg, dbeta, S0, dS_T, dS0, ws};
  for (const void* p : ptrs16)
    if (p && !aligned16(p))
      return fail(GDR_ERR_INVALID_ARG, "%s: every array and the workspace must be 16-byte aligned", who);
  // launch limits: kBwdColBlocks * B column-block CTAs on the grid's x dimension (B <= 65535 keeps
  // that within 2^31 - 1), B L tokens on the reducer's
  if ((long long)B > 65535 || (long long)B * L > 0x7fffffffLL || Hk > 65535)
    return fail(GDR_ERR_UNSUPPORTED, "%s: B=%d, B*L=%lld or Hk=%d too large (B <= 65535, B*L < 2^31)", who, B,
                (long long)B * L, Hk);
  const size_t need = backward_workspace_bytes(B, L, Hk, Hv);
  if (ws == nullptr || ws_bytes < need)
    return fail(GDR_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", who, need,
                ws == nullptr ? (size_t)0 : ws_bytes);
  st = check_backward_buffers(q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, ws, need, B, L, Hk, Hv,
                              dt == GDR_BF16 ? 2 : 4, who);
  if (st != GDR_OK) return st;
  BackwardArgs a{q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, ws, B, L, Hk, Hv, dt == GDR_BF16};
  return launch_status(launch_backward(a, reinterpret_cast<cudaStream_t>(stream)), who);
}

size_t gdr_backward_chunked_workspace_bytes(int B, int L, int Hk, int Hv, int D) {
  if (B < 1 || L < 1 || Hk < 1 || Hv < 1 || D != kD || Hv % Hk != 0) return 0;
  return chunk_bwd_workspace_bytes(B, L, Hk, Hv);
}

}  // extern "C"

// gdr_backward_chunked and gdr_backward_chunked_saved (saved: ws holds what gdr_chunk_fwd_save left)
static gdr_status backward_chunked(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                   const float* S0, const void* dO, const float* dS_T, float* dq, float* dk,
                                   float* dv, float* dg, float* dbeta, float* dS0, int B, int L, int Hk, int Hv,
                                   int D, gdr_dtype dt, void* ws, size_t ws_bytes, gdr_stream_t stream, bool saved,
                                   const char* who) {
  if (!dO) return fail(GDR_ERR_INVALID_ARG, "%s: dO must be non-NULL", who);
  gdr_status st = check_common(q, k, v, g, beta, dO, B, L, Hk, Hv, D, dt, who);
  if (st != GDR_OK) return st;
  if (dt != GDR_BF16) return fail(GDR_ERR_UNSUPPORTED, "%s: bf16 q, k, v, dO only (float32: gdr_backward)", who);
  if (!dq || !dk || !dv || !dg || !dbeta)
    return fail(GDR_ERR_INVALID_ARG, "%s: dq, dk, dv, dg and dbeta must be non-NULL", who);
  const void* ptrs16[] = {dq, dk, dv, dg, dbeta, S0, dS_T, dS0, ws};
  for (const void* p : ptrs16)
    if (p && !aligned16(p))
      return fail(GDR_ERR_INVALID_ARG, "%s: every array and the workspace must be 16-byte aligned", who);
  // launch limits: B Hv NC units on the grid's x dimension, B L positions on the reducer's
  const long long units = (long long)B * Hv * ((L + kChunk - 1) / kChunk);
  if (units > 0x7fffffffLL || (long long)B * L > 0x7fffffffLL || Hk > 65535 || Hv > 65535 || B > 65535)
    return fail(GDR_ERR_UNSUPPORTED, "%s: B=%d, L=%d, Hv=%d too large", who, B, L, Hv);
  const size_t need = chunk_bwd_workspace_bytes(B, L, Hk, Hv);
  if (ws == nullptr || ws_bytes < need)
    return fail(GDR_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", who, need,
                ws == nullptr ? (size_t)0 : ws_bytes);
  st = check_backward_buffers(q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, ws, need, B, L, Hk, Hv, 2,
                              who);
  if (st != GDR_OK) return st;
  int* err = device_error_word();
  if (!err) return fail(GDR_ERR_CUDA, "%s: no device error word", who);
  ChunkBackwardArgs a{q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, ws, B, L, Hk, Hv, err};
  a.saved = saved;
  return launch_status(launch_chunk_backward(a, reinterpret_cast<cudaStream_t>(stream)), who);
}

extern "C" {

gdr_status gdr_backward_chunked(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                const float* S0, const void* dO, const float* dS_T, float* dq, float* dk,
                                float* dv, float* dg, float* dbeta, float* dS0, int B, int L, int Hk, int Hv,
                                int D, gdr_dtype dt, void* ws, size_t ws_bytes, gdr_stream_t stream) {
  return backward_chunked(q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, B, L, Hk, Hv, D, dt, ws,
                          ws_bytes, stream, false, "gdr_backward_chunked");
}

gdr_status gdr_backward_chunked_saved(const void* q, const void* k, const void* v, const float* g,
                                      const float* beta, const float* S0, const void* dO, const float* dS_T,
                                      float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dS0, int B,
                                      int L, int Hk, int Hv, int D, gdr_dtype dt, void* saved, size_t saved_bytes,
                                      gdr_stream_t stream) {
  return backward_chunked(q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, B, L, Hk, Hv, D, dt, saved,
                          saved_bytes, stream, true, "gdr_backward_chunked_saved");
}

gdr_status gdr_chunk_fwd_save(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              const float* S0, void* o, float* S_T, int B, int L, int Hk, int Hv, int D,
                              gdr_dtype dt, void* saved, size_t saved_bytes, gdr_stream_t stream) {
  const char* who = "gdr_chunk_fwd_save";
  gdr_status st = check_common(q, k, v, g, beta, o, B, L, Hk, Hv, D, dt, who);
  if (st != GDR_OK) return st;
  if (dt != GDR_BF16) return fail(GDR_ERR_UNSUPPORTED, "%s: bf16 q, k, v only (the chunked backward's forward)", who);
  if ((S0 && !aligned16(S0)) || (S_T && !aligned16(S_T)) || (saved && !aligned16(saved)))
    return fail(GDR_ERR_INVALID_ARG, "%s: S0, S_T and saved must be 16-byte aligned", who);
  const long long units = (long long)B * Hv * ((L + kChunk - 1) / kChunk);
  if (units > 0x7fffffffLL || Hk > 65535 || Hv > 65535 || B > 65535)
    return fail(GDR_ERR_UNSUPPORTED, "%s: B=%d, L=%d, Hv=%d too large", who, B, L, Hv);
  const size_t need = chunk_bwd_workspace_bytes(B, L, Hk, Hv);
  if (saved == nullptr || saved_bytes < need)
    return fail(GDR_ERR_INVALID_ARG, "%s: saved buffer of %zu bytes needed, %zu given", who, need,
                saved == nullptr ? (size_t)0 : saved_bytes);
  // the saved buffer is written while every input is read and the outputs are written
  const size_t nq = (size_t)B * L * Hk * kD * 2, nv = (size_t)B * L * Hv * kD * 2, ng = (size_t)B * L * Hv * 4;
  const size_t ns = (size_t)B * Hv * kD * kD * 4;
  const struct { const void* p; size_t n; } others[] = {{q, nq}, {k, nq}, {v, nv}, {g, ng}, {beta, ng},
                                                        {S0, ns}, {o, nv}, {S_T, ns}};
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(saved), w1 = w0 + need;
  for (const auto& r : others) {
    const uintptr_t p0 = reinterpret_cast<uintptr_t>(r.p);
    if (r.p && p0 < w1 && w0 < p0 + r.n)
      return fail(GDR_ERR_INVALID_ARG, "%s: saved overlaps an input or an output", who);
  }
  int* err = device_error_word();
  if (!err) return fail(GDR_ERR_CUDA, "%s: no CUDA device available", who);
  return launch_status(launch_chunk_forward_saving(q, k, v, g, beta, S0, o, S_T, saved, B, L, Hk, Hv, err,
                                                   reinterpret_cast<cudaStream_t>(stream)),
                       who);
}

gdr_status gdr_sync_status(gdr_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "gdr_sync_status: %s", cudaGetErrorString(e));
  int* p = device_error_word();
  if (!p) return fail(GDR_ERR_CUDA, "gdr_sync_status: no CUDA device available");
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int));
  if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "gdr_sync_status: %s", cudaGetErrorString(e));
  if (word != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
    if (word == kErrDeviceIndex) return fail(GDR_ERR_DEVICE_INDEX, "a fork's trunk index was out of range");
    if (word == kErrTimeout) return fail(GDR_ERR_TIMEOUT, "a kernel wait ran past its limit");
    return fail(GDR_ERR_CUDA, "device error word %d", word);
  }
  return ok();
}

const char* gdr_status_string(gdr_status s) {
  switch (s) {
    case GDR_OK: return "GDR_OK";
    case GDR_ERR_INVALID_ARG: return "GDR_ERR_INVALID_ARG";
    case GDR_ERR_UNSUPPORTED: return "GDR_ERR_UNSUPPORTED";
    case GDR_ERR_CUDA: return "GDR_ERR_CUDA";
    case GDR_ERR_DEVICE_INDEX: return "GDR_ERR_DEVICE_INDEX";
    case GDR_ERR_TIMEOUT: return "GDR_ERR_TIMEOUT";
  }
  return "GDR_ERR_UNKNOWN";
}

const char* gdr_last_error_message(void) { return t_msg.c_str(); }

gdr_status gdr_debug_set_wait_budget(long long cycles) {
  g_wait_budget.store(cycles > 0 ? cycles : (cycles == 0 ? 0 : kDefaultWaitBudget));
  return ok();
}

gdr_status gdr_stage_timer_enable(int on, int capacity) {
  std::lock_guard<std::mutex> lk(g_timer.mu);
  for (cudaEvent_t e : g_timer.ev) cudaEventDestroy(e);
  g_timer.ev.clear();
  g_timer.id.clear();
  g_timer.used = 0;
  g_timer.cap = 0;
  g_timer.on = false;
  if (!on) return ok();
  if (capacity < 1 || capacity > (1 << 20))
    return fail(GDR_ERR_INVALID_ARG, "gdr_stage_timer_enable: capacity %d out of range", capacity);
  g_timer.ev.resize(2 * (size_t)capacity);
  g_timer.id.resize(capacity);
  for (auto& e : g_timer.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      g_timer.ev.clear();
      return fail(GDR_ERR_CUDA, "gdr_stage_timer_enable: cudaEventCreate failed");
    }
  }
  g_timer.cap = capacity;
  g_timer.on = true;
  return ok();
}

gdr_status gdr_stage_timer_collect(double* total_ms, int* launches, int max_ids) {
  if (!total_ms || !launches || max_ids < 1)
    return fail(GDR_ERR_INVALID_ARG, "gdr_stage_timer_collect: bad output arrays");
  std::lock_guard<std::mutex> lk(g_timer.mu);
  for (int i = 0; i < max_ids; ++i) { total_ms[i] = 0.0; launches[i] = 0; }
  for (int s = 0; s < g_timer.used; ++s) {
    if (cudaEventSynchronize(g_timer.ev[2 * s + 1]) != cudaSuccess)
      return fail(GDR_ERR_CUDA, "gdr_stage_timer_collect: event sync failed");
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_timer.ev[2 * s], g_timer.ev[2 * s + 1]) != cudaSuccess)
      return fail(GDR_ERR_CUDA, "gdr_stage_timer_collect: elapsed time failed");
    const int id = g_timer.id[s];
    if (id >= 0 && id < max_ids) { total_ms[id] += ms; launches[id] += 1; }
  }
  g_timer.used = 0;
  return ok();
}

const char* gdr_kernel_name(int id) {
  switch (id) {
    case kKernRecurrent: return "gdr_recurrent";
    case kKernChunkPrep: return "gdr_chunk_prep";
    case kKernChunkState: return "gdr_chunk_state";
    case kKernPrologue: return "gdr_prologue";
    case kKernEpilogue: return "gdr_gated_rmsnorm";
    case kKernBackward: return "gdr_backward";
    case kKernBackwardReduce: return "gdr_backward_reduce";
    case kKernChunkAdjoint: return "gdr_chunk_adjoint";
    case kKernChunkBwdLocal: return "gdr_chunk_bwd_local";
  }
  return nullptr;
}

}  // extern "C"

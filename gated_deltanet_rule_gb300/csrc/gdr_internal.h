// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gdr {

constexpr int kD = 128;      // head dimension (Dk = Dv) the kernels implement
constexpr int kChunk = 64;   // tokens per chunk of the tensor-core path

// Device error codes written into the sticky error word (same values as gdr_status).
constexpr int kErrDeviceIndex = 4;
constexpr int kErrTimeout = 5;

// Kernel ids for the stage timer.
enum KernelId : int {
  kKernRecurrent = 0,
  kKernChunkPrep = 1,
  kKernChunkState = 2,
  kKernPrologue = 3,
  kNumKernelIds = 4
};

// Token-by-token recurrence on CUDA cores (float32 state in registers).
// Row b reads its initial state from S_in[(idx ? idx[b] : b)] (NULL S_in = zeros) and writes its
// final state to S_out[b] (NULL = not written). Used for the float32 path, float32 forks and decode.
struct RecurrentArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* S_in;
  const int64_t* idx;
  int n_in;            // number of states S_in holds (bounds for idx)
  void* o;
  float* S_out;
  int B, L, Hk, Hv;
  bool bf16;
  int* err;            // device error word
  const int32_t* lengths = nullptr;   // valid tokens per row (NULL = L): later tokens are not run,
                                      // their o is not written; a length outside [0, L] skips the row
};
cudaError_t launch_recurrent(const RecurrentArgs& a, cudaStream_t s);

// Chunked tensor-core path for bf16 q/k/v (two kernels: per-chunk WY factors, then the state
// recurrence). ws must hold chunk_workspace_bytes(B, Hk, L, Hv) bytes. Row b starts from
// S0[S0_idx ? S0_idx[b] : b] (NULL S0 = zeros); with S0_idx set, an index outside [0, n_S0) skips
// the row (nothing written) and records kErrDeviceIndex. Used for prefill rows and bf16 forks.
struct ChunkLaunch {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* S0;
  void* o;
  float* S_T;
  void* ws;
  int B, L, Hk, Hv;
  int* err;
  const int64_t* S0_idx = nullptr;
  int n_S0 = 0;
  const int32_t* lengths = nullptr;   // valid tokens per row (NULL = L), as for RecurrentArgs
  // gated RMSNorm epilogue (NULL z = none): o is written as w * o / sqrt(mean(o^2) + eps) * silu(z)
  const void* z = nullptr;            // [B, L, Hv, 128] bf16
  const float* w = nullptr;           // [128]
  float eps = 0.f;
  // the GDN prologue fused into the prep kernel (NULL mixed = none; otherwise q, k, v, g, beta are
  // unused and the conv has 4 taps): mixed [B, L, C] bf16 with C = (2 Hk + Hv) 128, its carry tail [B, 3, C] bf16 (NULL
  // = zeros), conv_w [C, 4], proj_a, proj_b [B, L, Hv], A_log, dt_bias [Hv]; new_tail [B, 3, C]
  // receives the carry for the next call (NULL = not written)
  const void* mixed = nullptr;
  const void* tail = nullptr;
  const float* conv_w = nullptr;
  const float* proj_a = nullptr;
  const float* proj_b = nullptr;
  const float* A_log = nullptr;
  const float* dt_bias = nullptr;
  void* new_tail = nullptr;
};
size_t chunk_workspace_bytes(int B, int Hk, int L, int Hv);
// the workspace of launch_chunk_bf16 with the fused prologue (any L: rows of one chunk included)
size_t chunk_prologue_workspace_bytes(int B, int L, int Hv);
cudaError_t launch_chunk_bf16(const ChunkLaunch& p, cudaStream_t s);

// GDN prologue (causal depthwise conv + SiLU over [tail, mixed], the gates, the conv carry).
// mixed [B, L, C] bf16 with C = (2 Hk + Hv) kD; tail / new_tail [B, K-1, C] bf16; conv_w [C, K];
// proj_a, proj_b [B, L, Hv]; A_log, dt_bias [Hv]; lengths [B] (NULL = all L); q, k, v bf16.
struct PrologueArgs {
  const void* mixed;
  const void* tail;
  const float* conv_w;
  const float* proj_a;
  const float* proj_b;
  const float* A_log;
  const float* dt_bias;
  const int32_t* lengths;
  void* q;
  void* k;
  void* v;
  float* g;
  float* beta;
  void* new_tail;
  int B, L, Hk, Hv, C, K;
  int* err;
  long long wait_budget = 0;   // cycles a wait for the staged tile may take (wait_budget_cycles())
};
cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t s);

// Cycles a kernel wait may take before it gives up with GDR_ERR_TIMEOUT (about 1 s by default;
// gdr_debug_set_wait_budget changes it for later launches).
long long wait_budget_cycles();

// Record a one-line message for gdr_last_error_message() on this host thread; returns status.
int record_error(int status, const char* message);

// Device error word of the current device (address of a __device__ int), looked up again when the
// device's context has changed since the last lookup.
int* device_error_word();

// The calling thread's current CUDA context (a CUcontext, NULL if none or on failure); symbol
// addresses cached per device are keyed on it.
void* current_context();

// Stage timer hooks (no-ops unless enabled): bracket one kernel launch on stream s.
int stage_timer_begin(cudaStream_t s, int kernel_id);
void stage_timer_end(int slot, cudaStream_t s);

}  // namespace gdr

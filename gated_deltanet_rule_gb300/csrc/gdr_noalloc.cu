// gdr_chunk_fwd_noalloc: the prefill call for callers that cannot allocate device memory.
//
// Some hosts own all of a GPU's memory: a serving process or engine that reserves its whole device
// budget at start-up (and the plugins loaded into it), or a latency-critical loop where a device
// allocation, which can synchronise the device and can fail under memory pressure, is not allowed
// once running. Such callers cannot provide gdr_chunk_fwd's workspace. This entry point runs the
// same kernels with a fixed scratch array that lives in this file as a static __device__ array: the
// driver places it in device memory when this library's code is loaded on a GPU, and it stays there
// until the process exits. Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "gdr.h"
#include "gdr_internal.h"

namespace {

constexpr size_t kScratchBytes = GDR_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device; it keeps whatever the previous call left in it. The bf16 path
// writes every byte of it that it later reads, so nothing has to be cleared between calls.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
// Device address of g_scratch per device ordinal, with the CUDA context it was looked up in: the
// address belongs to that context (a context created after cudaDeviceReset loads the module anew,
// possibly elsewhere), so a change of context triggers a new lookup.
struct ScratchAddr {
  void* ctx = nullptr;
  void* ptr = nullptr;
};
ScratchAddr g_scratch_addr[128];

}  // namespace

extern "C" gdr_status gdr_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                            const float* beta, const float* S0, void* o, float* S_T, int B,
                                            int L, int Hk, int Hv, int D, gdr_dtype dt, gdr_stream_t stream) {
  // Size check first: no CUDA call is made for a request the scratch cannot hold.
  const size_t need = gdr_chunk_workspace_bytes(B, L, Hk, Hv, D, dt);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "gdr_chunk_fwd_noalloc: these sizes need %zu bytes of scratch, the fixed scratch holds %zu "
             "(use gdr_chunk_fwd with a workspace)",
             need, kScratchBytes);
    return static_cast<gdr_status>(gdr::record_error(GDR_ERR_UNSUPPORTED, msg));
  }
  // In host code g_scratch names a host-side stand-in, not device memory: the kernels must get the
  // device address, looked up once per device (and again if the device's context changes) with that
  // device current.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
    return static_cast<gdr_status>(gdr::record_error(GDR_ERR_CUDA, "gdr_chunk_fwd_noalloc: no CUDA device"));
  void* scratch = nullptr;
  {
    void* ctx = gdr::current_context();
    std::lock_guard<std::mutex> lk(g_mu);
    ScratchAddr& a = g_scratch_addr[dev];
    if (a.ptr == nullptr || ctx == nullptr || a.ctx != ctx) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess || p == nullptr) {
        char msg[256];
        snprintf(msg, sizeof(msg), "gdr_chunk_fwd_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        return static_cast<gdr_status>(gdr::record_error(GDR_ERR_CUDA, msg));
      }
      a.ptr = p;
      a.ctx = gdr::current_context();   // the lookup has made the device's primary context current
    }
    scratch = a.ptr;
  }
  return gdr_chunk_fwd(q, k, v, g, beta, S0, o, S_T, B, L, Hk, Hv, D, dt, scratch, kScratchBytes, stream);
}
